"""GPU parity of the attention kernels (target verify, drafter) against the oracle.

Small shapes are checked on every output element; the full-size workloads on
sampled rows (first and last block rows of every sequence plus a random
sample).  Both kernels are covered: path 1 (CUDA-core) is forced for every
case, and the tensor-core kernel (path 2) is required wherever it applies.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from serving_sd_verify_gb300 import workloads as W
from _util import check_attention, oracle_verify_rows, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def S():
    from serving_sd_verify_gb300 import build, sd_verify
    build.build()
    sd_verify.load()
    yield sd_verify
    sd_verify.sd_set_attention_path(0)


@pytest.fixture(autouse=True)
def _automatic_path(S):
    S.sd_set_attention_path(0)
    yield
    S.sd_set_attention_path(0)


def tc_applies(dtype, D, G, T):
    # the tensor-core kernel cuts G*T rows into row blocks of whole block rows
    return dtype == torch.bfloat16 and D == 128 and G <= 128


def run_verify(S, inp, path, max_ctx=None, out_rows=None):
    q, k, v, ctx = inp["q"].cuda(), inp["k"].cuda(), inp["v"].cuda(), inp["ctx"].cuda()
    B, T, Hq, D = q.shape
    Hkv = k.shape[2]
    mc = max_ctx or inp["max_ctx"]
    out = torch.full((B, T, Hq, D), float("nan"), dtype=torch.float32, device="cuda")
    ws = S.workspace(S.sd_verify_attention_workspace_size(B, T, Hq, Hkv, D, mc, S._dt(q)))
    S.sd_set_attention_path(path)
    S.sd_verify_attention(q, k, v, ctx, mc, out, inp["scale"], ws)
    used = S.sd_last_attention_path()
    torch.cuda.synchronize()
    assert S.sd_fault_word() == 0
    if path in (1, 2):
        assert used[0] == path
    return out.cpu().numpy().reshape(B * T * Hq, D), used


def run_draft(S, d, layer, path, max_ctx=None):
    L = d["layers"][layer]
    q, kb, vb = L["q"].cuda(), L["kb"].cuda(), L["vb"].cuda()
    kc, vc, n = d["kc"].cuda(), d["vc"].cuda(), d["n_ctx"].cuda()
    B, T, Hq, D = q.shape
    Hkv = kc.shape[2]
    mc = max_ctx or d["max_ctx"]
    out = torch.full((B, T, Hq, D), float("nan"), dtype=torch.float32, device="cuda")
    ws = S.workspace(S.sd_draft_block_attention_workspace_size(B, T, Hq, Hkv, D, mc, S._dt(q)))
    S.sd_set_attention_path(path)
    S.sd_draft_block_attention(q, kc, vc, n, mc, kb, vb, out, d["scale"], ws)
    used = S.sd_last_attention_path()
    torch.cuda.synchronize()
    assert S.sd_fault_word() == 0
    if path in (1, 2):
        assert used[0] == path
    return out.cpu().numpy().reshape(B * T * Hq, D)


def paths_for(dtype, D, G, T):
    return [1, 2] if tc_applies(dtype, D, G, T) else [1]


VERIFY_CASES = [
    # B, T, Hq, Hkv, D, ctx, dtype
    (1, 16, 4, 1, 64, [512], torch.float32),
    (1, 16, 28, 4, 128, [700], torch.bfloat16),     # several tiles + ragged tail
    (2, 16, 28, 4, 128, [1, 130], torch.bfloat16),  # ctx of one, tail inside a tile
    (3, 1, 28, 4, 128, [5, 64, 1000], torch.bfloat16),  # T = 1: decode
    (2, 2, 8, 8, 128, [63, 65], torch.bfloat16),    # MHA
    (1, 16, 64, 8, 128, [2000], torch.bfloat16),    # 72B-shaped, G*T = 128
    (2, 16, 16, 1, 64, [300, 77], torch.bfloat16),  # MQA, G*T = 256 (CUDA-core only: D 64)
    (2, 16, 16, 1, 128, [300, 77], torch.bfloat16),  # MQA, G*T = 256: two row blocks of 8 block rows
    (1, 16, 24, 1, 128, [390], torch.bfloat16),      # G 24: 5 block rows per row block, the last with 1
    (5, 16, 28, 4, 128, [1, 3000, 40, 9000, 128], torch.bfloat16),  # ragged: 1 to 71 tiles, splits by length
    (1, 5, 7, 1, 128, [333], torch.float32),
]


@pytest.mark.parametrize("B,T,Hq,Hkv,D,ctx,dtype", VERIFY_CASES)
def test_verify_small_all_elements(S, B, T, Hq, Hkv, D, ctx, dtype):
    inp = W.verify_inputs(B=B, T=T, Hq=Hq, Hkv=Hkv, D=D, ctx=ctx, dtype=dtype, seed=sum(ctx) + T,
                          prescale_q=dtype != torch.float32)
    want = oracle.attention_rows(inp["q"], inp["k"], inp["v"], inp["ctx"], inp["scale"])
    for path in paths_for(dtype, D, Hq // Hkv, T):
        got, _ = run_verify(S, inp, path)
        check_attention(got, want)


def test_verify_max_ctx_larger_than_ctx(S):
    # a preallocated cache with spare slots; unused slots hold NaN and must not leak
    B, T, Hq, Hkv, D = 2, 16, 28, 4, 128
    inp = W.verify_inputs(B=B, T=T, Hq=Hq, Hkv=Hkv, D=D, ctx=[100, 900], seed=3, s_max=1200)
    k, v = inp["k"].clone(), inp["v"].clone()
    k[0, 100 + T - 1:] = float("nan"); v[0, 100 + T - 1:] = float("nan")
    k[1, 900 + T - 1:] = float("nan"); v[1, 900 + T - 1:] = float("nan")
    inp2 = dict(inp, k=k, v=v)
    want = oracle_verify_rows(inp["q"], inp["k"], inp["v"], inp["ctx"], 1.0, np.arange(B * T * Hq))
    for path in (1, 2):
        got, _ = run_verify(S, inp2, path, max_ctx=1100)
        check_attention(got, want)


def test_verify_strided_cache(S):
    # cache stored as [B, Hkv, S, D] (head-major) and passed through strides
    B, T, Hq, Hkv, D = 2, 16, 28, 4, 128
    inp = W.verify_inputs(B=B, T=T, Hq=Hq, Hkv=Hkv, D=D, ctx=[200, 333], seed=4)
    want = oracle.attention_rows(inp["q"], inp["k"], inp["v"], inp["ctx"], 1.0)
    kh = inp["k"].permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3)
    vh = inp["v"].permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3)
    q, ctx = inp["q"].cuda(), inp["ctx"].cuda()
    kd = inp["k"].permute(0, 2, 1, 3).contiguous().cuda().permute(0, 2, 1, 3)
    vd = inp["v"].permute(0, 2, 1, 3).contiguous().cuda().permute(0, 2, 1, 3)
    assert kd.stride(1) == D and kh.stride(1) == D
    for path in (1, 2):
        out = torch.zeros(B, T, Hq, D, device="cuda")
        ws = S.workspace(S.sd_verify_attention_workspace_size(B, T, Hq, Hkv, D, 333, S.SD_BF16))
        S.sd_set_attention_path(path)
        S.sd_verify_attention(q, kd, vd, ctx, 333, out, 1.0, ws)
        torch.cuda.synchronize()
        check_attention(out.cpu().numpy().reshape(-1, D), want)


def test_verify_row_sees_exactly_ctx_plus_j(S):
    # perturbing slot ctx+j changes rows > j only (GPU, both paths)
    B, T, Hq, Hkv, D, ctx = 1, 16, 28, 4, 128, 500
    inp = W.verify_inputs(B=B, T=T, Hq=Hq, Hkv=Hkv, D=D, ctx=ctx, seed=8)
    for path in (1, 2):
        base, _ = run_verify(S, inp, path)
        k2, v2 = inp["k"].clone(), inp["v"].clone()
        k2[0, ctx + 6] += 2.0
        v2[0, ctx + 6] += 4.0
        pert, _ = run_verify(S, dict(inp, k=k2, v=v2), path)
        base, pert = base.reshape(T, Hq, D), pert.reshape(T, Hq, D)
        assert np.array_equal(base[:7], pert[:7])
        assert (np.abs(base[7:] - pert[7:]).max(axis=(1, 2)) > 1e-3).all()


@pytest.mark.parametrize("direction", [1.0, -1.0])
def test_verify_moving_running_max(S, direction):
    # keys carry a component along q that grows (or shrinks) along the sequence,
    # so the running max moves by many powers of two across tiles
    B, T, Hq, Hkv, D, ctx = 1, 16, 28, 4, 128, 2000
    inp = W.verify_inputs(B=B, T=T, Hq=Hq, Hkv=Hkv, D=D, ctx=ctx, seed=21)
    u = torch.ones(D) / math.sqrt(D)
    ramp = torch.linspace(0.0, 1.0, ctx + T - 1)
    if direction < 0:
        ramp = 1.0 - ramp
    k = (0.2 * inp["k"].float() + 60.0 * ramp.view(1, -1, 1, 1) * u).to(torch.bfloat16)
    q = (inp["q"].float() + u).to(torch.bfloat16)
    inp2 = dict(inp, k=k, q=q)
    want = oracle.attention_rows(q, k, inp["v"], inp["ctx"], 1.0)
    for path in (1, 2):
        got, _ = run_verify(S, inp2, path)
        check_attention(got, want)


@pytest.mark.parametrize("n", [1, 2, 3, 5])
def test_verify_full_size_workloads(S, n):
    cfg = W.config(n)
    inp, dims = cfg["attn"], cfg["dims"]
    B, T, Hq, Hkv, D = dims["B"], dims["T"], dims["Hq"], dims["Hkv"], dims["D"]
    rows = sample_rows(B, T, Hq, 64 if n != 1 else B * T * Hq, seed=n)
    want = oracle_verify_rows(inp["q"], inp["k"], inp["v"], inp["ctx"], inp["scale"], rows)
    dtype = inp["q"].dtype
    for path in [0] + paths_for(dtype, D, Hq // Hkv, T):
        got, used = run_verify(S, inp, path)
        check_attention(got[rows], want)
        if path == 0 and tc_applies(dtype, D, Hq // Hkv, T) and n != 1:
            assert used[0] == 2, "the tensor-core kernel should serve this workload"


DRAFT_CASES = [
    (1, 16, 28, 4, 128, [25], torch.bfloat16),
    (2, 16, 28, 4, 128, [1, 700], torch.bfloat16),
    (1, 16, 4, 1, 64, [300], torch.float32),
    (2, 3, 8, 2, 128, [64, 129], torch.bfloat16),
    (1, 16, 32, 2, 128, [500], torch.bfloat16),   # G*T = 256: two row blocks
    (1, 1, 28, 4, 128, [300], torch.bfloat16),    # T = 1: a block tile of one row (the copy zero-fills the rest)
    (3, 16, 28, 4, 128, [10, 2000, 129], torch.bfloat16),  # ragged: the block tile leads each unit's first split
]


@pytest.mark.parametrize("B,T,Hq,Hkv,D,nctx,dtype", DRAFT_CASES)
def test_draft_small_all_elements(S, B, T, Hq, Hkv, D, nctx, dtype):
    d = W.drafter_inputs(B=B, T=T, Hq=Hq, Hkv=Hkv, D=D, n_ctx=nctx, layers=1, seed=sum(nctx),
                         dtype=dtype)
    L = d["layers"][0]
    want = oracle.attention_rows(L["q"], d["kc"], d["vc"], d["n_ctx"], 1.0, mode=1, kb=L["kb"], vb=L["vb"])
    for path in paths_for(dtype, D, Hq // Hkv, T):
        check_attention(run_draft(S, d, 0, path), want)


def test_draft_workload4_full_size(S):
    cfg = W.config(4)
    kc, vc = W.project_kv(cfg["hidden"], cfg["wk"], cfg["wv"], device="cuda")
    d = W.drafter_layers(kc, vc)
    B, T, Hq = 1, 16, 28
    rows = sample_rows(B, T, Hq, 48, seed=4)
    for layer in range(4):
        L = d["layers"][layer]
        want = oracle_verify_rows(L["q"], kc, vc, d["n_ctx"], 1.0, rows, mode=1, kb=L["kb"], vb=L["vb"])
        for path in (0, 1, 2, 3):
            check_attention(run_draft(S, d, layer, path)[rows], want)


def test_attention_errors_are_reported(S):
    q = torch.zeros(1, 16, 28, 128, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(1, 100, 4, 128, dtype=torch.bfloat16, device="cuda")
    ctx = torch.tensor([80], dtype=torch.int32, device="cuda")
    out = torch.zeros(1, 16, 28, 128, device="cuda")
    with pytest.raises(S.SdError) as e:
        S.sd_verify_attention(q, k, k, ctx, 80, out, 1.0, torch.zeros(64, dtype=torch.uint8, device="cuda"))
    assert e.value.status == S.SD_ERR_WORKSPACE
    q96 = torch.zeros(1, 16, 28, 96, dtype=torch.bfloat16, device="cuda")
    k96 = torch.zeros(1, 100, 4, 96, dtype=torch.bfloat16, device="cuda")
    ws = S.workspace(1 << 24)
    with pytest.raises(S.SdError) as e:
        S.sd_verify_attention(q96, k96, k96, ctx, 80, torch.zeros(1, 16, 28, 96, device="cuda"), 1.0, ws)
    assert e.value.status == S.SD_ERR_UNSUPPORTED
    assert S.sd_fault_word() == 0


def test_bad_ctx_len_sets_fault_word_without_faulting(S):
    # a ctx_len beyond max_ctx is clamped on the device and flagged
    inp = W.verify_inputs(B=1, T=16, Hq=28, Hkv=4, D=128, ctx=[300], seed=2)
    q, k, v = inp["q"].cuda(), inp["k"].cuda(), inp["v"].cuda()
    ctx = torch.tensor([5000], dtype=torch.int32, device="cuda")
    out = torch.zeros(1, 16, 28, 128, device="cuda")
    ws = S.workspace(S.sd_verify_attention_workspace_size(1, 16, 28, 4, 128, 300, S.SD_BF16))
    for path in (1, 2):
        S.sd_set_attention_path(path)
        S.sd_verify_attention(q, k, v, ctx, 300, out, 1.0, ws)
        assert S.sd_fault_word() & 1
        want = oracle.attention_rows(inp["q"], inp["k"], inp["v"], inp["ctx"], 1.0)
        check_attention(out.cpu().numpy().reshape(-1, 128), want)


def test_verify_in_kernel_merge_reuses_its_workspace(S):
    """The tensor-core kernel merges its splits inside the kernel through one
    counter per (sequence, kv head) kept in the workspace: every completed call
    leaves the counters at zero, so a second call on the same workspace gives
    the same bits; a single split writes the output directly (one launch)."""
    cfg = W.config(2)
    inp, dims = cfg["attn"], cfg["dims"]
    B, T, Hq, Hkv, D = dims["B"], dims["T"], dims["Hq"], dims["Hkv"], dims["D"]
    q, k, v, ctx = inp["q"].cuda(), inp["k"].cuda(), inp["v"].cuda(), inp["ctx"].cuda()
    mc = inp["max_ctx"]
    ws = S.workspace(S.sd_verify_attention_workspace_size(B, T, Hq, Hkv, D, mc, S._dt(q)))
    outs = []
    S.sd_set_attention_path(2)
    for _ in range(2):
        out = torch.full((B, T, Hq, D), float("nan"), dtype=torch.float32, device="cuda")
        S.sd_verify_attention(q, k, v, ctx, mc, out, inp["scale"], ws)
        path, n_splits = S.sd_last_attention_path()
        launches = S.sd_last_attention_launches()
        torch.cuda.synchronize()
        assert S.sd_fault_word() == 0
        assert path == 2 and n_splits > 1 and launches == 1
        assert int(ws[256:256 + 4 * B * Hkv].abs().sum()) == 0, "merge counters not returned to zero"
        outs.append(out.cpu())
    assert torch.equal(outs[0], outs[1])
    rows = sample_rows(B, T, Hq, 16, seed=22)
    want = oracle_verify_rows(inp["q"], inp["k"], inp["v"], inp["ctx"], inp["scale"], rows)
    check_attention(outs[1].numpy().reshape(B * T * Hq, D)[rows], want)
    # a context of one tile per kv head: one CTA per (sequence, kv head), each
    # writing its output itself
    small = W.verify_inputs(B=1, T=16, Hq=28, Hkv=4, D=128, ctx=[100], dtype=torch.bfloat16, seed=23)
    got, used = run_verify(S, small, 2)
    assert used == (2, 4) and S.sd_last_attention_launches() == 1
    check_attention(got, oracle_verify_rows(small["q"], small["k"], small["v"], small["ctx"], small["scale"],
                                            list(range(16 * 28))))
    S.sd_set_attention_path(0)
