"""Tree verification on the GPU against the oracle ("VFlash-FM" project page,
speedup table: the fastest variant verifies a draft tree).

Tree-masked attention on both attention kernels (every element on small
shapes, sampled rows at the 25,119-token workload) and greedy tree acceptance
(bit-exact lengths, correction ids and paths).  A chain-shaped tree must give
the chain calls' results.
"""
import numpy as np
import pytest
import torch

import oracle
from serving_sd_verify_gb300 import workloads as W
from _util import check_attention, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def S():
    from serving_sd_verify_gb300 import build, sd_verify
    build.build()
    sd_verify.load()
    yield sd_verify
    sd_verify.sd_set_attention_path(0)


def random_tree(rng, T, span=3):
    parents = np.full(T, -1, dtype=np.int32)
    for j in range(1, T):
        parents[j] = rng.integers(max(0, j - span), j)
    return parents


def masks(parents):
    """One 64-bit ancestor mask per node (bit k: node k is the node or an ancestor)."""
    m = np.zeros(len(parents), dtype=np.uint64)
    for j in range(len(parents)):
        v, bits = j, 0
        while v != -1:
            bits |= 1 << int(v)
            v = parents[v]
        m[j] = np.uint64(bits)
    return m


def run_tree_attention(S, inp, mask, path):
    q, k, v, ctx = inp["q"].cuda(), inp["k"].cuda(), inp["v"].cuda(), inp["ctx"].cuda()
    B, T, Hq, D = q.shape
    Hkv = k.shape[2]
    mc = inp["max_ctx"]
    tm = torch.from_numpy(np.ascontiguousarray(mask, dtype=np.uint64).view(np.int64)).reshape(B, T).cuda()
    out = torch.full((B, T, Hq, D), float("nan"), dtype=torch.float32, device="cuda")
    ws = S.workspace(S.sd_verify_tree_attention_workspace_size(B, T, Hq, Hkv, D, mc, S._dt(q)))
    S.sd_set_attention_path(path)
    S.sd_verify_tree_attention(q, k, v, ctx, mc, tm, out, inp["scale"], ws)
    used = S.sd_last_attention_path()
    torch.cuda.synchronize()
    assert S.sd_fault_word() == 0
    if path in (1, 2):
        assert used[0] == path
    return out.cpu().numpy().reshape(B * T * Hq, D)


TREE_CASES = [
    # B, T, Hq, Hkv, D, ctx, dtype, paths
    (2, 16, 28, 4, 128, [700, 130], torch.bfloat16, (1, 2)),   # several tiles, ragged tails
    (1, 16, 28, 4, 128, [1], torch.bfloat16, (1, 2)),          # the anchor is the only context key
    (2, 8, 4, 1, 64, [300, 5], torch.float32, (1,)),           # CUDA-core kernel only
    (1, 60, 28, 4, 128, [700], torch.bfloat16, (1, 2)),        # Tree-60: 4 row blocks of 18/18/18/6 nodes
    (2, 64, 8, 1, 128, [300, 40], torch.bfloat16, (1, 2)),     # 64 nodes (mask bit 63): 4 row blocks of 16
    (2, 33, 28, 4, 128, [129, 1], torch.bfloat16, (1, 2)),     # mask bit 32, the anchor alone as context
    (1, 40, 4, 1, 64, [100], torch.float32, (1,)),             # CUDA-core kernel, 40 nodes
]


@pytest.mark.parametrize("B,T,Hq,Hkv,D,ctx,dtype,paths", TREE_CASES)
def test_tree_attention_small_all_elements(S, B, T, Hq, Hkv, D, ctx, dtype, paths):
    rng = np.random.default_rng(B * 100 + T)
    inp = W.verify_inputs(B=B, T=T, Hq=Hq, Hkv=Hkv, D=D, ctx=ctx, dtype=dtype, seed=B + T + D)
    mask = np.stack([masks(random_tree(rng, T)) for _ in range(B)])
    want = oracle.tree_attention_rows(inp["q"], inp["k"], inp["v"], inp["ctx"], mask, inp["scale"])
    for path in paths:
        check_attention(run_tree_attention(S, inp, mask, path), want)


def test_chain_tree_gives_chain_attention(S):
    inp = W.verify_inputs(B=2, T=16, Hq=28, Hkv=4, D=128, ctx=[900, 77], dtype=torch.bfloat16, seed=9)
    chain = np.arange(-1, 15, dtype=np.int32)
    mask = np.stack([masks(chain)] * 2)
    for path in (1, 2):
        got = run_tree_attention(S, inp, mask, path)
        q, k, v, ctx = inp["q"].cuda(), inp["k"].cuda(), inp["v"].cuda(), inp["ctx"].cuda()
        out = torch.zeros(2, 16, 28, 128, dtype=torch.float32, device="cuda")
        ws = S.workspace(S.sd_verify_attention_workspace_size(2, 16, 28, 4, 128, inp["max_ctx"], S.SD_BF16))
        S.sd_set_attention_path(path)
        S.sd_verify_attention(q, k, v, ctx, inp["max_ctx"], out, inp["scale"], ws)
        torch.cuda.synchronize()
        assert np.abs(got - out.cpu().numpy().reshape(got.shape)).max() < 1e-6


def test_tree_attention_full_size_workload(S):
    cfg = W.config(2)
    inp = cfg["attn"]
    rng = np.random.default_rng(60)
    mask = masks(random_tree(rng, 16))[None]
    rows = sample_rows(1, 16, 28, 64, seed=60)
    want = oracle.tree_attention_rows(inp["q"], inp["k"], inp["v"], inp["ctx"], mask, inp["scale"], rows=rows)
    for path in (0, 2):
        check_attention(run_tree_attention(S, inp, mask, path)[rows], want)


def tree60(rng, T=60, span=3):
    """A seeded draft tree of T nodes, each node's parent among the span nodes before it."""
    return random_tree(rng, T, span)


def test_tree60_attention_full_size_workload(S):
    """The pages' Tree-60 at the 25,119-token workload (LLaVA-OneVision-7B
    shape): 60 nodes verified in one call, sampled rows against the oracle."""
    T = 60
    inp = W.verify_inputs(B=1, T=T, Hq=28, Hkv=4, D=128, ctx=25_119, seed=2)
    rng = np.random.default_rng(61)
    mask = masks(tree60(rng, T))[None]
    rows = sample_rows(1, T, 28, 96, seed=61)
    want = oracle.tree_attention_rows(inp["q"], inp["k"], inp["v"], inp["ctx"], mask, inp["scale"], rows=rows)
    for path in (0, 2):
        check_attention(run_tree_attention(S, inp, mask, path)[rows], want)


def run_tree_greedy(S, tokens, parents, logits):
    B, T, V = logits.shape
    n = torch.full((B,), -1, dtype=torch.int32, device="cuda")
    c = torch.full((B,), -1, dtype=torch.int32, device="cuda")
    path = torch.full((B, T), -7, dtype=torch.int32, device="cuda")
    ws = S.workspace(S.sd_accept_tree_greedy_workspace_size(B, T, V, S._dt(logits)))
    S.sd_accept_tree_greedy(torch.from_numpy(tokens).cuda(), torch.from_numpy(parents).cuda(), logits.cuda(),
                            n, c, path, ws)
    torch.cuda.synchronize()
    assert S.sd_fault_word() == 0
    assert int(ws[:256].abs().sum()) == 0, "ticket counter not returned to zero"
    return n.cpu().numpy(), c.cpu().numpy(), path.cpu().numpy()


@pytest.mark.parametrize("B,T,V,dtype", [(4, 16, 152_064, torch.bfloat16), (8, 9, 1_000, torch.float32),
                                         (3, 1, 500, torch.bfloat16), (2, 60, 152_064, torch.bfloat16),
                                         (5, 64, 2_000, torch.bfloat16), (3, 33, 700, torch.float32)])
def test_tree_greedy_matches_oracle(S, B, T, V, dtype):
    rng = np.random.default_rng(B * T)
    g = W.greedy_inputs(B=B, T=T, V=V, dtype=dtype, seed=B + T)
    logits = g["logits"]
    am = logits.float().numpy().argmax(-1)
    parents = np.stack([random_tree(rng, T) for _ in range(B)])
    tokens = np.zeros((B, T), dtype=np.int32)
    for b in range(B):
        for j in range(1, T):
            # mostly the parent's argmax (accepted), sometimes not
            tokens[b, j] = am[b, parents[b, j]] if rng.random() < 0.7 else rng.integers(0, V)
    n, c, path = run_tree_greedy(S, tokens, parents, logits)
    on, oc, ob, op = oracle.accept_tree_greedy(tokens, parents, logits)
    assert (n == on).all() and (c == oc).all() and (path == op).all()


def test_chain_tree_greedy_gives_chain_greedy(S):
    g = W.greedy_inputs(B=3, T=16, V=152_064, seed=77)
    B, T = 3, 16
    tokens = np.zeros((B, T), dtype=np.int32)
    tokens[:, 1:] = g["draft"].numpy()
    parents = np.stack([np.arange(-1, T - 1, dtype=np.int32)] * B)
    n, c, path = run_tree_greedy(S, tokens, parents, g["logits"])
    n2 = torch.zeros(B, dtype=torch.int32, device="cuda")
    c2 = torch.zeros(B, dtype=torch.int32, device="cuda")
    ws = S.workspace(S.sd_accept_greedy_workspace_size(B, T, 152_064, S.SD_BF16))
    S.sd_accept_greedy(g["draft"].cuda(), g["logits"].cuda(), n2, c2, ws)
    torch.cuda.synchronize()
    assert (n == n2.cpu().numpy()).all() and (c == c2.cpu().numpy()).all()
    assert (n == np.array(g["k"]).clip(max=15)).all()


def test_tree_greedy_bad_parent_sets_the_fault_word(S):
    g = W.greedy_inputs(B=1, T=4, V=100, seed=3)
    tokens = np.zeros((1, 4), dtype=np.int32)
    parents = np.array([[-1, 0, 3, 1]], dtype=np.int32)   # node 2's parent is not before it
    S.sd_fault_word()  # cleared
    n = torch.zeros(1, dtype=torch.int32, device="cuda")
    c = torch.zeros(1, dtype=torch.int32, device="cuda")
    path = torch.zeros(1, 4, dtype=torch.int32, device="cuda")
    ws = S.workspace(S.sd_accept_tree_greedy_workspace_size(1, 4, 100, S.SD_BF16))
    S.sd_accept_tree_greedy(torch.from_numpy(tokens).cuda(), torch.from_numpy(parents).cuda(), g["logits"].cuda(),
                            n, c, path, ws)
    torch.cuda.synchronize()
    assert S.sd_fault_word() != 0   # read and cleared
