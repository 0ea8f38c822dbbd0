"""GPU parity of the drafter K/V projector against the fp64 oracle.

The kernels accumulate in fp32 and round once to bf16, so every element must
lie within half a bf16 ulp of the exact value plus the fp32 summation bound
(Hd * 2^-23 * sum_f |h_f w_f|), and nearly every element must equal the exact
value rounded to bf16.
"""
import numpy as np
import pytest
import torch

from _util import check_projection
from serving_sd_verify_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def S():
    from serving_sd_verify_gb300 import build, sd_verify
    build.build()
    sd_verify.load()
    return sd_verify


@pytest.fixture(autouse=True)
def _auto_path(S):
    yield
    S.sd_set_projector_path(0)


def inputs(N, Hd, Dout, seed):
    g = torch.Generator().manual_seed(seed)
    h = torch.randn(N, Hd, generator=g).to(torch.bfloat16)
    a = (6.0 / (Hd + Dout)) ** 0.5
    wk = ((torch.rand(Dout, Hd, generator=g) * 2 - 1) * a).to(torch.bfloat16)
    wv = ((torch.rand(Dout, Hd, generator=g) * 2 - 1) * a).to(torch.bfloat16)
    return h, wk, wv


def check(got, h, w, rows=None, min_exact=0.99):
    check_projection(got, h, w, rows, min_exact)


def run(S, h, wk, wv, path=0):
    S.sd_set_projector_path(path)
    N, Dout = h.shape[0], wk.shape[0]
    k = torch.full((N, Dout), 7.0, dtype=torch.bfloat16, device="cuda")
    v = torch.full((N, Dout), 7.0, dtype=torch.bfloat16, device="cuda")
    S.sd_project_kv(h.cuda(), wk.cuda(), wv.cuda(), k, v)
    torch.cuda.synchronize()
    used = S.sd_last_projector_path()
    return k.cpu(), v.cpu(), used


@pytest.mark.parametrize("N,Hd,Dout", [
    (1, 3584, 512), (5, 3584, 512), (8, 3584, 512), (13, 200, 96), (16, 1024, 64), (9, 8192, 64),
])
def test_append_rows_cuda_cores(S, N, Hd, Dout):
    h, wk, wv = inputs(N, Hd, Dout, seed=N * 7 + Hd)
    k, v, used = run(S, h, wk, wv)
    assert used == 1
    check(k, h, wk)
    check(v, h, wv)


@pytest.mark.parametrize("N,Hd,Dout", [
    (17, 3584, 512),      # just above the CUDA-core bound
    (12, 16384, 64),      # 16 rows of 16384 features do not fit the CUDA-core kernel's shared memory
    (300, 3584, 512),     # ragged last row tile
    (257, 200, 96),       # feature tail inside one 64-wide step; a partial column tile
    (640, 1024, 288),     # columns 256..287 in a second tile
])
def test_prefill_rows_tensor_cores(S, N, Hd, Dout):
    h, wk, wv = inputs(N, Hd, Dout, seed=N + Dout)
    k, v, used = run(S, h, wk, wv)
    assert used == 2
    check(k, h, wk)
    check(v, h, wv)


@pytest.mark.parametrize("path,N", [(1, 300), (2, 5), (2, 1)])
def test_forced_paths_agree_with_oracle(S, path, N):
    h, wk, wv = inputs(N, 512, 128, seed=99 + N)
    k, v, used = run(S, h, wk, wv, path=path)
    assert used == path
    check(k, h, wk)
    check(v, h, wv)


@pytest.mark.parametrize("N", [8, 200])
def test_append_into_cache_rows_with_strides(S, N):
    """Hidden rows read from a wider buffer; outputs written into rows
    [pos, pos + N) of a [S, Hkv*D] cache whose other rows stay untouched."""
    Hd, Hkv, D, pos, Srows = 512, 2, 64, 37, 300
    g = torch.Generator().manual_seed(N)
    hbuf = torch.randn(N, Hd + 24, generator=g).to(torch.bfloat16)
    h = hbuf[:, :Hd]
    _, wk, wv = inputs(1, Hd, Hkv * D, seed=3)
    kc = torch.full((Srows, Hkv, D), -3.0, dtype=torch.bfloat16, device="cuda")
    vc = torch.full((Srows, Hkv, D), -3.0, dtype=torch.bfloat16, device="cuda")
    hd = hbuf.cuda()[:, :Hd]
    S.sd_project_kv(hd, wk.cuda(), wv.cuda(), kc.view(Srows, Hkv * D)[pos:pos + N],
                    vc.view(Srows, Hkv * D)[pos:pos + N])
    torch.cuda.synchronize()
    kc, vc = kc.cpu().view(Srows, Hkv * D), vc.cpu().view(Srows, Hkv * D)
    check(kc[pos:pos + N], h.contiguous(), wk)
    check(vc[pos:pos + N], h.contiguous(), wv)
    for c in (kc, vc):
        assert (c[:pos] == -3.0).all() and (c[pos + N:] == -3.0).all()


def test_prefill_full_context_sampled_rows(S):
    """The 25,119-row context of the LLaVA-OneVision-7B workload (Qwen2-7B
    hidden size 3584, 4 KV heads x 128) on the tensor-core path, checked on
    256 random rows plus the ragged last row tile, and for determinism."""
    N, Hd, Dout = 25_119, 3584, 512
    h, wk32, wv32 = W.hidden_and_projector(N=N, seed=4)
    wk = wk32.t().contiguous().to(torch.bfloat16)
    wv = wv32.t().contiguous().to(torch.bfloat16)
    hd, wkd, wvd = h.cuda(), wk.cuda(), wv.cuda()
    k = torch.empty(N, Dout, dtype=torch.bfloat16, device="cuda")
    v = torch.empty_like(k)
    S.sd_project_kv(hd, wkd, wvd, k, v)
    assert S.sd_last_projector_path() == 2
    k2, v2 = torch.empty_like(k), torch.empty_like(v)
    S.sd_project_kv(hd, wkd, wvd, k2, v2)
    torch.cuda.synchronize()
    assert torch.equal(k, k2) and torch.equal(v, v2)
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([rng.integers(0, N, 256), np.arange(N - 31, N)]))
    sel = torch.from_numpy(rows)
    check(k[sel.cuda()].cpu(), h[sel], wk)
    check(v[sel.cuda()].cpu(), h[sel], wv)
    assert S.sd_fault_word() == 0


def test_projector_argument_errors(S):
    h = torch.zeros(4, 64, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(64, 64, dtype=torch.bfloat16, device="cuda")
    o = torch.zeros(4, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(S.SdError) as e:
        S.sd_project_kv(h.float(), w, w, o, o)
    assert e.value.status == S.SD_ERR_UNSUPPORTED
    w48 = torch.zeros(48, 64, dtype=torch.bfloat16, device="cuda")
    o48 = torch.zeros(4, 48, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(S.SdError) as e:
        S.sd_project_kv(h, w48, w48, o48, o48)
    assert e.value.status == S.SD_ERR_INVALID_ARG
    obuf = torch.zeros(4 * 64 + 1, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(S.SdError) as e:       # 2-byte offset: not 16-byte aligned
        S.sd_project_kv(h, w, w, obuf[1:].view(4, 64), o)
    assert e.value.status == S.SD_ERR_INVALID_ARG
    S.sd_project_kv(h[:0], w, w, o[:0], o[:0])   # N = 0 launches nothing
    assert S.sd_last_projector_path() == 0
    assert S.sd_fault_word() == 0
