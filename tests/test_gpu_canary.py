"""Canary padding around every output, workspace and id array of each call class.

A substitute for a bounds-checking build: each buffer a call receives sits in
the middle of a larger allocation whose head and tail (4 KB each, plus the
alignment slack) hold a fixed byte pattern.  After the call the padding must
be untouched, and every input buffer must still hold what it held before: no
kernel writes outside the buffers it is given, or into its inputs.  Covered:
verify, drafter and tree attention (both kernels), greedy, tree-greedy and
sampled acceptance (both forms), each at a shape with ragged edges.
"""
import numpy as np
import pytest
import torch

from serving_sd_verify_gb300 import workloads as W

pytestmark = pytest.mark.gpu

PAD = 4096
CANARY = 0xA5


@pytest.fixture(scope="module")
def S():
    from serving_sd_verify_gb300 import build, sd_verify
    build.build()
    sd_verify.load()
    yield sd_verify
    sd_verify.sd_set_attention_path(0)
    sd_verify.sd_set_sample_path(0)


class Arena:
    """Buffers carved out of canary-padded allocations."""

    def __init__(self):
        self.outs = []     # (allocation, nbytes)
        self.ins = []      # (allocation, nbytes, copy of the contents)

    def _alloc(self, shape, dtype):
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        slack = (-n) % 256
        buf = torch.full((PAD + n + slack + PAD,), CANARY, dtype=torch.uint8, device="cuda")
        return buf, n, buf[PAD:PAD + n].view(dtype).view(shape)

    def out(self, shape, dtype, fill):
        buf, n, t = self._alloc(shape, dtype)
        t.fill_(fill)
        self.outs.append((buf, n))
        return t

    def workspace(self, nbytes):
        buf, n, t = self._alloc((max(int(nbytes), 256),), torch.uint8)
        t.zero_()
        self.outs.append((buf, n))
        return t

    def inp(self, x):
        buf, n, t = self._alloc(tuple(x.shape), x.dtype)
        t.copy_(x.to("cuda"))
        self.ins.append((buf, n, buf.clone()))
        return t

    def check(self):
        torch.cuda.synchronize()
        for i, (buf, n) in enumerate(self.outs):
            assert bool((buf[:PAD] == CANARY).all()), f"output buffer {i}: write before its start"
            assert bool((buf[PAD + n:] == CANARY).all()), f"output buffer {i}: write past its end"
        for i, (buf, n, saved) in enumerate(self.ins):
            assert torch.equal(buf, saved), f"input buffer {i} changed"


# --------------------------------------------------------------------------
# attention
# --------------------------------------------------------------------------

@pytest.mark.parametrize("path", [1, 2])
@pytest.mark.parametrize("B,T,Hq,Hkv,ctx", [
    (2, 16, 28, 4, [300, 1001]),      # ragged, several splits
    (1, 16, 16, 1, [5000]),           # G = 16: two row blocks per kv head
])
def test_verify_attention_canary(S, path, B, T, Hq, Hkv, ctx):
    inp = W.verify_inputs(B=B, T=T, Hq=Hq, Hkv=Hkv, D=128, ctx=ctx, seed=B + T)
    a = Arena()
    q, k, v, c = a.inp(inp["q"]), a.inp(inp["k"]), a.inp(inp["v"]), a.inp(inp["ctx"])
    out = a.out((B, T, Hq, 128), torch.float32, float("nan"))
    ws = a.workspace(S.sd_verify_attention_workspace_size(B, T, Hq, Hkv, 128, inp["max_ctx"], S.SD_BF16))
    S.sd_set_attention_path(path)
    S.sd_verify_attention(q, k, v, c, inp["max_ctx"], out, inp["scale"], ws)
    assert S.sd_last_attention_path()[0] == path
    a.check()
    assert bool(torch.isfinite(out).all())
    assert S.sd_fault_word() == 0


@pytest.mark.parametrize("path", [1, 2])
def test_draft_attention_canary(S, path):
    B, T, Hq, Hkv = 2, 16, 28, 4
    d = W.drafter_inputs(B=B, T=T, Hq=Hq, Hkv=Hkv, D=128, n_ctx=[700, 2500], seed=9)
    L = d["layers"][0]
    a = Arena()
    q, kb, vb = a.inp(L["q"]), a.inp(L["kb"]), a.inp(L["vb"])
    kc, vc, n = a.inp(d["kc"]), a.inp(d["vc"]), a.inp(d["n_ctx"])
    out = a.out((B, T, Hq, 128), torch.float32, float("nan"))
    ws = a.workspace(S.sd_draft_block_attention_workspace_size(B, T, Hq, Hkv, 128, d["max_ctx"], S.SD_BF16))
    S.sd_set_attention_path(path)
    S.sd_draft_block_attention(q, kc, vc, n, d["max_ctx"], kb, vb, out, d["scale"], ws)
    assert S.sd_last_attention_path()[0] == path
    a.check()
    assert bool(torch.isfinite(out).all())
    assert S.sd_fault_word() == 0


@pytest.mark.parametrize("path", [1, 2])
def test_tree_attention_canary(S, path):
    B, T, Hq, Hkv = 1, 60, 28, 4
    rng = np.random.default_rng(60)
    parents = np.full(T, -1, dtype=np.int64)
    for j in range(1, T):
        parents[j] = rng.integers(max(0, j - 3), j)
    mask = np.zeros(T, dtype=np.uint64)
    for j in range(T):
        u, bits = j, 0
        while u != -1:
            bits |= 1 << int(u)
            u = int(parents[u])
        mask[j] = np.uint64(bits)
    inp = W.verify_inputs(B=B, T=T, Hq=Hq, Hkv=Hkv, D=128, ctx=[1500], seed=61)
    a = Arena()
    q, k, v, c = a.inp(inp["q"]), a.inp(inp["k"]), a.inp(inp["v"]), a.inp(inp["ctx"])
    tm = a.inp(torch.from_numpy(mask.view(np.int64)).reshape(B, T))
    out = a.out((B, T, Hq, 128), torch.float32, float("nan"))
    ws = a.workspace(S.sd_verify_tree_attention_workspace_size(B, T, Hq, Hkv, 128, inp["max_ctx"], S.SD_BF16))
    S.sd_set_attention_path(path)
    S.sd_verify_tree_attention(q, k, v, c, inp["max_ctx"], tm, out, inp["scale"], ws)
    assert S.sd_last_attention_path()[0] == path
    a.check()
    assert bool(torch.isfinite(out).all())
    assert S.sd_fault_word() == 0


# --------------------------------------------------------------------------
# acceptance
# --------------------------------------------------------------------------

def test_accept_greedy_canary(S):
    B, T, V = 3, 16, 5_001          # odd V: rows start unaligned
    g = W.greedy_inputs(B=B, T=T, V=V, seed=31)
    a = Arena()
    draft, logits = a.inp(g["draft"].to(torch.int32)), a.inp(g["logits"])
    n = a.out((B,), torch.int32, -1)
    c = a.out((B,), torch.int32, -1)
    ws = a.workspace(S.sd_accept_greedy_workspace_size(B, T, V, S.SD_BF16))
    S.sd_accept_greedy(draft, logits, n, c, ws)
    a.check()
    assert ((n >= 0) & (n < T)).all() and ((c >= 0) & (c < V)).all()
    assert S.sd_fault_word() == 0


def test_accept_tree_greedy_canary(S):
    B, T, V = 2, 60, 20_000
    rng = np.random.default_rng(62)
    parents = np.full((B, T), -1, dtype=np.int32)
    for b in range(B):
        for j in range(1, T):
            parents[b, j] = rng.integers(max(0, j - 3), j)
    g = W.greedy_inputs(B=B, T=T, V=V, seed=63)
    logits = g["logits"]
    am = logits.float().argmax(-1).numpy()
    tokens = np.zeros((B, T), dtype=np.int32)
    for b in range(B):
        for j in range(1, T):   # most nodes match the target's pick after their parent
            tokens[b, j] = am[b, parents[b, j]] if rng.random() < 0.7 else rng.integers(0, V)
    a = Arena()
    tk, pa, lg = a.inp(torch.from_numpy(tokens)), a.inp(torch.from_numpy(parents)), a.inp(logits)
    n = a.out((B,), torch.int32, -1)
    c = a.out((B,), torch.int32, -1)
    path = a.out((B, T), torch.int32, -7)
    ws = a.workspace(S.sd_accept_tree_greedy_workspace_size(B, T, V, S.SD_BF16))
    S.sd_accept_tree_greedy(tk, pa, lg, n, c, path, ws)
    a.check()
    assert ((n >= 0) & (n < T)).all() and ((c >= 0) & (c < V)).all()
    assert bool((path >= -1).all()) and bool((path < T).all())
    assert S.sd_fault_word() == 0


@pytest.mark.parametrize("path", [1, 2])
@pytest.mark.parametrize("B,T,V,dtype", [
    (4, 16, 20_000, torch.bfloat16),
    (3, 5, 5_003, torch.float32),    # odd V
])
def test_accept_sample_canary(S, path, B, T, V, dtype):
    smp = W.sample_inputs(B=B, T=T, V=V, seed=B * 7 + T, dtype=dtype)
    a = Arena()
    d, q, lg = a.inp(smp["draft"].to(torch.int32)), a.inp(smp["q"]), a.inp(smp["logits"])
    n = a.out((B,), torch.int32, -1)
    nx = a.out((B,), torch.int32, -1)
    ws = a.workspace(S.sd_accept_sample_workspace_size(B, T, V, S._dt(smp["logits"])))
    prev = S.sd_set_sample_path(path)
    try:
        S.sd_accept_sample(d, q, lg, 0.9, 4321, 3, n, nx, ws)
        assert S.sd_last_sample_path() == path
    finally:
        S.sd_set_sample_path(prev)
    a.check()
    assert ((n >= 0) & (n < T)).all() and ((nx >= 0) & (nx < V)).all()
    assert S.sd_fault_word() == 0
