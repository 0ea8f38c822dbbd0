"""GPU parity of the on-device commit: token / length bookkeeping and tree
K/V compaction bit-exact against the oracle, the commit-time drafter append
within the projector tolerance, and whole cycles (accept -> compact -> append
-> commit) captured in one CUDA graph and replayed with no host round trip,
against the oracle run cycle by cycle."""
import numpy as np
import pytest
import torch

import oracle
from _util import check_projection

pytestmark = pytest.mark.gpu

BAD_COMMIT = 1 << 6


@pytest.fixture(scope="module")
def S():
    from serving_sd_verify_gb300 import build, sd_verify
    build.build()
    sd_verify.load()
    return sd_verify


def cuda_i32(x):
    return torch.as_tensor(np.ascontiguousarray(x, dtype=np.int32)).cuda()


def random_paths(rng, B, T, V=50):
    """Valid tree paths from the oracle's tree acceptance on random trees."""
    parents = np.zeros((B, T), np.int32)
    parents[:, 0] = -1
    for j in range(1, T):
        parents[:, j] = rng.integers(max(0, j - 4), j, B)
    logits = rng.standard_normal((B, T, V))
    am = logits.argmax(-1)
    tokens = rng.integers(0, V, (B, T)).astype(np.int32)
    for b in range(B):
        for j in range(1, T):
            if rng.random() < 0.7:
                tokens[b, j] = am[b, parents[b, j]]
    n, c, best, path = oracle.accept_tree_greedy(tokens, parents, logits)
    return tokens, parents, logits, n, c, path


def deep_first(n, path, T):
    """Sequence 0 keeps a whole chain of T - 1 nodes (the deepest commit a tree
    of T nodes allows), so trees of up to 64 nodes reach their last rows."""
    n, path = n.copy(), path.copy()
    n[0] = T - 1
    path[0, :] = np.arange(1, T + 1)
    path[0, T - 1] = -1
    return n, path


@pytest.mark.parametrize("tree,T", [(False, 16), (True, 16), (True, 64)])
def test_commit_tokens_match_oracle(S, tree, T):
    rng = np.random.default_rng(3 + tree + (T if T > 16 else 0))
    B, cap = 40, 64 if T <= 16 else 2 * T + 40
    if tree:
        prop, _, _, n, nx, path = random_paths(rng, B, T)
        if T > 16:
            n, path = deep_first(n, path, T)
    else:
        prop = rng.integers(0, 1000, (B, T - 1)).astype(np.int32)
        n = rng.integers(0, T, B).astype(np.int32)
        n[:3] = [0, T - 1, 5]
        nx = rng.integers(0, 1000, B).astype(np.int32)
        path = None
    ctx = rng.integers(1, 3000, B).astype(np.int32)
    olen = rng.integers(0, 40, B).astype(np.int32)
    toks = rng.integers(0, 1000, (B, cap)).astype(np.int32)
    ctx_cap = 3000
    # out of range: n too large, output full, ctx past its cap, ctx 0
    n[5] = T
    olen[6] = cap - int(n[6])
    ctx[7] = ctx_cap - int(n[7])
    ctx[8] = 0
    if tree:
        path = path.copy()
        n[9] = max(int(n[9]), 1)
        path[9, 0] = 0
    want = oracle.commit_tokens(prop, n, nx, ctx, toks, olen, ctx_cap, path=path)
    d = {k: cuda_i32(v) for k, v in (("ctx", ctx), ("olen", olen), ("toks", toks))}
    dctx = torch.full((B,), -5, dtype=torch.int32, device="cuda")
    anchor = torch.full((B,), -1, dtype=torch.int32, device="cuda")
    status = torch.full((B,), 9, dtype=torch.int32, device="cuda")
    S.sd_fault_word(clear=True)
    S.sd_commit_tokens(cuda_i32(prop), cuda_i32(n), cuda_i32(nx), d["ctx"], d["toks"], d["olen"], anchor, ctx_cap,
                       path=None if path is None else cuda_i32(path), draft_ctx=dctx, status=status)
    torch.cuda.synchronize()
    assert S.sd_fault_word() & BAD_COMMIT
    st = want["status"]
    assert st[5] == st[6] == st[7] == st[8] == 1 and (not tree or st[9] == 1)
    assert status.cpu().numpy().tolist() == st.tolist()
    assert d["ctx"].cpu().numpy().tolist() == want["ctx_len"].tolist()
    assert d["olen"].cpu().numpy().tolist() == want["out_len"].tolist()
    assert np.array_equal(d["toks"].cpu().numpy(), want["out_tokens"])
    got_anchor = anchor.cpu().numpy()
    assert got_anchor.tolist() == want["anchor"].tolist()
    ok = st == 0
    assert (dctx.cpu().numpy()[ok] == want["draft_ctx"][ok]).all()
    assert (dctx.cpu().numpy()[~ok] == -5).all()


@pytest.mark.parametrize("dtype,D,strided,T", [(torch.bfloat16, 128, False, 16), (torch.bfloat16, 128, True, 16),
                                               (torch.float32, 64, False, 16), (torch.bfloat16, 128, True, 60)])
def test_compact_tree_kv_matches_oracle(S, dtype, D, strided, T):
    rng = np.random.default_rng(D + strided + (T if T > 16 else 0))
    B, Sl, Hkv = 5, 160, 4
    _, _, _, n, _, path = random_paths(rng, B, T)
    if T > 16:
        n, path = deep_first(n, path, T)
        # sequence 4: a deep path over every other node
        path[4, :] = -1
        path[4, :T // 2 - 1] = np.arange(2, T, 2)[: T // 2 - 1]
        n[4] = T // 2 - 1
    ctx = rng.integers(1, Sl - T + 2, B).astype(np.int32)
    ctx[0] = 1
    ctx[1] = Sl - T + 1                     # block ends at the last position
    ctx[2] = Sl - T + 2                     # one past: skipped, flagged
    n[3] = 15 if n[3] == 0 else n[3]
    extra = 8 if strided else 0
    big_k = torch.randn(B, Sl + extra, Hkv, D).to(dtype).cuda()
    big_v = torch.randn(B, Sl + extra, Hkv, D).to(dtype).cuda()
    k, v = big_k[:, :Sl], big_v[:, :Sl]
    pad_k, pad_v = big_k[:, Sl:].cpu(), big_v[:, Sl:].cpu()
    iv = torch.int16 if dtype == torch.bfloat16 else torch.int32
    k0 = k.cpu().contiguous().view(iv).numpy()
    v0 = v.cpu().contiguous().view(iv).numpy()
    wk, wv, st = oracle.compact_tree_kv(k0, v0, ctx, path, n)
    assert st.tolist() == [0, 0, 1, 0, 0]
    S.sd_fault_word(clear=True)
    S.sd_compact_tree_kv(k, v, cuda_i32(ctx), cuda_i32(path), cuda_i32(n))
    torch.cuda.synchronize()
    assert S.sd_fault_word() & BAD_COMMIT
    assert np.array_equal(k.cpu().contiguous().view(iv).numpy(), wk)
    assert np.array_equal(v.cpu().contiguous().view(iv).numpy(), wv)
    # the padding positions between sequences are never touched
    assert torch.equal(big_k[:, Sl:].cpu(), pad_k) and torch.equal(big_v[:, Sl:].cpu(), pad_v)


@pytest.mark.parametrize("tree,T", [(False, 16), (True, 16), (True, 60)])
def test_project_kv_commit_matches_oracle(S, tree, T):
    rng = np.random.default_rng(11 + tree + (T if T > 16 else 0))
    B, Hd, Dout, Sd = 4, 512, 256, 100
    g = torch.Generator().manual_seed(5)
    hid = torch.randn(B, T, Hd, generator=g).to(torch.bfloat16)
    wk = (torch.randn(Dout, Hd, generator=g) * 0.05).to(torch.bfloat16)
    wv = (torch.randn(Dout, Hd, generator=g) * 0.05).to(torch.bfloat16)
    if tree:
        _, _, _, n, _, path = random_paths(rng, B, T)
        if T > 16:
            n, path = deep_first(n, path, T)   # 60 rows: four row groups of 16
    else:
        n, path = np.array([0, 7, 15, 3], np.int32), None
    d0 = np.array([10, 50, Sd - 1 - int(n[2]), Sd - int(n[3])], np.int32)   # last: one row too many
    kc = torch.full((B, Sd, Dout), -2.0, dtype=torch.bfloat16, device="cuda")
    vc = torch.full((B, Sd, Dout), -2.0, dtype=torch.bfloat16, device="cuda")
    S.sd_fault_word(clear=True)
    S.sd_project_kv_commit(hid.cuda(), wk.cuda(), wv.cuda(), cuda_i32(n), cuda_i32(d0), kc, vc,
                           path=None if path is None else cuda_i32(path))
    torch.cuda.synchronize()
    assert S.sd_fault_word() & BAD_COMMIT
    kc, vc = kc.cpu(), vc.cpu()
    for b in range(B):
        m = int(n[b]) + 1
        if b == 3:
            assert (kc[b] == -2.0).all() and (vc[b] == -2.0).all()
            continue
        src = [0] + [int(path[b, r - 1]) if tree else r for r in range(1, m)]
        rows = slice(int(d0[b]), int(d0[b]) + m)
        check_projection(kc[b, rows], hid[b], wk, np.array(src))
        check_projection(vc[b, rows], hid[b], wv, np.array(src))
        assert (kc[b, :d0[b]] == -2.0).all() and (kc[b, d0[b] + m:] == -2.0).all()
        assert (vc[b, :d0[b]] == -2.0).all() and (vc[b, d0[b] + m:] == -2.0).all()


@pytest.mark.parametrize("tree", [False, True])
def test_cycles_in_one_cuda_graph_match_the_oracle(S, tree):
    """accept -> (compact) -> append -> commit, captured once and replayed
    `cycles` times; the oracle runs the same cycles one by one."""
    rng = np.random.default_rng(21 + tree)
    B, T, V, Hd, Hkv, D, cycles = 2, 16, 3000, 256, 2, 64, 6
    Dout = Hkv * D
    g = torch.Generator().manual_seed(7)
    logits = (torch.randn(B, T, V, generator=g) * 3).to(torch.bfloat16)
    am = logits.float().argmax(-1).numpy()
    if tree:
        parents = np.zeros((B, T), np.int32)
        parents[:, 0] = -1
        for j in range(1, T):
            parents[:, j] = rng.integers(max(0, j - 3), j, B)
        prop = np.array([[0] + [int(am[b, parents[b, j]]) if rng.random() < 0.75 else int(rng.integers(0, V))
                               for j in range(1, T)] for b in range(B)], np.int32)
    else:
        prop = np.array([[int(am[b, j]) if j < 4 + 5 * b else int(rng.integers(0, V)) for j in range(T - 1)]
                         for b in range(B)], np.int32)
    hid = torch.randn(B, T, Hd, generator=g).to(torch.bfloat16)
    wk = (torch.randn(Dout, Hd, generator=g) * 0.05).to(torch.bfloat16)
    wv = (torch.randn(Dout, Hd, generator=g) * 0.05).to(torch.bfloat16)
    Sl, Sd, cap = 200, 200, 120
    kc = torch.randn(B, Sl, Hkv, D).to(torch.bfloat16)
    vc = torch.randn(B, Sl, Hkv, D).to(torch.bfloat16)
    ctx0 = np.array([5, 30], np.int32)
    # device state
    dk, dv = kc.cuda(), vc.cuda()
    dkd = torch.zeros(B, Sd, Dout, dtype=torch.bfloat16, device="cuda")
    dvd = torch.zeros_like(dkd)
    dctx, ddctx = cuda_i32(ctx0), cuda_i32(ctx0 - 1)
    dtoks = torch.full((B, cap), -1, dtype=torch.int32, device="cuda")
    dolen = torch.zeros(B, dtype=torch.int32, device="cuda")
    danchor = torch.full((B,), -1, dtype=torch.int32, device="cuda")
    dn = torch.zeros(B, dtype=torch.int32, device="cuda")
    dc = torch.zeros(B, dtype=torch.int32, device="cuda")
    dpath = torch.zeros(B, T, dtype=torch.int32, device="cuda")
    dprop, dlog, dhid = cuda_i32(prop), logits.cuda(), hid.cuda()
    dparents = cuda_i32(parents) if tree else None
    dwk, dwv = wk.cuda(), wv.cuda()
    if tree:
        ws = S.workspace(S.sd_accept_tree_greedy_workspace_size(B, T, V))
    else:
        ws = S.workspace(S.sd_accept_greedy_workspace_size(B, T, V))

    def cycle():
        if tree:
            S.sd_accept_tree_greedy(dprop, dparents, dlog, dn, dc, dpath, ws)
            S.sd_compact_tree_kv(dk, dv, dctx, dpath, dn)
        else:
            S.sd_accept_greedy(dprop, dlog, dn, dc, ws)
        S.sd_project_kv_commit(dhid, dwk, dwv, dn, ddctx, dkd, dvd, path=dpath if tree else None)
        S.sd_commit_tokens(dprop, dn, dc, dctx, dtoks, dolen, danchor, Sl - T + 1,
                           path=dpath if tree else None, draft_ctx=ddctx)

    S.sd_fault_word(clear=True)
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(st):
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=st):
            cycle()
        for _ in range(cycles):
            graph.replay()
    torch.cuda.synchronize()
    assert S.sd_fault_word() == 0

    # the oracle, cycle by cycle
    ctx, toks, olen = ctx0.copy(), np.full((B, cap), -1, np.int32), np.zeros(B, np.int32)
    dctx_o = ctx0 - 1
    k_np = kc.view(torch.int16).numpy().copy()
    v_np = vc.view(torch.int16).numpy().copy()
    rows = {b: {} for b in range(B)}
    anchor = None
    for _ in range(cycles):
        if tree:
            n, c, _, path = oracle.accept_tree_greedy(prop, parents, logits)
            k_np, v_np, cst = oracle.compact_tree_kv(k_np, v_np, ctx, path, n)
            assert (cst == 0).all()
        else:
            n, c = oracle.accept_greedy(prop, logits)
            path = None
        for b in range(B):
            for r in range(int(n[b]) + 1):
                rows[b][int(dctx_o[b]) + r] = 0 if r == 0 else (int(path[b, r - 1]) if tree else r)
        res = oracle.commit_tokens(prop, n, c, ctx, toks, olen, Sl - T + 1, path=path)
        assert (res["status"] == 0).all()
        ctx, toks, olen, dctx_o, anchor = res["ctx_len"], res["out_tokens"], res["out_len"], res["draft_ctx"], \
            res["anchor"]
    assert dctx.cpu().numpy().tolist() == ctx.tolist()
    assert ddctx.cpu().numpy().tolist() == dctx_o.tolist()
    assert dolen.cpu().numpy().tolist() == olen.tolist()
    assert np.array_equal(dtoks.cpu().numpy(), toks)
    assert danchor.cpu().numpy().tolist() == anchor.tolist()
    assert np.array_equal(dk.cpu().view(torch.int16).numpy(), k_np)
    assert np.array_equal(dv.cpu().view(torch.int16).numpy(), v_np)
    kd, vd = dkd.cpu(), dvd.cpu()
    for b in range(B):
        pos = sorted(rows[b])
        assert pos == list(range(int(ctx0[b]) - 1, int(ctx[b]) - 1))
        src = np.array([rows[b][p] for p in pos])
        check_projection(kd[b, pos], hid[b], wk, src)
        check_projection(vd[b, pos], hid[b], wv, src)
        assert (kd[b, :pos[0]] == 0).all() and (kd[b, pos[-1] + 1:] == 0).all()
