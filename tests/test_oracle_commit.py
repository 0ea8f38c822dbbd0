"""Pins of the oracle's commit / rollback routines.

Fixed to things other than their own formulas: the worked cycle of the
VFlash-FM project page (7 accepted, 8 committed, the correction becomes the
next anchor), chain/tree agreement, rejection of commits that do not fit,
and the lossless property over many cycles -- chain and tree speculation
with a toy language model commit exactly the tokens of autoregressive greedy
decoding, the compacted KV cache holds exactly the rows autoregressive
decoding would have written, and the drafter context appended a few rows per
cycle equals the projection of the whole committed sequence at once.
"""
import json
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_cycle.json")


def _state(B, out_cap, ctx0=10):
    return (np.full(B, ctx0, dtype=np.int32), np.full((B, out_cap), -7, dtype=np.int32),
            np.zeros(B, dtype=np.int32))


def test_worked_cycle_commits_prefix_and_correction():
    g = json.load(open(GOLDEN))
    V = g["vocab"]
    logits = np.zeros((1, 16, V))
    for j, t in enumerate(g["target_choice"]):
        logits[0, j, t] = 1.0
    draft = np.array([g["draft"]], dtype=np.int32)
    n, c = oracle.accept_greedy(draft, logits)
    ctx, toks, olen = _state(1, 40, ctx0=25_119)
    r = oracle.commit_tokens(draft, n, c, ctx, toks, olen, ctx_cap=1 << 20)
    e = g["expect"]
    assert r["status"][0] == 0
    assert r["out_len"][0] == e["committed"] == 8
    assert list(r["out_tokens"][0, :8]) == g["draft"][:7] + [e["correction"]]
    assert (r["out_tokens"][0, 8:] == -7).all()
    assert r["anchor"][0] == e["next_anchor"]
    assert r["ctx_len"][0] == 25_119 + 8 and r["draft_ctx"][0] == 25_119 + 7


def test_commit_appends_after_earlier_output_and_leaves_it():
    rng = np.random.default_rng(1)
    B, T, cap = 30, 16, 200
    draft = rng.integers(0, 1000, (B, T - 1)).astype(np.int32)
    n = rng.integers(0, T, B).astype(np.int32)
    nx = rng.integers(0, 1000, B).astype(np.int32)
    ctx = rng.integers(1, 5000, B).astype(np.int32)
    olen = rng.integers(0, 50, B).astype(np.int32)
    toks = rng.integers(0, 1000, (B, cap)).astype(np.int32)
    r = oracle.commit_tokens(draft, n, nx, ctx, toks, olen, ctx_cap=1 << 20)
    assert (r["status"] == 0).all()
    for b in range(B):
        k = int(n[b])
        assert r["out_len"][b] - olen[b] == r["ctx_len"][b] - ctx[b] == k + 1
        assert list(r["out_tokens"][b, olen[b]:olen[b] + k + 1]) == list(draft[b, :k]) + [nx[b]]
        assert (r["out_tokens"][b, :olen[b]] == toks[b, :olen[b]]).all()
        assert (r["out_tokens"][b, olen[b] + k + 1:] == toks[b, olen[b] + k + 1:]).all()
    assert (r["anchor"] == nx).all() and (r["draft_ctx"] == r["ctx_len"] - 1).all()


def test_chain_commit_equals_tree_commit_with_a_chain_path():
    rng = np.random.default_rng(2)
    B, T = 12, 16
    draft = rng.integers(0, 500, (B, T - 1)).astype(np.int32)
    tokens = np.concatenate([np.zeros((B, 1), np.int32), draft], axis=1)
    n = rng.integers(0, T, B).astype(np.int32)
    path = np.full((B, T), -1, dtype=np.int32)
    for b in range(B):
        path[b, :n[b]] = np.arange(1, n[b] + 1)
    nx = rng.integers(0, 500, B).astype(np.int32)
    ctx, toks, olen = _state(B, 64)
    a = oracle.commit_tokens(draft, n, nx, ctx, toks, olen, 1 << 20)
    t = oracle.commit_tokens(tokens, n, nx, ctx, toks, olen, 1 << 20, path=path)
    for key in a:
        assert np.array_equal(a[key], t[key]), key


@pytest.mark.parametrize("case", ["ctx_cap", "out_cap", "bad_n", "bad_path"])
def test_commit_that_does_not_fit_leaves_the_sequence_alone(case):
    B, T = 3, 16
    draft = np.arange(B * (T - 1), dtype=np.int32).reshape(B, T - 1)
    tokens = np.concatenate([np.zeros((B, 1), np.int32), draft], axis=1)
    n = np.array([4, 15, 0], dtype=np.int32)
    nx = np.array([100, 101, 102], dtype=np.int32)
    ctx, toks, olen = _state(B, 30)
    path = np.tile(np.arange(1, T + 1, dtype=np.int32), (B, 1))
    path[:, T - 1] = -1
    ctx_cap = 1 << 20
    if case == "ctx_cap":
        ctx_cap = 10 + 15          # sequence 1 would reach 26
    elif case == "out_cap":
        olen[1] = 30 - 15          # 16 more tokens do not fit in 30
    elif case == "bad_n":
        n[1] = 16
    else:
        path[1, 3] = 0             # node 0 (the anchor) cannot be a kept proposal
    r = oracle.commit_tokens(tokens, n, nx, ctx, toks, olen, ctx_cap,
                             path=path if case == "bad_path" else None) if case == "bad_path" else \
        oracle.commit_tokens(draft, n, nx, ctx, toks, olen, ctx_cap)
    assert list(r["status"]) == [0, 1, 0]
    assert r["ctx_len"][1] == ctx[1] and r["out_len"][1] == olen[1] and r["anchor"][1] == -1
    assert (r["out_tokens"][1] == toks[1]).all()
    assert r["ctx_len"][0] == 15 and r["ctx_len"][2] == 11


def _toy_lm(prefix, V=12):
    h = hash(tuple(prefix)) & 0xFFFFFFFF
    return np.random.default_rng(h).standard_normal(V) * 2.0


def _toy_row(token, pos, width):
    """A deterministic stand-in for the K (or V, or hidden) row a forward
    writes for `token` at position `pos`."""
    return np.random.default_rng(1_000_003 * (token + 1) + pos).standard_normal(width)


def _ar(prompt, n_new, V):
    ar = list(prompt)
    while len(ar) < len(prompt) + n_new:
        ar.append(int(np.argmax(_toy_lm(ar, V))))
    return ar


def test_chain_cycles_commit_autoregressive_tokens_and_drafter_context():
    """Chain speculation over many cycles with device-style state: ctx_len,
    out_tokens, the anchor, and the drafter's context (hidden rows 0..n of
    each block appended at draft_ctx) -- the last equals projecting the
    hidden rows of the whole committed sequence in one prefill call."""
    V, T, n_new, Hd, Dout = 12, 16, 90, 24, 8
    prompt = [3, 1, 4]
    ar = _ar(prompt, n_new + 40, V)
    rng = np.random.default_rng(5)
    w = rng.standard_normal((Dout, Hd))
    # state after prefill: the prompt is context, ar[len(prompt)] the first anchor
    ctx = np.array([len(prompt) + 1], np.int32)
    out_cap = n_new + 2 * T
    toks = np.full((1, out_cap), -1, np.int32)
    olen = np.zeros(1, np.int32)
    anchor = ar[len(prompt)]
    drafter_cache = np.full((len(prompt) + out_cap + T, Dout), np.nan)
    drafter_cache[:len(prompt)] = oracle.project_rows(
        np.stack([_toy_row(t, p, Hd) for p, t in enumerate(prompt)]), w)
    draft_ctx = np.array([len(prompt)], np.int32)
    cycles = 0
    while olen[0] < n_new:
        seq = ar[:ctx[0]]                       # committed tokens incl. the anchor
        assert seq[-1] == anchor
        pos0 = ctx[0] - 1
        right = [ar[pos0 + 1 + i] if pos0 + 1 + i < len(ar) else 0 for i in range(T - 1)]
        draft = [r if rng.random() < 0.75 else int(rng.integers(0, V)) for r in right]
        block = [anchor] + draft
        logits = np.stack([_toy_lm(seq + draft[:j], V) for j in range(T)])[None]
        n, c = oracle.accept_greedy(np.array([draft], np.int32), logits)
        # the drafter appends hidden rows 0..n of the block (anchor + kept)
        hid = np.stack([_toy_row(block[j], pos0 + j, Hd) for j in range(T)])
        rows = oracle.project_rows(hid, w, np.arange(n[0] + 1))
        drafter_cache[draft_ctx[0]:draft_ctx[0] + n[0] + 1] = rows
        r = oracle.commit_tokens(np.array([draft], np.int32), n, c, ctx, toks, olen, 1 << 20)
        assert r["status"][0] == 0
        ctx, toks, olen, anchor, draft_ctx = r["ctx_len"], r["out_tokens"], r["out_len"], r["anchor"][0], \
            r["draft_ctx"]
        cycles += 1
    assert list(toks[0, :olen[0]]) == ar[len(prompt) + 1:len(prompt) + 1 + olen[0]]
    assert ctx[0] == len(prompt) + 1 + olen[0] and draft_ctx[0] == ctx[0] - 1
    committed = ar[:ctx[0] - 1]
    want = oracle.project_rows(np.stack([_toy_row(t, p, Hd) for p, t in enumerate(committed)]), w)
    assert np.allclose(drafter_cache[:ctx[0] - 1], want, rtol=0, atol=1e-12)
    assert cycles < n_new // 2


def test_chain_path_compaction_moves_nothing():
    rng = np.random.default_rng(7)
    B, S, Hkv, D, T = 3, 64, 2, 8, 16
    k = rng.integers(-30000, 30000, (B, S, Hkv, D)).astype(np.int16)
    v = rng.integers(-30000, 30000, (B, S, Hkv, D)).astype(np.int16)
    n = np.array([0, 7, 15], np.int32)
    path = np.full((B, T), -1, np.int32)
    for b in range(B):
        path[b, :n[b]] = np.arange(1, n[b] + 1)
    k2, v2, st = oracle.compact_tree_kv(k, v, np.array([5, 20, 40], np.int32), path, n)
    assert (st == 0).all() and np.array_equal(k2, k) and np.array_equal(v2, v)


def test_compaction_by_hand_and_bounds():
    # one head, D = 1, cache positions hold their own index; ctx = 4, so block
    # slot k is position 3 + k; kept nodes 2, 5, 6 land at positions 4, 5, 6
    k = np.arange(20, dtype=np.float32).reshape(1, 20, 1, 1)
    v = -k
    path = np.array([[2, 5, 6] + [-1] * 5], np.int32)
    k2, v2, st = oracle.compact_tree_kv(k, v, np.array([4], np.int32), path, np.array([3], np.int32))
    want = np.arange(20, dtype=np.float32)
    want[4:7] = [3 + 2, 3 + 5, 3 + 6]
    assert st[0] == 0 and list(k2.reshape(-1)) == list(want) and list(v2.reshape(-1)) == list(-want)
    # block past the cache end, bad node: untouched, flagged
    for ctx, p in ((14, path), (4, np.array([[2, 0, 6] + [-1] * 5], np.int32))):
        k3, _, st = oracle.compact_tree_kv(k, v, np.array([ctx], np.int32), p, np.array([3], np.int32))
        assert st[0] == 1 and np.array_equal(k3, k)


def test_tree_cycles_leave_the_cache_autoregressive():
    """Tree speculation for many cycles: node j's K/V row is written at block
    slot j for position ctx-1+depth(j); after compaction and commit, cache
    positions [0, ctx-1) hold exactly the rows autoregressive decoding writes
    (token at p, position p), and the committed tokens are the greedy ones."""
    V, n_new, Hkv, D = 12, 70, 2, 4
    prompt = [2, 9, 4]
    ar = _ar(prompt, n_new + 40, V)
    rng = np.random.default_rng(11)
    S = len(prompt) + n_new + 40
    width = Hkv * D
    kc = np.zeros((1, S, Hkv, D))
    vc = np.zeros((1, S, Hkv, D))
    for p, t in enumerate(prompt):
        kc[0, p] = _toy_row(t, p, width).reshape(Hkv, D)
        vc[0, p] = -_toy_row(t, p, width).reshape(Hkv, D)
    ctx = np.array([len(prompt) + 1], np.int32)
    toks = np.full((1, n_new + 40), -1, np.int32)
    olen = np.zeros(1, np.int32)
    anchor = ar[len(prompt)]
    while olen[0] < n_new:
        seq = ar[:ctx[0]]
        pos0 = ctx[0] - 1
        parents, tokens, depth, paths = [-1], [anchor], [0], [[]]
        main = 0
        for lvl in range(1, 6):
            q = pos0 + lvl
            right = ar[q] if q < len(ar) else 0
            cands = [right if rng.random() < 0.6 else int(rng.integers(0, V)),
                     right if rng.random() < 0.5 else int(rng.integers(0, V)),
                     int(rng.integers(0, V))]
            first = len(parents)
            for t in cands:
                parents.append(main)
                tokens.append(t)
                depth.append(lvl)
                paths.append(paths[main] + [t])
            main = first + int(rng.integers(0, 3))
        T = len(parents)
        for j in range(T):   # the target's forward writes node j at slot j
            kc[0, pos0 + j] = _toy_row(tokens[j], pos0 + depth[j], width).reshape(Hkv, D)
            vc[0, pos0 + j] = -_toy_row(tokens[j], pos0 + depth[j], width).reshape(Hkv, D)
        logits = np.stack([_toy_lm(seq + paths[j], V) for j in range(T)])[None]
        n, c, best, path = oracle.accept_tree_greedy(np.array([tokens]), np.array([parents]), logits)
        kc, vc, st = oracle.compact_tree_kv(kc, vc, ctx, path, n)
        assert st[0] == 0
        r = oracle.commit_tokens(np.array([tokens], np.int32), n, c, ctx, toks, olen, S - T + 1, path=path)
        assert r["status"][0] == 0
        ctx, toks, olen, anchor = r["ctx_len"], r["out_tokens"], r["out_len"], int(r["anchor"][0])
    assert list(toks[0, :olen[0]]) == ar[len(prompt) + 1:len(prompt) + 1 + olen[0]]
    for p in range(ctx[0] - 1):
        assert np.array_equal(kc[0, p].reshape(-1), _toy_row(ar[p], p, width)), p
        assert np.array_equal(vc[0, p].reshape(-1), -_toy_row(ar[p], p, width)), p
