"""Pins for the oracle's tree verification ("VFlash-FM" project page, speedup
table: its fastest variant verifies a draft tree, "Tree-60", instead of a
chain).

The pages give no tree layout; the reading here (also in the oracle):
the block's T slots are the tree's nodes in topological order, node 0 the
anchor, with their K/V at cache slots ctx-1 .. ctx-2+T as in the chain case.
Node j attends to the context before the anchor and to the slots of its
ancestors and itself (a bitmask per node).  Greedy tree acceptance keeps the
deepest node whose whole root path matches the target's greedy picks.

The pins: a chain-shaped tree gives exactly the chain oracle (same keys, same
order); torch's scaled_dot_product_attention with an explicit boolean mask on
random trees; a hand-checked acceptance example; and the lossless property
(tree speculation reproduces autoregressive greedy decoding with a toy LM).
"""
import numpy as np
import pytest
import torch

import oracle
from serving_sd_verify_gb300 import workloads as W


def _random_tree(rng, T):
    parents = np.full(T, -1, dtype=np.int32)
    for j in range(1, T):
        parents[j] = rng.integers(0, j)
    return parents


def _masks_from_parents(parents):
    T = len(parents)
    m = np.zeros(T, dtype=np.uint64)
    for j in range(T):
        v = j
        bits = 0
        while v != -1:
            bits |= 1 << int(v)
            v = parents[v]
        m[j] = np.uint64(bits)
    return m


def _chain_parents(T):
    return np.arange(-1, T - 1, dtype=np.int32)


@pytest.mark.parametrize("T", [6, 60, 64])
def test_chain_tree_equals_chain_attention_exactly(T):
    """A chain of up to 64 nodes (mask bits up to 63) is the chain verify."""
    inp = W.verify_inputs(B=2, T=T, Hq=4, Hkv=2, D=8, ctx=[7, 3], dtype=torch.float32, seed=11)
    B = 2
    mask = np.stack([_masks_from_parents(_chain_parents(T))] * B)
    got = oracle.tree_attention_rows(inp["q"], inp["k"], inp["v"], inp["ctx"], mask, 0.3)
    want = oracle.attention_rows(inp["q"], inp["k"], inp["v"], inp["ctx"], 0.3, mode=0)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("seed,T", [(0, 8), (1, 8), (2, 8), (3, 60), (4, 64)])
def test_random_trees_match_sdpa_with_the_ancestor_mask(seed, T):
    rng = np.random.default_rng(seed)
    B, Hq, Hkv, D = 2, 6, 2, 16
    ctx = [5, 12]
    inp = W.verify_inputs(B=B, T=T, Hq=Hq, Hkv=Hkv, D=D, ctx=ctx, dtype=torch.float32, seed=20 + seed)
    parents = np.stack([_random_tree(rng, T) for _ in range(B)])
    mask = np.stack([_masks_from_parents(p) for p in parents])
    got = oracle.tree_attention_rows(inp["q"], inp["k"], inp["v"], inp["ctx"], mask, 0.25)
    G = Hq // Hkv
    want = np.zeros((B, T, Hq, D))
    for b in range(B):
        n = ctx[b]
        L = n - 1 + T
        am = torch.zeros(T, L, dtype=torch.bool)
        am[:, : n - 1] = True
        for j in range(T):
            for k in range(T):
                if (int(mask[b, j]) >> k) & 1:
                    am[j, n - 1 + k] = True
        q = inp["q"][b].double().permute(1, 0, 2)                    # [Hq, T, D]
        kk = inp["k"][b, :L].double().permute(1, 0, 2).repeat_interleave(G, 0)
        vv = inp["v"][b, :L].double().permute(1, 0, 2).repeat_interleave(G, 0)
        o = torch.nn.functional.scaled_dot_product_attention(q, kk, vv, attn_mask=am, scale=0.25)
        want[b] = o.permute(1, 0, 2).numpy()
    assert np.abs(got - want.reshape(-1, D)).max() < 1e-12


def test_last_of_64_nodes_sees_only_context_anchor_and_itself():
    """Mask bit 63: in a 64-node star, node 63 attends to the context, the
    anchor and itself, which equals plain attention over those keys."""
    T, n = 64, 10
    inp = W.verify_inputs(B=1, T=T, Hq=2, Hkv=1, D=8, ctx=[n], dtype=torch.float32, seed=6)
    parents = np.array([-1] + [0] * (T - 1), dtype=np.int32)
    mask = _masks_from_parents(parents)[None]
    assert int(mask[0, 63]) == (1 << 63) | 1
    got = oracle.tree_attention_rows(inp["q"], inp["k"], inp["v"], inp["ctx"], mask, 0.5).reshape(T, 2, 8)
    keys = list(range(n)) + [n - 1 + 63]
    for h in range(2):
        qv = inp["q"][0, 63, h].double().numpy()
        kk = inp["k"][0, keys, 0].double().numpy()
        vv = inp["v"][0, keys, 0].double().numpy()
        s_ = 0.5 * kk @ qv
        w = np.exp(s_ - s_.max())
        want = (w / w.sum()) @ vv
        assert np.abs(got[63, h] - want).max() < 1e-12


def test_star_tree_node_sees_context_anchor_and_itself():
    """Perturbing a sibling's K/V leaves a node unchanged; perturbing the anchor's does not."""
    inp = W.verify_inputs(B=1, T=5, Hq=2, Hkv=1, D=8, ctx=[9], dtype=torch.float32, seed=5)
    parents = np.array([-1, 0, 0, 0, 0], dtype=np.int32)
    mask = _masks_from_parents(parents)[None]
    base = oracle.tree_attention_rows(inp["q"], inp["k"], inp["v"], inp["ctx"], mask, 0.5).reshape(5, 2, 8)
    k2 = inp["k"].clone()
    k2[0, 9 - 1 + 2] += 3.0                      # node 2's key
    pert = oracle.tree_attention_rows(inp["q"], k2, inp["v"], inp["ctx"], mask, 0.5).reshape(5, 2, 8)
    assert np.array_equal(pert[[0, 1, 3, 4]], base[[0, 1, 3, 4]])
    assert not np.array_equal(pert[2], base[2])
    k3 = inp["k"].clone()
    k3[0, 9 - 1] += 3.0                          # the anchor's key
    pert = oracle.tree_attention_rows(inp["q"], k3, inp["v"], inp["ctx"], mask, 0.5).reshape(5, 2, 8)
    assert all(not np.array_equal(pert[j], base[j]) for j in range(5))


def test_chain_tree_acceptance_equals_chain_greedy():
    for seed in range(5):
        inp = W.greedy_inputs(B=3, T=16, V=500, seed=seed)
        B, T = 3, 16
        tokens = np.zeros((B, T), dtype=np.int32)
        tokens[:, 1:] = inp["draft"].numpy()
        parents = np.stack([_chain_parents(T)] * B)
        n, c, best, path = oracle.accept_tree_greedy(tokens, parents, inp["logits"])
        n2, c2 = oracle.accept_greedy(inp["draft"], inp["logits"])
        assert (n == n2).all() and (c == c2).all()
        assert (best == n).all()
        for b in range(B):
            assert list(path[b, : n[b]]) == list(range(1, n[b] + 1)) and (path[b, n[b]:] == -1).all()


def test_tree_acceptance_hand_example():
    # node:     0   1   2   3   4   5   6
    # parent:  -1   0   0   1   1   2   3
    V = 10
    parents = np.array([[-1, 0, 0, 1, 1, 2, 3]], dtype=np.int32)
    amax = [5, 7, 3, 4, 1, 8, 2]            # the target's greedy pick after each node
    logits = np.zeros((1, 7, V))
    for j, a in enumerate(amax):
        logits[0, j, a] = 1.0
    # node 1 = 5 = a_0 (accepted), node 2 = 9 != a_0 (rejected), node 3 = 7 = a_1 (accepted),
    # node 4 = 2 != a_1 (rejected), node 5 = 3 = a_2 but its parent is rejected,
    # node 6 = 0 != a_3 (rejected): the deepest accepted node is 3, depth 2
    tokens = np.array([[0, 5, 9, 7, 2, 3, 0]], dtype=np.int32)
    n, c, best, path = oracle.accept_tree_greedy(tokens, parents, logits)
    assert n[0] == 2 and best[0] == 3 and c[0] == amax[3]
    assert list(path[0]) == [1, 3, -1, -1, -1, -1, -1]
    # equal depths: the lower node index wins
    tokens2 = np.array([[0, 5, 5, 7, 2, 3, 0]], dtype=np.int32)   # node 2 also accepted; node 5 = 3 = a_2
    n, c, best, path = oracle.accept_tree_greedy(tokens2, parents, logits)
    assert n[0] == 2 and best[0] == 3          # nodes 3 and 5 both at depth 2: node 3
    assert list(path[0, :2]) == [1, 3]


def _toy_lm(prefix, V=12):
    h = hash(tuple(prefix)) & 0xFFFFFFFF
    return np.random.default_rng(h).standard_normal(V) * 2.0


def test_tree_speculation_reproduces_autoregressive_decoding():
    """Each cycle drafts a two-branch tree (two candidates per level, chained
    under the first); the committed tokens equal greedy decoding."""
    V, n_new = 12, 80
    prompt = [2, 9, 4]
    ar = list(prompt)
    while len(ar) < len(prompt) + n_new:
        ar.append(int(np.argmax(_toy_lm(ar, V))))
    rng = np.random.default_rng(3)
    seq = list(prompt)
    cycles, depths = 0, []
    while len(seq) < len(prompt) + n_new:
        # nodes: 0 anchor; level l (1..7) has a main node and a side node,
        # both children of the previous main node
        parents, tokens, paths = [-1], [0], [[]]
        main = 0
        for lvl in range(1, 8):
            pos = len(seq) + lvl - 1
            right = ar[pos] if pos < len(ar) else 0
            cands = [right if rng.random() < 0.6 else int(rng.integers(0, V)),
                     right if rng.random() < 0.5 else int(rng.integers(0, V))]
            first = len(parents)
            for t in cands:
                parents.append(main)
                tokens.append(t)
                paths.append(paths[main] + [t])
            main = first
        T = len(parents)
        logits = np.stack([_toy_lm(seq + paths[j], V) for j in range(T)])[None]
        n, c, best, path = oracle.accept_tree_greedy(np.array([tokens]), np.array([parents]), logits)
        toks = [tokens[v] for v in path[0, : n[0]]]
        seq += toks + [int(c[0])]
        cycles += 1
        depths.append(int(n[0]))
    assert seq[: len(ar)] == ar[: len(seq)]
    assert cycles < n_new and len(set(depths)) > 1
