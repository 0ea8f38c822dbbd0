"""Pins for the oracle's attention (target verify and drafter block attention).

Each test fixes the oracle to something other than itself: a hand-computed
example, closed forms, torch's scaled_dot_product_attention (a library
routine) on the special cases it covers, and structural invariants of the
causal-within-block mask ("VFlash-FM" project page, "How VFlash-FM works":
the target scores all 16 block slots in one forward, so slot j may only see
what precedes it).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from serving_sd_verify_gb300 import workloads as W


def _flat_rows(B, T, Hq):
    return np.arange(B * T * Hq)


def _sdpa_reference(q, k, v, nctx, scale, mode, kb=None, vb=None):
    """torch SDPA (fp64, CPU) with an explicit boolean mask per sequence."""
    B, T, Hq, D = q.shape
    Hkv = k.shape[2]
    G = Hq // Hkv
    outs = []
    for b in range(B):
        n = int(nctx[b])
        if mode == 0:
            kk = k[b, : n + T - 1].double()
            vv = v[b, : n + T - 1].double()
            L = n + T - 1
            mask = torch.zeros(T, L, dtype=torch.bool)
            for j in range(T):
                mask[j, : n + j] = True
        else:
            kk = torch.cat([k[b, :n], kb[b]], 0).double()
            vv = torch.cat([v[b, :n], vb[b]], 0).double()
            mask = torch.ones(T, n + T, dtype=torch.bool)
        # [heads, L, D] with the kv head of query head h = h // G
        kk = kk.permute(1, 0, 2).repeat_interleave(G, 0)
        vv = vv.permute(1, 0, 2).repeat_interleave(G, 0)
        qq = q[b].double().permute(1, 0, 2)  # [Hq, T, D]
        o = torch.nn.functional.scaled_dot_product_attention(
            qq, kk, vv, attn_mask=mask.unsqueeze(0), scale=scale)
        outs.append(o.permute(1, 0, 2))  # [T, Hq, D]
    return torch.stack(outs).reshape(-1, D).numpy()


def test_hand_computed_example():
    # one head, D = 1, scale 1, q = 1: weights are exp(k) / sum exp(k)
    # keys 0, ln2, ln3 -> weights 1/6, 2/6, 3/6; values 6, 0, 12
    # ctx = 2, T = 2: row 0 sees 2 keys -> (1*6 + 2*0)/3 = 2; row 1 sees 3 -> 1 + 0 + 6 = 7
    q = np.ones((1, 2, 1, 1))
    k = np.array([0.0, math.log(2.0), math.log(3.0)]).reshape(1, 3, 1, 1)
    v = np.array([6.0, 0.0, 12.0]).reshape(1, 3, 1, 1)
    out, lse = oracle.attention_rows(q, k, v, [2], 1.0, return_lse=True)
    assert out[0, 0] == pytest.approx(2.0, abs=1e-14)
    assert out[1, 0] == pytest.approx(7.0, abs=1e-14)
    assert lse[0] == pytest.approx(math.log(3.0), abs=1e-14)
    assert lse[1] == pytest.approx(math.log(6.0), abs=1e-14)


def test_single_key_returns_that_value():
    # T = 1, ctx = 1: ordinary decode over one key returns v exactly
    rng = np.random.default_rng(0)
    q = rng.standard_normal((2, 1, 4, 8))
    k = rng.standard_normal((2, 3, 2, 8))
    v = rng.standard_normal((2, 3, 2, 8))
    out = oracle.attention_rows(q, k, v, [1, 1], 0.3)
    for b in range(2):
        for h in range(4):
            assert np.array_equal(out[b * 4 + h], v[b, 0, h // 2])


@pytest.mark.parametrize("Hq,Hkv", [(4, 1), (4, 4), (6, 2), (7, 1)])
def test_decode_T1_matches_sdpa(Hq, Hkv):
    inp = W.verify_inputs(B=2, T=1, Hq=Hq, Hkv=Hkv, D=16, ctx=[5, 37], dtype=torch.float32,
                          seed=11, prescale_q=False)
    got = oracle.attention_rows(inp["q"], inp["k"], inp["v"], inp["ctx"], 0.25)
    want = _sdpa_reference(inp["q"], inp["k"], inp["v"], inp["ctx"], 0.25, 0)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("T", [2, 5, 16])
def test_block_verify_matches_masked_sdpa(T):
    inp = W.verify_inputs(B=3, T=T, Hq=4, Hkv=2, D=8, ctx=[1, 9, 30], dtype=torch.bfloat16,
                          seed=12)
    got = oracle.attention_rows(inp["q"], inp["k"], inp["v"], inp["ctx"], 1.0)
    want = _sdpa_reference(inp["q"], inp["k"], inp["v"], inp["ctx"], 1.0, 0)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_drafter_matches_unmasked_sdpa():
    d = W.drafter_inputs(B=2, T=16, Hq=6, Hkv=2, D=8, n_ctx=[3, 40], layers=1, seed=13,
                         dtype=torch.float32)
    L = d["layers"][0]
    got = oracle.attention_rows(L["q"], d["kc"], d["vc"], d["n_ctx"], 0.5, mode=1,
                                kb=L["kb"], vb=L["vb"])
    want = _sdpa_reference(L["q"], d["kc"], d["vc"], d["n_ctx"], 0.5, 1, L["kb"], L["vb"])
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_row_j_sees_exactly_ctx_plus_j_keys():
    B, T, Hq, Hkv, D, ctx = 1, 16, 2, 1, 8, 20
    inp = W.verify_inputs(B=B, T=T, Hq=Hq, Hkv=Hkv, D=D, ctx=ctx, dtype=torch.float32, seed=14)
    base = oracle.attention_rows(inp["q"], inp["k"], inp["v"], inp["ctx"], 1.0).reshape(T, Hq, D)
    for j in range(T - 1):
        k2, v2 = inp["k"].clone(), inp["v"].clone()
        k2[0, ctx + j] += 3.0
        v2[0, ctx + j] -= 5.0
        pert = oracle.attention_rows(inp["q"], k2, v2, inp["ctx"], 1.0).reshape(T, Hq, D)
        # rows 0..j do not see slot ctx+j; rows j+1.. do
        assert np.array_equal(pert[: j + 1], base[: j + 1])
        assert np.all(np.abs(pert[j + 1:] - base[j + 1:]).max(axis=(1, 2)) > 1e-6)


def test_drafter_is_bidirectional_in_block():
    d = W.drafter_inputs(B=1, T=16, Hq=2, Hkv=1, D=8, n_ctx=10, layers=1, seed=15,
                         dtype=torch.float32)
    L = d["layers"][0]
    base = oracle.attention_rows(L["q"], d["kc"], d["vc"], d["n_ctx"], 1.0, mode=1,
                                 kb=L["kb"], vb=L["vb"])
    vb2 = L["vb"].clone()
    vb2[0, 15] += 4.0  # the last block slot changes every row, row 0 included
    pert = oracle.attention_rows(L["q"], d["kc"], d["vc"], d["n_ctx"], 1.0, mode=1,
                                 kb=L["kb"], vb=vb2)
    assert np.all(np.abs(pert - base).max(axis=1) > 1e-6)


def test_constant_keys_give_mean_of_values():
    rng = np.random.default_rng(3)
    B, T, Hq, Hkv, D, ctx = 2, 16, 4, 2, 8, 11
    q = rng.standard_normal((B, T, Hq, D))
    k = np.broadcast_to(rng.standard_normal((1, 1, Hkv, D)), (B, ctx + T - 1, Hkv, D)).copy()
    v = rng.standard_normal((B, ctx + T - 1, Hkv, D))
    out = oracle.attention_rows(q, k, v, [ctx, ctx], 0.7).reshape(B, T, Hq, D)
    for b in range(B):
        for j in range(T):
            for h in range(Hq):
                want = v[b, : ctx + j, h // 2].mean(axis=0)
                np.testing.assert_allclose(out[b, j, h], want, rtol=1e-13, atol=1e-13)


def test_weights_sum_to_one():
    # constant values c: the output is c exactly when the weights sum to 1
    rng = np.random.default_rng(4)
    q = rng.standard_normal((1, 16, 4, 8)) * 3
    k = rng.standard_normal((1, 60, 1, 8)) * 3
    v = np.full((1, 60, 1, 8), 2.5)
    out = oracle.attention_rows(q, k, v, [45], 1.0)
    np.testing.assert_allclose(out, 2.5, rtol=1e-14)


def test_head_permutation_within_group():
    inp = W.verify_inputs(B=1, T=4, Hq=6, Hkv=2, D=8, ctx=9, dtype=torch.float32, seed=16)
    base = oracle.attention_rows(inp["q"], inp["k"], inp["v"], inp["ctx"], 1.0).reshape(4, 6, 8)
    perm = [2, 0, 1, 5, 3, 4]  # permutes heads inside each group of 3
    q2 = inp["q"][:, :, perm]
    got = oracle.attention_rows(q2, inp["k"], inp["v"], inp["ctx"], 1.0).reshape(4, 6, 8)
    np.testing.assert_array_equal(got, base[:, perm])


@pytest.mark.parametrize("mode", [0, 1])
def test_split_then_lse_merge_equals_whole(mode):
    B, T, Hq, Hkv, D = 2, 16, 4, 2, 8
    if mode == 0:
        inp = W.verify_inputs(B=B, T=T, Hq=Hq, Hkv=Hkv, D=D, ctx=[7, 50], dtype=torch.float32,
                              seed=17)
        args = (inp["q"], inp["k"], inp["v"], inp["ctx"], 1.0)
        kw = {}
    else:
        d = W.drafter_inputs(B=B, T=T, Hq=Hq, Hkv=Hkv, D=D, n_ctx=[7, 50], layers=1, seed=18,
                             dtype=torch.float32)
        L = d["layers"][0]
        args = (L["q"], d["kc"], d["vc"], d["n_ctx"], 1.0)
        kw = dict(mode=1, kb=L["kb"], vb=L["vb"])
    whole, lse_whole = oracle.attention_rows(*args, return_lse=True, **kw)
    bounds = [0, 5, 13, 40, 52, 70]  # the later ranges are empty for sequence 0
    parts, lses = [], []
    for lo, hi in zip(bounds[:-1], bounds[1:]):
        o, l = oracle.attention_rows(*args, key_range=(lo, hi), return_lse=True, **kw)
        parts.append(o)
        lses.append(l)
    parts, lses = np.stack(parts), np.stack(lses)
    assert np.isneginf(lses).any()  # some ranges hold no key
    for r in range(whole.shape[0]):
        out, m = oracle.lse_merge(parts[:, r], lses[:, r])
        np.testing.assert_allclose(out, whole[r], rtol=1e-12, atol=1e-13)
        assert m == pytest.approx(lse_whole[r], abs=1e-12)


def test_rows_subset_matches_full():
    inp = W.verify_inputs(B=2, T=16, Hq=4, Hkv=1, D=8, ctx=[5, 9], dtype=torch.float32, seed=19)
    full = oracle.attention_rows(inp["q"], inp["k"], inp["v"], inp["ctx"], 1.0)
    rows = np.array([127, 0, 64, 5])
    sub = oracle.attention_rows(inp["q"], inp["k"], inp["v"], inp["ctx"], 1.0, rows=rows)
    np.testing.assert_array_equal(sub, full[rows])
