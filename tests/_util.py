"""Shared helpers of the GPU parity tests (tolerances, oracle slicing)."""
from __future__ import annotations

import numpy as np
import torch

import oracle

# Attention tolerance: max abs error 2e-3 over all elements, and max abs error
# of a (b, j, h) output vector over that vector's max |value| at most 1e-2
# (elementwise relative error is undefined near 0).  bf16 inputs are exact in
# fp32; the kernels accumulate in fp32 and round P to bf16 for the tensor-core
# product (relative 2^-9 per weight, averaging out over the keys), so the
# observed errors sit one to two orders of magnitude below these bounds.
ATOL = 2e-3
RTOL_VEC = 1e-2


def check_attention(got, want, atol=ATOL, rtol=RTOL_VEC):
    got = np.asarray(got, dtype=np.float64).reshape(want.shape)
    err = np.abs(got - want)
    assert np.isfinite(got).all(), "non-finite attention output"
    amax = float(err.max()) if err.size else 0.0
    scale = np.maximum(np.abs(want).max(axis=-1), 1e-30)
    rel = float((err.max(axis=-1) / scale).max()) if err.size else 0.0
    assert amax <= atol, f"max abs error {amax:.3e} > {atol}"
    assert rel <= rtol, f"max vector-relative error {rel:.3e} > {rtol}"
    return amax, rel


def oracle_verify_rows(q, k, v, ctx, scale, rows, mode=0, kb=None, vb=None):
    """Oracle attention for flat rows (b*T + j)*Hq + h, slicing each (b, kv head)
    out of the cache first so that large workloads stay cheap."""
    B, T, Hq, D = q.shape
    Hkv = k.shape[2]
    G = Hq // Hkv
    rows = np.asarray(rows, dtype=np.int64)
    out = np.zeros((rows.size, D))
    ctx = [int(c) for c in (ctx.tolist() if hasattr(ctx, "tolist") else ctx)]
    groups = {}
    for i, r in enumerate(rows):
        h = int(r % Hq)
        j = int((r // Hq) % T)
        b = int(r // (Hq * T))
        groups.setdefault((b, h // G), []).append((i, j, h % G))
    for (b, g), items in groups.items():
        n = ctx[b] + T - 1 if mode == 0 else ctx[b]
        qs = q[b:b + 1, :, g * G:(g + 1) * G]
        ks = k[b:b + 1, :n, g:g + 1]
        vs = v[b:b + 1, :n, g:g + 1]
        kbs = kb[b:b + 1, :, g:g + 1] if kb is not None else None
        vbs = vb[b:b + 1, :, g:g + 1] if vb is not None else None
        sub = np.array([j * G + hl for (_, j, hl) in items], dtype=np.int64)
        o = oracle.attention_rows(qs, ks, vs, [ctx[b]], scale, mode=mode, kb=kbs, vb=vbs, rows=sub)
        for (i, _, _), orow in zip(items, o):
            out[i] = orow
    return out


def sample_rows(B, T, Hq, n, seed=0):
    """n flat rows, always including the first and last rows of every sequence."""
    rng = np.random.default_rng(seed)
    must = []
    for b in range(B):
        for j in (0, T - 1):
            must += [(b * T + j) * Hq, (b * T + j) * Hq + Hq - 1]
    extra = rng.choice(B * T * Hq, size=min(n, B * T * Hq), replace=False)
    return np.unique(np.concatenate([np.array(must), extra]))


def to_dev(d, device="cuda"):
    return {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


def check_projection(got, h, w, rows=None, min_exact=0.99):
    """Projector output (bf16, fp32 accumulation, one rounding) against the
    fp64 oracle: every element within half a bf16 ulp of the exact value plus
    the fp32 summation bound Hd * 2^-23 * sum_f |h_f w_f|, and at least
    `min_exact` of them equal to the exact value rounded to bf16."""
    ref = oracle.project_rows(h, w, rows)
    absum = oracle.project_rows(np.abs(np.asarray(h.double() if hasattr(h, "double") else h, dtype=np.float64)),
                                np.abs(np.asarray(w.double() if hasattr(w, "double") else w, dtype=np.float64)),
                                rows)
    acc = h.shape[1] * 2.0 ** -23 * absum
    tol = 2.0 ** -8 * (np.abs(ref) + acc) + acc
    g = got.double().numpy() if hasattr(got, "double") else np.asarray(got, dtype=np.float64)
    g = g.reshape(ref.shape)
    err = np.abs(g - ref)
    assert (err <= tol).all(), (err.max(), np.unravel_index(np.argmax(err - tol), err.shape))
    exact = torch.from_numpy(ref).to(torch.bfloat16).double().numpy()
    frac = float((g == exact).mean())
    assert frac >= min_exact, frac
