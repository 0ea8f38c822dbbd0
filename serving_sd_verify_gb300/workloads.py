"""Seeded synthetic inputs for block verification.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic, and both the CUDA path and the CPU oracle take their
inputs from it.  Shapes and distributions follow the five workloads the
library is measured on:

1. tiny verify: B=1, ctx 512, Hq 4 / Hkv 1, D 64, fp32 Q/K/V ~ N(0,1);
   fp32 logits [1,16,1000] ~ N(0, sd 2); drafts equal the row argmax for
   rows 0..4, differ from it at row 5, uniform afterwards.
2. LLaVA-OneVision-7B-shaped verify: B=1, ctx 25,119, Hq 28 / Hkv 4, D 128,
   bf16 K/V ~ N(0,1), Q ~ N(0,1)/sqrt(128); bf16 logits [1,16,152,064]
   ~ N(0, sd 3); drafts match the argmax for k ~ Geometric(0.12) rows
   (failures before the first success, capped at 15), differ at row k.
3. ragged batch: B=8, ctx ~ U{4096..32768} per sequence, else as 2.
4. drafter: hidden states bf16 [25,119, 3584] ~ N(0,1), W_k / W_v
   [3584 -> 4x128] Glorot-uniform, projected once into drafter K/V shared by
   4 layers, each with its own block Q/K/V; then workload 1.
5. LLaVA-OneVision-72B-shaped sampling: B=4, ctx 32,768, Hq 64 / Hkv 8,
   D 128; bf16 logits [4,16,V] ~ N(0, sd 3); draft probs
   softmax(logits + N(0,1)) in fp32; drafts d_j ~ q_j; temperature 1,
   Philox seed 1234.

Every tensor is a CPU torch tensor; callers move them to the device.
"""
from __future__ import annotations

import math

import numpy as np
import torch

BLOCK = 16          # anchor + 15 proposals
VOCAB = 152_064     # LLaVA-OneVision / Qwen2 vocabulary


def _to(x: np.ndarray, dtype: torch.dtype) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(dtype)


def _normal(rng, shape, sd=1.0):
    return rng.standard_normal(shape, dtype=np.float32) * np.float32(sd)


# --------------------------------------------------------------------------
# attention inputs
# --------------------------------------------------------------------------

def verify_inputs(*, B, T, Hq, Hkv, D, ctx, dtype=torch.bfloat16, seed=0,
                  prescale_q=True, s_max=None):
    """Query block + preallocated KV cache.

    ctx: int or list of per-sequence ctx_len (the anchor's K/V sits at slot
    ctx-1, block row j at ctx-1+j).  The cache holds s_max >= max(ctx)+T-1
    slots, every slot filled with N(0,1) values.  prescale_q folds 1/sqrt(D)
    into Q (the caller then passes scale = 1).
    """
    rng = np.random.default_rng(seed)
    ctx_l = [int(ctx)] * B if np.isscalar(ctx) else [int(c) for c in ctx]
    assert len(ctx_l) == B
    s_max = s_max or (max(ctx_l) + T - 1)
    q = _normal(rng, (B, T, Hq, D))
    if prescale_q:
        q = q / np.float32(math.sqrt(D))
    k = _normal(rng, (B, s_max, Hkv, D))
    v = _normal(rng, (B, s_max, Hkv, D))
    return {
        "q": _to(q, dtype), "k": _to(k, dtype), "v": _to(v, dtype),
        "ctx": torch.tensor(ctx_l, dtype=torch.int32),
        "scale": 1.0 if prescale_q else 1.0 / math.sqrt(D),
        "max_ctx": max(ctx_l),
    }


def ragged_ctx(B, lo, hi, seed):
    rng = np.random.default_rng(seed)
    return [int(x) for x in rng.integers(lo, hi + 1, size=B)]


def drafter_inputs(*, B, T, Hq, Hkv, D, n_ctx, layers=1, dtype=torch.bfloat16, seed=0,
                   kc=None, vc=None):
    """Per-layer block Q/K/V for the drafter's block attention.

    kc / vc [B, S, Hkv, D] are the projected context keys / values (from
    project_kv, or drawn N(0,1) here when not given).
    """
    rng = np.random.default_rng(seed)
    n_l = [int(n_ctx)] * B if np.isscalar(n_ctx) else [int(c) for c in n_ctx]
    if kc is None:
        s = max(n_l)
        kc = _to(_normal(rng, (B, s, Hkv, D)), dtype)
        vc = _to(_normal(rng, (B, s, Hkv, D)), dtype)
    lay = []
    for _ in range(layers):
        q = _normal(rng, (B, T, Hq, D)) / np.float32(math.sqrt(D))
        lay.append({"q": _to(q, dtype),
                    "kb": _to(_normal(rng, (B, T, Hkv, D)), dtype),
                    "vb": _to(_normal(rng, (B, T, Hkv, D)), dtype)})
    return {"kc": kc, "vc": vc, "n_ctx": torch.tensor(n_l, dtype=torch.int32),
            "layers": lay, "scale": 1.0, "max_ctx": max(n_l)}


def hidden_and_projector(*, N, hidden=3584, Hkv=4, D=128, seed=0):
    """Target hidden states bf16 [N, hidden] ~ N(0,1) and Glorot-uniform W_k, W_v
    [hidden, Hkv*D] (fp32)."""
    rng = np.random.default_rng(seed)
    h = _to(_normal(rng, (N, hidden)), torch.bfloat16)
    a = math.sqrt(6.0 / (hidden + Hkv * D))
    wk = torch.from_numpy(rng.uniform(-a, a, size=(hidden, Hkv * D)).astype(np.float32))
    wv = torch.from_numpy(rng.uniform(-a, a, size=(hidden, Hkv * D)).astype(np.float32))
    return h, wk, wv


def project_kv(h, wk, wv, *, Hkv=4, D=128, device="cpu"):
    """Set-up step (outside the verified path): K = bf16(H @ W_k) as
    [1, N, Hkv, D], and the same for V.  Computed in fp32 on `device`; both
    the oracle and the kernels then consume the identical bf16 tensors."""
    hd = h.to(device=device, dtype=torch.float32)
    k = (hd @ wk.to(device)).to(torch.bfloat16).reshape(1, h.shape[0], Hkv, D)
    v = (hd @ wv.to(device)).to(torch.bfloat16).reshape(1, h.shape[0], Hkv, D)
    return k.cpu().contiguous(), v.cpu().contiguous()


# --------------------------------------------------------------------------
# acceptance inputs
# --------------------------------------------------------------------------

def greedy_inputs(*, B, T, V, dtype=torch.bfloat16, sd=3.0, seed=0, k=None, geo_p=0.12):
    """Target logits [B,T,V] ~ N(0, sd) and drafts [B,T-1].

    Sequence b's drafts equal the row argmax (np.argmax: lowest index on
    ties, compared on the stored values) for rows < k_b and differ from it at
    row k_b (when k_b < T-1); later rows are uniform.  k is an int, a list,
    or None to draw k_b ~ Geometric(geo_p) failures, capped at T-1.
    Returns logits, draft, and k (the accept length the construction fixes).
    """
    rng = np.random.default_rng(seed)
    logits = _to(_normal(rng, (B, T, V), sd), dtype)
    stored = logits.float().numpy()
    if k is None:
        ks = [min(int(rng.geometric(geo_p)) - 1, T - 1) for _ in range(B)]
    elif np.isscalar(k):
        ks = [min(int(k), T - 1)] * B
    else:
        ks = [min(int(x), T - 1) for x in k]
    draft = rng.integers(0, V, size=(B, max(T - 1, 0))).astype(np.int32)
    for b in range(B):
        for j in range(T - 1):
            a = int(np.argmax(stored[b, j]))
            if j < ks[b]:
                draft[b, j] = a
            elif j == ks[b]:
                if V == 1:
                    raise ValueError("cannot force a mismatch with V == 1")
                x = int(rng.integers(0, V - 1))
                draft[b, j] = x + 1 if x >= a else x
    return {"logits": logits, "draft": torch.from_numpy(draft), "k": ks}


def sample_inputs(*, B, T, V, sd=3.0, noise_sd=1.0, seed=0, draft_seed=None,
                  dtype=torch.bfloat16):
    """Target logits [B,T,V] ~ N(0, sd); draft probs q = softmax(logits + N(0, noise_sd))
    (fp32, rows normalised in fp64 before rounding); drafts d_j ~ q_j drawn with
    a second seeded generator."""
    rng = np.random.default_rng(seed)
    logits = _to(_normal(rng, (B, T, V), sd), dtype)
    z = logits.double().numpy() + rng.standard_normal((B, T, V))
    z -= z.max(axis=-1, keepdims=True)
    e = np.exp(z)
    q64 = e / e.sum(axis=-1, keepdims=True)
    q = torch.from_numpy(q64.astype(np.float32))
    drng = np.random.default_rng(seed + 1 if draft_seed is None else draft_seed)
    draft = np.zeros((B, max(T - 1, 0)), dtype=np.int32)
    for b in range(B):
        for j in range(T - 1):
            c = np.cumsum(q64[b, j])
            draft[b, j] = min(int(np.searchsorted(c, drng.random() * c[-1], side="right")), V - 1)
    return {"logits": logits, "q": q, "draft": torch.from_numpy(draft)}


# --------------------------------------------------------------------------
# the five measured workloads
# --------------------------------------------------------------------------

def latent_inputs(*, frames, N, Cq, d, seed=0):
    """SpecFLASH compressor inputs: visual features bf16 [frames, N, d] ~ N(0,1)
    and learned queries bf16 [Cq, d] ~ N(0, 1/d) (so the scores are ~ N(0,1))."""
    rng = np.random.default_rng(seed)
    f = _to(_normal(rng, (frames, N, d)), torch.bfloat16)
    q = _to(_normal(rng, (Cq, d), sd=1.0 / math.sqrt(d)), torch.bfloat16)
    return q, f


CONFIG_NAMES = {
    1: "tiny-verify-ctx512-h4kv1-d64-fp32",
    2: "llava-ov-7b-verify-ctx25119-h28kv4-d128-bf16",
    3: "ragged-b8-ctx4096to32768-h28kv4-d128-bf16",
    4: "drafter-4x-block-attn-ctx25119-h28kv4-d128-bf16+tiny-verify",
    5: "llava-ov-72b-sampling-b4-ctx32768-h64kv8-d128-bf16",
}


def config(n: int):
    """Inputs of workload n (1..5) as described in the module docstring."""
    T = BLOCK
    if n == 1:
        att = verify_inputs(B=1, T=T, Hq=4, Hkv=1, D=64, ctx=512, dtype=torch.float32,
                            seed=1, prescale_q=False)
        acc = greedy_inputs(B=1, T=T, V=1000, dtype=torch.float32, sd=2.0, seed=101, k=5)
        return {"attn": att, "greedy": acc, "dims": dict(B=1, T=T, Hq=4, Hkv=1, D=64, V=1000)}
    if n == 2:
        att = verify_inputs(B=1, T=T, Hq=28, Hkv=4, D=128, ctx=25_119, seed=2)
        acc = greedy_inputs(B=1, T=T, V=VOCAB, seed=102)
        return {"attn": att, "greedy": acc, "dims": dict(B=1, T=T, Hq=28, Hkv=4, D=128, V=VOCAB)}
    if n == 3:
        ctx = ragged_ctx(8, 4096, 32768, seed=3)
        att = verify_inputs(B=8, T=T, Hq=28, Hkv=4, D=128, ctx=ctx, seed=3)
        acc = greedy_inputs(B=8, T=T, V=VOCAB, seed=103)
        return {"attn": att, "greedy": acc, "dims": dict(B=8, T=T, Hq=28, Hkv=4, D=128, V=VOCAB)}
    if n == 4:
        h, wk, wv = hidden_and_projector(N=25_119, seed=4)
        return {"hidden": h, "wk": wk, "wv": wv, "tail": config(1),
                "dims": dict(B=1, T=T, Hq=28, Hkv=4, D=128, N=25_119, layers=4)}
    if n == 5:
        att = verify_inputs(B=4, T=T, Hq=64, Hkv=8, D=128, ctx=32_768, seed=5)
        smp = sample_inputs(B=4, T=T, V=VOCAB, seed=105, draft_seed=1235)
        return {"attn": att, "sample": smp, "temperature": 1.0, "philox_seed": 1234,
                "dims": dict(B=4, T=T, Hq=64, Hkv=8, D=128, V=VOCAB)}
    raise ValueError(f"no workload {n}")


def drafter_layers(kc, vc, *, n_ctx=25_119, layers=4, seed=44):
    """Block Q/K/V of the drafter layers of workload 4 over given context K/V."""
    return drafter_inputs(B=1, T=BLOCK, Hq=28, Hkv=4, D=128, n_ctx=n_ctx, layers=layers,
                          seed=seed, kc=kc, vc=vc)
