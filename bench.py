#!/usr/bin/env python3
"""Benchmark: verified 16-token blocks per second at a 25,119-token context.

One step = one pass of the whole hot path over one block (B = 1):
  1. drafter block attention, 4 layers (Hq 28 / Hkv 4, D 128) over 25,119
     context keys projected from seeded hidden states (shared by the layers);
  2. target block-verify attention over the 25,119-token cache (+15 block slots);
  3. greedy acceptance over the block's bf16 logits [16, 152,064];
  4. sampled acceptance over the same logits with draft probs
     softmax(logits + N(0,1)), temperature 1, Philox seed 1234.
A real cycle runs one of the two acceptance rules; timing both keeps every
step of the path in the measured step (blocks/s is then a lower bound).

Inputs live in HBM before timing starts and rotate over several copies whose
total exceeds twice the L2, so each step reads cold K/V and logits (the four
drafter layers share one projected context, which stays in L2 after the first
layer -- that reuse is part of the method).  The steps are replayed from CUDA
graphs captured from the C-ABI calls.

`--impl reference` times the fp64 CPU oracle on the host on a bounded sample
of the same step (see reference_arm).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verified 16-token blocks/sec and HBM GB/s (% of peak) at 25,119-token ctx"
WORKLOAD = "llava-ov-7b-verify-ctx25119-h28kv4-d128-bf16 + 4-layer drafter + greedy & sampled accept (V=152064)"
CTX, T, HQ, HKV, D, V, LAYERS = 25_119, 16, 28, 4, 128, 152_064, 4
HD = 3584           # target hidden size (Qwen2-7B), the projector's input width
APPEND = 8          # rows one cycle appends to the drafter's context (accepted + correction)
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
L2_BYTES = 129 * 1024 * 1024


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# ---------------------------------------------------------------------------
# algorithmic bytes of one launch (minimal traffic: every input read once,
# every output written once; split partials excluded)
# ---------------------------------------------------------------------------

def attn_bytes(n_keys, extra_block_keys=0):
    kv = 2 * n_keys * HKV * D * 2
    blk = 2 * extra_block_keys * HKV * D * 2
    q = T * HQ * D * 2
    out = T * HQ * D * 4
    return kv + blk + q + out


BYTES = {
    "verify_attention": attn_bytes(CTX + T - 1),
    "draft_attention": attn_bytes(CTX, T),
    "accept_greedy": T * V * 2 + (T - 1) * 4 + 8,
    # logits read twice (stats, then the deciding row), q gathered + one q row
    "accept_sample": T * V * 2 + V * 2 + V * 4 + (T - 1) * 8 + 8,
    # the tree rows (not part of the timed step): the same reads plus the tree
    "verify_tree_attention": attn_bytes(CTX + T - 1) + T * 4,
    "accept_tree_greedy": T * V * 2 + T * 8 + T * 4 + 8,
    # projector append: both weights read once, the new rows in and out
    "project_append": 2 * HKV * D * HD * 2 + APPEND * HD * 2 + 2 * APPEND * HKV * D * 2,
}
PROJ_PREFILL_FLOPS = 2 * CTX * HD * 2 * HKV * D
# SpecFLASH latent compressor: 16 frames of LLaVA-1.5-7B visual features
# (576 per frame, d 4096) compressed to 64 latents each
LC_FRAMES, LC_N, LC_C, LC_D = 16, 576, 64, 4096
LC_BYTES = LC_FRAMES * LC_N * LC_D * 2 + LC_C * LC_D * 2 + LC_FRAMES * LC_C * LC_D * 2
LC_FLOPS = 2 * 2 * LC_FRAMES * LC_C * LC_N * LC_D


# ---------------------------------------------------------------------------
# inputs
# ---------------------------------------------------------------------------

def make_inputs(device):
    import numpy as np
    import torch
    from serving_sd_verify_gb300 import workloads as W
    t0 = time.time()
    cfg2 = W.config(2)
    h, wk, wv = W.hidden_and_projector(N=CTX, seed=4)
    kc, vc = W.project_kv(h, wk, wv, device=device)
    dr = W.drafter_layers(kc, vc)
    smp = W.sample_inputs(B=1, T=T, V=V, seed=105, draft_seed=1235)
    smp["logits"] = cfg2["greedy"]["logits"]
    # draft probs / drafts for the sampled rule drawn around the same logits
    z = smp["logits"].double().numpy() + np.random.default_rng(205).standard_normal((1, T, V))
    z -= z.max(-1, keepdims=True)
    q = np.exp(z)
    q /= q.sum(-1, keepdims=True)
    rng = np.random.default_rng(1235)
    draft = np.array([[min(int(np.searchsorted(np.cumsum(q[0, j]), rng.random(), side="right")), V - 1)
                       for j in range(T - 1)]], dtype=np.int32)
    smp["q"] = torch.from_numpy(q.astype(np.float32))
    smp["draft"] = torch.from_numpy(draft)
    # a seeded 16-node draft tree (each node's parent among the 3 before it);
    # node tokens mostly equal the target's pick after the parent
    trng = np.random.default_rng(60)
    parents = np.full(T, -1, dtype=np.int32)
    for j in range(1, T):
        parents[j] = trng.integers(max(0, j - 3), j)
    mask = np.zeros(T, dtype=np.int64)
    for j in range(T):
        v = j
        while v != -1:
            mask[j] |= 1 << v
            v = parents[v]
    am = cfg2["greedy"]["logits"].float().numpy().argmax(-1)[0]
    tokens = np.array([0] + [int(am[parents[j]]) if trng.random() < 0.7 else int(trng.integers(0, V))
                             for j in range(1, T)], dtype=np.int32)
    tree = {"mask": torch.from_numpy(mask).reshape(1, T),
            "parents": torch.from_numpy(parents).reshape(1, T), "tokens": torch.from_numpy(tokens).reshape(1, T)}
    # the drafter K/V projector in a linear layer's [out, in] layout, bf16
    proj = {"h": h, "wk": wk.t().contiguous().to(torch.bfloat16), "wv": wv.t().contiguous().to(torch.bfloat16)}
    log(f"[bench] inputs generated in {time.time() - t0:.1f}s")
    return {"attn": cfg2["attn"], "greedy": cfg2["greedy"], "drafter": dr, "sample": smp, "tree": tree,
            "proj": proj}


class DeviceSet:
    """One full copy of a step's inputs and outputs in HBM."""

    def __init__(self, host, device, S):
        import torch
        a, g, d, s = host["attn"], host["greedy"], host["drafter"], host["sample"]
        dv = lambda t: t.to(device).contiguous()
        self.q, self.k, self.v, self.ctx = dv(a["q"]), dv(a["k"]), dv(a["v"]), dv(a["ctx"])
        self.kc, self.vc, self.nctx = dv(d["kc"]), dv(d["vc"]), dv(d["n_ctx"])
        self.layers = [(dv(L["q"]), dv(L["kb"]), dv(L["vb"])) for L in d["layers"]]
        self.logits, self.draft = dv(g["logits"]), dv(g["draft"])
        self.sq, self.sdraft = dv(s["q"]), dv(s["draft"])
        self.out = torch.zeros(1, T, HQ, D, device=device)
        self.dout = [torch.zeros(1, T, HQ, D, device=device) for _ in range(LAYERS)]
        self.n = torch.zeros(1, dtype=torch.int32, device=device)
        self.c = torch.zeros(1, dtype=torch.int32, device=device)
        self.sn = torch.zeros(1, dtype=torch.int32, device=device)
        self.snx = torch.zeros(1, dtype=torch.int32, device=device)
        self.ws_v = S.workspace(S.sd_verify_attention_workspace_size(1, T, HQ, HKV, D, CTX), device)
        self.ws_d = S.workspace(S.sd_draft_block_attention_workspace_size(1, T, HQ, HKV, D, CTX), device)
        self.ws_g = S.workspace(S.sd_accept_greedy_workspace_size(1, T, V), device)
        self.ws_s = S.workspace(S.sd_accept_sample_workspace_size(1, T, V), device)
        tr = host["tree"]
        self.tmask, self.tparents, self.ttokens = dv(tr["mask"]), dv(tr["parents"]), dv(tr["tokens"])
        self.tpath = torch.zeros(1, T, dtype=torch.int32, device=device)
        self.tn = torch.zeros(1, dtype=torch.int32, device=device)
        self.tc = torch.zeros(1, dtype=torch.int32, device=device)
        self.ws_tv = S.workspace(S.sd_verify_tree_attention_workspace_size(1, T, HQ, HKV, D, CTX), device)
        self.ws_tg = S.workspace(S.sd_accept_tree_greedy_workspace_size(1, T, V), device)

    def nbytes(self):
        ts = [self.q, self.k, self.v, self.kc, self.vc, self.logits, self.sq]
        return sum(t.numel() * t.element_size() for t in ts)


class ProjSet:
    """The drafter K/V projector's operands in HBM: the context's target hidden
    states [CTX, HD], W_k / W_v [HKV*D, HD], and the projected context."""

    def __init__(self, hp, device):
        import torch
        self.h = hp["h"].to(device).contiguous()
        self.wk, self.wv = hp["wk"].to(device), hp["wv"].to(device)
        self.k = torch.empty(CTX, HKV * D, dtype=torch.bfloat16, device=device)
        self.v = torch.empty_like(self.k)

    def run(self, S, stream, n_rows):
        r0 = CTX - n_rows
        S.sd_project_kv(self.h[r0:], self.wk, self.wv, self.k[r0:], self.v[r0:], stream)


ROOM = 1024         # spare cache positions of the cycle measurement (the context grows each replay)


class CycleSet:
    """A whole speculative cycle on resident state, captured in one CUDA
    graph: the drafter's 4 layers, the target verify, greedy acceptance, the
    drafter-context append of the committed rows and the commit (ctx_len,
    tokens, anchor) -- nothing returns to the host between cycles.  The caches
    hold ROOM spare positions, so every replay really extends the context."""

    def __init__(self, ds, proj, device, S):
        import torch
        bf = torch.bfloat16
        self.ds, self.proj = ds, proj
        self.k = torch.zeros(1, CTX + ROOM + T - 1, HKV, D, dtype=bf, device=device)
        self.v = torch.zeros_like(self.k)
        self.k[:, :CTX + T - 1] = ds.k
        self.v[:, :CTX + T - 1] = ds.v
        self.kc = torch.zeros(1, CTX + ROOM, HKV, D, dtype=bf, device=device)
        self.vc = torch.zeros_like(self.kc)
        self.kc[:, :CTX] = ds.kc
        self.vc[:, :CTX] = ds.vc
        self.ctx, self.dctx = ds.ctx.clone(), ds.nctx.clone()
        g = torch.Generator(device="cpu").manual_seed(77)
        self.hid = torch.randn(1, T, HD, generator=g).to(bf).to(device)
        self.n = torch.zeros(1, dtype=torch.int32, device=device)
        self.c = torch.zeros(1, dtype=torch.int32, device=device)
        self.toks = torch.full((1, 64 * T), -1, dtype=torch.int32, device=device)
        self.olen = torch.zeros(1, dtype=torch.int32, device=device)
        self.anchor = torch.zeros(1, dtype=torch.int32, device=device)
        self.ws_v = S.workspace(S.sd_verify_attention_workspace_size(1, T, HQ, HKV, D, CTX + ROOM), device)
        self.ws_d = S.workspace(S.sd_draft_block_attention_workspace_size(1, T, HQ, HKV, D, CTX + ROOM), device)
        self.launches = 0

    def commit(self, S, stream):
        kcv = self.kc.view(1, CTX + ROOM, HKV * D)
        vcv = self.vc.view(1, CTX + ROOM, HKV * D)
        S.sd_project_kv_commit(self.hid, self.proj.wk, self.proj.wv, self.n, self.dctx, kcv, vcv, stream=stream)
        S.sd_commit_tokens(self.ds.draft, self.n, self.c, self.ctx, self.toks, self.olen, self.anchor, CTX + ROOM,
                           draft_ctx=self.dctx, stream=stream)

    def cycle(self, S, stream):
        ds = self.ds
        launches = 0
        for li, (q, kb, vb) in enumerate(ds.layers):
            S.sd_draft_block_attention(q, self.kc, self.vc, self.dctx, CTX + ROOM, kb, vb, ds.dout[li], 1.0,
                                       self.ws_d, stream)
            launches += S.sd_last_attention_launches()
        S.sd_verify_attention(ds.q, self.k, self.v, self.ctx, CTX + ROOM, ds.out, 1.0, self.ws_v, stream)
        launches += S.sd_last_attention_launches()
        S.sd_accept_greedy(ds.draft, ds.logits, self.n, self.c, ds.ws_g, stream)
        self.commit(S, stream)
        self.launches = launches + 3


# kernels of one step: 5 attention calls (1 launch each when the splits merge
# inside the split kernel, else 2), greedy 1, sampled 1 (one cooperative
# launch) or 2; set from the library after a warm-up step
ATTN_LAUNCHES = {"draft": 2, "verify": 2, "sample": 2}
def kernels_per_step():
    return LAYERS * ATTN_LAUNCHES["draft"] + ATTN_LAUNCHES["verify"] + 1 + ATTN_LAUNCHES["sample"]


def verify_bytes(ctx_list, T_, Hq, Hkv, D_):
    """Algorithmic bytes of one verify call: every cache key a row can see,
    K and V (bf16), read once; Q read once (bf16); the output written once (fp32)."""
    n_keys = sum(int(c) + T_ - 1 for c in ctx_list)
    B = len(ctx_list)
    return 2 * n_keys * Hkv * D_ * 2 + B * T_ * Hq * D_ * 2 + B * T_ * Hq * D_ * 4


def time_back_to_back(calls, n_copies, stream, reps=10):
    """Average seconds per call of calls[i % n_copies] issued 2 x n_copies times
    in one CUDA graph, replayed `reps` times after 3 warm-up replays."""
    import torch
    with torch.cuda.stream(stream):
        for c in calls:
            c()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(2 * n_copies):
            calls[i % n_copies]()
    with torch.cuda.stream(stream):
        for _ in range(3):
            g.replay()
        e_a, e_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e_a.record(stream)
        for _ in range(reps):
            g.replay()
        e_b.record(stream)
    torch.cuda.synchronize()
    del g
    return e_a.elapsed_time(e_b) / 1e3 / (reps * 2 * n_copies)


def config_verify_pass(S, device, stream, n):
    """Verify attention of the ragged batch (workload 3) or the 72B-shaped
    batch (workload 5) at full size, calls back to back over 2 input copies
    (each copy alone is larger than L2).  Returns (seconds per call, bytes)."""
    import torch
    from serving_sd_verify_gb300 import workloads as W
    att = W.config(n)["attn"]
    B_, T_, Hq, D_ = att["q"].shape
    Hkv = att["k"].shape[2]
    max_ctx = att["max_ctx"]
    copies = []
    for _ in range(2):
        q, k, v, ctx = (att[x].to(device).contiguous() for x in ("q", "k", "v", "ctx"))
        out = torch.zeros(B_, T_, Hq, D_, device=device)
        ws = S.workspace(S.sd_verify_attention_workspace_size(B_, T_, Hq, Hkv, D_, att["max_ctx"]), device)
        copies.append((q, k, v, ctx, out, ws))
    del att

    def call(c):
        return lambda: S.sd_verify_attention(c[0], c[1], c[2], c[3], max_ctx, c[4], 1.0, c[5], stream)
    calls = [call(c) for c in copies]
    per = time_back_to_back(calls, len(copies), stream)
    ctx_list = copies[0][3].cpu().tolist()
    del copies, calls
    torch.cuda.empty_cache()
    return per, verify_bytes(ctx_list, T_, Hq, Hkv, D_)


def profile_case(S, device, args):
    """One call class alone for a profiler, launched --warmup + --steps times on
    one stream: verify attention of workload 3 (8 sequences, ragged contexts)
    or 5 (4 sequences, 64 query / 8 kv heads, 32,768-token contexts); greedy
    acceptance over 8 sequences' logits or the sampled rule over 4 (the batched
    workloads); the projector at prefill (25,119 rows) or for an 8-row append;
    the latent compressor (16 frames x 576 features, d 4096 -> 64)."""
    import torch
    from serving_sd_verify_gb300 import workloads as W
    case = args.profile_case
    if case in ("cfg3-verify", "cfg5-verify"):
        att = W.config(3 if case == "cfg3-verify" else 5)["attn"]
        B_, T_, Hq, D_ = att["q"].shape
        Hkv = att["k"].shape[2]
        q, k, v, ctx = (att[x].to(device).contiguous() for x in ("q", "k", "v", "ctx"))
        out = torch.zeros(B_, T_, Hq, D_, device=device)
        ws = S.workspace(S.sd_verify_attention_workspace_size(B_, T_, Hq, Hkv, D_, att["max_ctx"]), device)
        call = lambda: S.sd_verify_attention(q, k, v, ctx, att["max_ctx"], out, 1.0, ws)
    elif case == "accept-greedy-b8":
        g = W.greedy_inputs(B=8, T=T, V=V, seed=103)
        d, lg = g["draft"].to(device), g["logits"].to(device)
        n = torch.zeros(8, dtype=torch.int32, device=device)
        c = torch.zeros_like(n)
        ws = S.workspace(S.sd_accept_greedy_workspace_size(8, T, V), device)
        call = lambda: S.sd_accept_greedy(d, lg, n, c, ws)
    elif case == "accept-sample-b4":
        sm = W.sample_inputs(B=4, T=T, V=V, seed=105, draft_seed=1235)
        d, q, lg = sm["draft"].to(device), sm["q"].to(device), sm["logits"].to(device)
        n = torch.zeros(4, dtype=torch.int32, device=device)
        c = torch.zeros_like(n)
        ws = S.workspace(S.sd_accept_sample_workspace_size(4, T, V), device)
        call = lambda: S.sd_accept_sample(d, q, lg, 1.0, 1234, 0, n, c, ws)
    elif case in ("project-prefill", "project-append"):
        h, wk, wv = W.hidden_and_projector(N=CTX, seed=4)
        h = h.to(device).contiguous()
        wk = wk.t().contiguous().to(torch.bfloat16).to(device)
        wv = wv.t().contiguous().to(torch.bfloat16).to(device)
        kk = torch.empty(CTX, HKV * D, dtype=torch.bfloat16, device=device)
        vv = torch.empty_like(kk)
        r0 = 0 if case == "project-prefill" else CTX - APPEND
        call = lambda: S.sd_project_kv(h[r0:], wk, wv, kk[r0:], vv[r0:])
    else:
        lq, lf = W.latent_inputs(frames=LC_FRAMES, N=LC_N, Cq=LC_C, d=LC_D, seed=16)
        lq, lf = lq.to(device), lf.to(device)
        lout = torch.empty(LC_FRAMES, LC_C, LC_D, dtype=torch.bfloat16, device=device)
        lws = S.workspace(S.sd_latent_compress_workspace_size(LC_FRAMES, LC_N, LC_C, LC_D), device)
        call = lambda: S.sd_latent_compress(lq, lf, lout, lws)
    torch.cuda.synchronize()
    for _ in range(args.warmup + args.steps):
        call()
    torch.cuda.synchronize()
    assert S.sd_fault_word() == 0


def tree60_pass(S, device, stream, n_nodes=60):
    """The pages' Tree-60 at the 25,119-token workload: verify attention over a
    seeded 60-node draft tree (each node's parent among the 3 before it) and
    greedy tree acceptance over its [1, 60, V] logits, each back to back over
    input copies larger than L2 in total.  Returns (attention s, acceptance s,
    attention bytes, acceptance bytes)."""
    import numpy as np
    import torch
    from serving_sd_verify_gb300 import workloads as W
    Tt = n_nodes
    att = W.verify_inputs(B=1, T=Tt, Hq=HQ, Hkv=HKV, D=D, ctx=CTX, seed=2)
    rng = np.random.default_rng(61)
    parents = np.full(Tt, -1, dtype=np.int32)
    for j in range(1, Tt):
        parents[j] = rng.integers(max(0, j - 3), j)
    mask = np.zeros(Tt, dtype=np.uint64)
    for j in range(Tt):
        v, bits = j, 0
        while v != -1:
            bits |= 1 << int(v)
            v = parents[v]
        mask[j] = np.uint64(bits)
    tm = torch.from_numpy(mask.view(np.int64)).reshape(1, Tt).to(device)
    acopies = []
    for _ in range(4):   # 4 x 51.6 MB of K/V
        q, k, v, ctx = (att[x].to(device).contiguous() for x in ("q", "k", "v", "ctx"))
        out = torch.zeros(1, Tt, HQ, D, device=device)
        ws = S.workspace(S.sd_verify_tree_attention_workspace_size(1, Tt, HQ, HKV, D, CTX), device)
        acopies.append((q, k, v, ctx, out, ws))
    del att
    calls = [(lambda c=c: S.sd_verify_tree_attention(c[0], c[1], c[2], c[3], CTX, tm, c[4], 1.0, c[5], stream))
             for c in acopies]
    t_att = time_back_to_back(calls, len(acopies), stream)
    a_bytes = verify_bytes([CTX], Tt, HQ, HKV, D) + Tt * 8
    del acopies, calls
    g = W.greedy_inputs(B=1, T=Tt, V=V, seed=160, k=0)
    am = g["logits"].float().numpy().argmax(-1)[0]
    tokens = np.array([0] + [int(am[parents[j]]) if rng.random() < 0.7 else int(rng.integers(0, V))
                             for j in range(1, Tt)], dtype=np.int32)
    tok = torch.from_numpy(tokens).reshape(1, Tt).to(device)
    par = torch.from_numpy(parents).reshape(1, Tt).to(device)
    gcopies = []
    for _ in range(8):   # 8 x 18.2 MB of logits
        lg = g["logits"].to(device)
        n_ = torch.zeros(1, dtype=torch.int32, device=device)
        c_ = torch.zeros(1, dtype=torch.int32, device=device)
        path = torch.zeros(1, Tt, dtype=torch.int32, device=device)
        ws = S.workspace(S.sd_accept_tree_greedy_workspace_size(1, Tt, V), device)
        gcopies.append((lg, n_, c_, path, ws))
    calls = [(lambda c=c: S.sd_accept_tree_greedy(tok, par, c[0], c[1], c[2], c[3], c[4], stream)) for c in gcopies]
    t_acc = time_back_to_back(calls, len(gcopies), stream)
    g_bytes = Tt * V * 2 + Tt * 8 + Tt * 4 + 8
    del gcopies, calls
    torch.cuda.empty_cache()
    return t_att, t_acc, a_bytes, g_bytes


def drafter_layer_pass(S, ds, stream, flush, reps=20):
    """The step's 4 drafter layers, one graph replay after an L2 flush, with
    events between the calls: layer 1 streams the projected context from HBM,
    layers 2-4 find it in L2.  Returns (layer-1 seconds, mean of layers 2-4)."""
    import torch
    with torch.cuda.stream(stream):
        run_step(S, ds, stream, ("draft",))
    torch.cuda.synchronize()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(LAYERS + 1)]
    t1, t234 = [], []
    for i in range(reps):
        with torch.cuda.stream(stream):
            flush.zero_()
            evs[0].record(stream)
            for li, (q, kb, vb) in enumerate(ds.layers):
                S.sd_draft_block_attention(q, ds.kc, ds.vc, ds.nctx, CTX, kb, vb, ds.dout[li], 1.0, ds.ws_d,
                                           stream)
                evs[li + 1].record(stream)
        torch.cuda.synchronize()
        if i >= 3:
            t1.append(evs[0].elapsed_time(evs[1]) / 1e3)
            t234.append(evs[1].elapsed_time(evs[LAYERS]) / 1e3 / (LAYERS - 1))
    return statistics.median(t1), statistics.median(t234)


def run_step(S, ds, stream=None, parts=("draft", "verify", "greedy", "sample")):
    if "draft" in parts:
        for li, (q, kb, vb) in enumerate(ds.layers):
            S.sd_draft_block_attention(q, ds.kc, ds.vc, ds.nctx, CTX, kb, vb, ds.dout[li], 1.0, ds.ws_d, stream)
        ATTN_LAUNCHES["draft"] = S.sd_last_attention_launches()
    if "verify" in parts:
        S.sd_verify_attention(ds.q, ds.k, ds.v, ds.ctx, CTX, ds.out, 1.0, ds.ws_v, stream)
        ATTN_LAUNCHES["verify"] = S.sd_last_attention_launches()
    if "greedy" in parts:
        S.sd_accept_greedy(ds.draft, ds.logits, ds.n, ds.c, ds.ws_g, stream)
    if "sample" in parts:
        S.sd_accept_sample(ds.sdraft, ds.sq, ds.logits, 1.0, 1234, 0, ds.sn, ds.snx, ds.ws_s, stream)
        ATTN_LAUNCHES["sample"] = 1 if S.sd_last_sample_path() == 2 else 2
    if "tree_verify" in parts:
        S.sd_verify_tree_attention(ds.q, ds.k, ds.v, ds.ctx, CTX, ds.tmask, ds.out, 1.0, ds.ws_tv, stream)
    if "tree_greedy" in parts:
        S.sd_accept_tree_greedy(ds.ttokens, ds.tparents, ds.logits, ds.tn, ds.tc, ds.tpath, ds.ws_tg, stream)


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        self.lines = []
        self.gpu = gpu_index
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.th = threading.Thread(target=self._read, daemon=True)
            self.th.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        rows = [l for (t, l) in self.lines if t0 - 0.25 <= t <= t1 + 0.25]
        note = "sampled inside the timed region"
        if len(rows) < 2:
            rows = [l for (t, l) in self.lines if t0 - 3.0 <= t <= t1 + 0.25]
            note = "timed region shorter than the sampling period: samples from the soak just before it"
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            f = [x.strip() for x in r.split(",")]
            if len(f) < 10:
                continue
            try:
                sm.append(float(f[2]))
                mx.append(float(f[3]))
            except ValueError:
                continue
            for name, val in zip(names, f[6:10]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "note": "nvidia-smi unavailable"}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "note": note}


# ---------------------------------------------------------------------------
# peaks, ncu traffic
# ---------------------------------------------------------------------------

def hbm_peak(sustained: bool):
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            mp = json.load(f)
        for key in (["hbm_gbs_sustained", "hbm_gbs"] if sustained else ["hbm_gbs"]):
            if key in mp and mp[key]:
                v = mp[key]
                v = v.get("value", v) if isinstance(v, dict) else v
                return float(v), f"measured ({key}, MEASURED_PEAKS.json)"
    except (OSError, ValueError, TypeError):
        pass
    return FALLBACK_HBM_GBS, "fallback (6.8 TB/s, earlier GB300 measurement; MEASURED_PEAKS.json absent)"


def bf16_peak(sustained: bool):
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            mp = json.load(f)
        for key in (["bf16_tflops_sustained", "bf16_tflops"] if sustained else ["bf16_tflops"]):
            if key in mp and mp[key]:
                v = mp[key]
                v = v.get("value", v) if isinstance(v, dict) else v
                return float(v), f"measured ({key}, MEASURED_PEAKS.json)"
    except (OSError, ValueError, TypeError):
        pass
    return FALLBACK_BF16_TFLOPS, "fallback (1.9 PFLOP/s bf16 burst, earlier GB300 measurement; MEASURED_PEAKS.json absent)"


# sources that define each measured kernel (a capture is valid while they are unchanged)
KERNEL_SOURCES = {
    "verify_attention": ["attn_tc.cu", "tcgen05.cuh", "common.cuh", "internal.h"],
}


def csrc_digest(files):
    h = hashlib.sha256()
    d = os.path.join(ROOT, "serving_sd_verify_gb300", "csrc")
    for name in files:
        with open(os.path.join(d, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel_key):
    """Per-launch DRAM bytes (read + write) of `kernel_key` from
    profiles/traffic.txt, if that capture was taken from the current kernel
    sources; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    try:
        lines = open(path).read().splitlines()
    except OSError:
        return None
    dig = csrc_digest(KERNEL_SOURCES[kernel_key])
    for line in lines:
        f = line.split()
        if len(f) >= 3 and not line.startswith("#") and f[0] == kernel_key and f[2] == dig:
            return float(f[1])
    return None


# ---------------------------------------------------------------------------
# timing helpers
# ---------------------------------------------------------------------------

def graph_of(S, sets, stream, parts):
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for ds in sets:
            run_step(S, ds, torch.cuda.current_stream(), parts)
    return g


def time_graph(g, reps, stream):
    import torch
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(reps):
        g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / 1e3  # seconds


# ---------------------------------------------------------------------------
# CPU baseline: the oracle on a bounded sample of one step
# ---------------------------------------------------------------------------

def cpu_step_sample(host, rows_per_call, threads=1):
    """Oracle time of one step, extrapolated from `rows_per_call` query rows per
    attention call (all rows of both acceptance calls run in full).  With
    threads > 1 each attention call's rows are cut into that many slices run
    by a thread pool (the oracle's C routines release the GIL), so the
    attention part uses that many host cores; the acceptance calls stay on one."""
    import numpy as np
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    a, g, d, s = host["attn"], host["greedy"], host["drafter"], host["sample"]
    G = HQ // HKV
    rng = np.random.default_rng(0)
    total_rows = T * HQ
    rows = rng.choice(total_rows, size=rows_per_call, replace=False)
    # pre-widen the slices the sampled rows read (not timed: input preparation)
    def sliced(q, k, v, n, kb=None, vb=None):
        return q.double().numpy(), k[:, :n].double().numpy(), v[:, :n].double().numpy(), \
            None if kb is None else kb.double().numpy(), None if vb is None else vb.double().numpy()
    qv, kv_, vv_, _, _ = sliced(a["q"], a["k"], a["v"], CTX + T - 1)
    lay = [sliced(L["q"], d["kc"], d["vc"], CTX, L["kb"], L["vb"]) for L in d["layers"]]
    lg = g["logits"].double().numpy()
    sq = s["q"].double().numpy()
    slices = [sl for sl in np.array_split(rows, max(1, threads)) if sl.size]
    pool = ThreadPoolExecutor(max_workers=len(slices)) if len(slices) > 1 else None

    def attn(*a, **kw):
        if pool is None:
            oracle.attention_rows(*a, rows=rows, **kw)
        else:
            list(pool.map(lambda sl: oracle.attention_rows(*a, rows=sl, **kw), slices))
    t0 = time.perf_counter()
    for (q, kk, vv, kb, vb) in lay:
        attn(q, kk, vv, [CTX], 1.0, mode=1, kb=kb, vb=vb)
    attn(qv, kv_, vv_, [CTX], 1.0)
    t_attn = time.perf_counter() - t0
    if pool is not None:
        pool.shutdown()
    t1 = time.perf_counter()
    oracle.accept_greedy(g["draft"].numpy(), lg)
    oracle.accept_sample(s["draft"].numpy(), sq, lg, 1.0, 1234, 0)
    t_acc = time.perf_counter() - t1
    step = t_attn * (total_rows / rows_per_call) + t_acc
    return step, t_attn + t_acc


def host_cores():
    """Host cores this process may run on (the thread count of the all-core legs)."""
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def reference_arm(args, host=None):
    import numpy as np  # noqa: F401
    import oracle
    oracle.build()
    if host is None:
        import torch
        host = make_inputs("cuda" if torch.cuda.is_available() else "cpu")
    cores = host_cores()
    rows = min(T * HQ, args.ref_rows * cores)
    for _ in range(args.warmup):
        cpu_step_sample(host, max(cores, rows // 4), cores)
    times, work = [], 0.0
    for _ in range(args.steps):
        st, w = cpu_step_sample(host, rows, cores)
        times.append(st)
        work += w
    ms = 1e3 * statistics.mean(times)
    v = 1e3 / ms
    sample = (f"each step: {rows} of {T * HQ} query rows per attention call (4 drafter + 1 verify) sliced over "
              f"{cores} threads, scaled by {T * HQ}/{rows}; greedy and sampled acceptance over all 16 x {V} "
              "logits in full on one thread")
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "blocks/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "global_batch": 1, "seq_len": CTX,
                   "parallelism": f"none ({cores} host threads)", "l2": "n/a (CPU)"},
        "cpu_baseline": {"value": v, "unit": "blocks/s", "cores": cores, "kind": "oracle", "sample": sample,
                         "cpu_seconds": work},
        "e2e": {"value": v, "unit": "blocks/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# ranks (one replica per GPU; no collective on the data path)
# ---------------------------------------------------------------------------

def max_over_ranks(x, world, device):
    """The largest of the ranks' values (every rank passes its own): the
    timed region of a run is that of its slowest rank."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(world, steps_per_rank, secs):
    """Blocks verified by all ranks together per second of the slowest rank."""
    return world * steps_per_rank / secs


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--copies", type=int, default=4, help="rotated input copies (> 2x L2 in total)")
    ap.add_argument("--no-graph", action="store_true", help="launch eagerly (profiling)")
    ap.add_argument("--skip-cpu-baseline", action="store_true")
    ap.add_argument("--skip-extras", action="store_true", help="no per-kernel / e2e passes (profiling)")
    ap.add_argument("--no-soak", action="store_true", help="no 1.5 s soak before timing (profiling)")
    ap.add_argument("--ref-rows", type=int, default=8)
    ap.add_argument("--cpu-rows", type=int, default=32)
    ap.add_argument("--profile-case", choices=["cfg3-verify", "cfg5-verify", "accept-greedy-b8", "accept-sample-b4",
                                               "project-prefill", "project-append", "latent"], default=None,
                    help="profiling: run only this call, --warmup + --steps times eagerly, print nothing")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return 0
        reference_arm(args)
        return 0

    import torch
    import torch.distributed as dist
    from serving_sd_verify_gb300 import build, sd_verify as S

    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    if rank == 0:
        build.build()
    if world > 1:
        dist.barrier()
    S.load()

    if args.profile_case:
        profile_case(S, device, args)
        return 0

    host = make_inputs(device)
    sets = [DeviceSet(host, device, S) for _ in range(args.copies)]
    torch.cuda.synchronize()   # inputs and zeroed workspaces are written before another stream reads them
    resident = sum(s.nbytes() for s in sets)
    log(f"[bench] {args.copies} input copies, {resident / 1e6:.0f} MB resident (L2 {L2_BYTES / 1e6:.0f} MB)")
    stream = torch.cuda.Stream(device)

    # warm-up (eager; also primes per-device state before any capture)
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            run_step(S, sets[i % len(sets)], stream)
    torch.cuda.synchronize()
    assert S.sd_fault_word() == 0, "device guard fired during warm-up"

    graph = None
    if not args.no_graph:
        graph = graph_of(S, sets, stream, ("draft", "verify", "greedy", "sample"))
        graph.replay()
        torch.cuda.synchronize()

    sampler = ClockSampler(local_rank)
    # soak so that the clock sampler sees the GPU under this load before timing
    soak_until = time.time() + (0.0 if args.no_soak else 1.5)
    with torch.cuda.stream(stream):
        while time.time() < soak_until:
            if graph is not None:
                graph.replay()
            else:
                run_step(S, sets[0], stream)
            torch.cuda.synchronize()

    reps = max(1, math.ceil(args.steps / len(sets))) if graph is not None else args.steps
    steps_done = reps * len(sets) if graph is not None else args.steps
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_wall0 = time.time()
    with torch.cuda.stream(stream):
        e0.record(stream)
        if graph is not None:
            for _ in range(reps):
                graph.replay()
        else:
            for i in range(steps_done):
                run_step(S, sets[i % len(sets)], stream)
        e1.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    if world > 1:
        dist.barrier()
    sampler.stop()
    secs = max_over_ranks(e0.elapsed_time(e1) / 1e3, world, device)
    clocks = sampler.summary(t_wall0, t_wall1)
    ms_per_step = 1e3 * secs / steps_done
    value = whole_job_value(world, steps_done, secs)
    assert S.sd_fault_word() == 0, "device guard fired during the timed region"

    # ---- per-call timing of each kernel class: L2 flushed before every call,
    # CUDA events on the launching stream around the call ----
    kernels = {}
    if not args.skip_extras:
        flush = torch.empty(320 * 1024 * 1024, dtype=torch.uint8, device=device)
        n_rep = 30
        for name, part, launches in (("draft_attention", "draft", LAYERS), ("verify_attention", "verify", 1),
                                     ("accept_greedy", "greedy", 1), ("accept_sample", "sample", 1),
                                     ("verify_tree_attention", "tree_verify", 1),
                                     ("accept_tree_greedy", "tree_greedy", 1)):
            evs = []
            with torch.cuda.stream(stream):
                for i in range(n_rep):
                    flush.zero_()
                    e_a, e_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e_a.record(stream)
                    run_step(S, sets[i % len(sets)], stream, (part,))
                    e_b.record(stream)
                    evs.append((e_a, e_b))
            torch.cuda.synchronize()
            per_launch = sum(a.elapsed_time(b) for a, b in evs[3:]) / 1e3 / ((n_rep - 3) * launches)
            kernels[name] = {"us_per_call": per_launch * 1e6, "calls_per_step": launches,
                             "algorithmic_bytes_per_call": BYTES[name],
                             "GBps": BYTES[name] / per_launch / 1e9}
        proj = ProjSet(host["proj"], device)
        for name, n_rows in (("project_prefill", CTX), ("project_append", APPEND)):
            # one call captured in a graph, so the binding's host time stays
            # out of the event window
            with torch.cuda.stream(stream):
                proj.run(S, stream, n_rows)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                proj.run(S, stream, n_rows)
            evs = []
            with torch.cuda.stream(stream):
                for i in range(n_rep):
                    flush.zero_()
                    e_a, e_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e_a.record(stream)
                    g.replay()
                    e_b.record(stream)
                    evs.append((e_a, e_b))
            torch.cuda.synchronize()
            del g
            per = sum(a.elapsed_time(b) for a, b in evs[3:]) / 1e3 / (n_rep - 3)
            kernels[name] = {"us_per_call": per * 1e6, "calls_per_step": 0, "kernel_launches_per_call": 1,
                             "rows": n_rows, "path": S.sd_last_projector_path()}
        # a whole cycle (draft x4, verify, accept, append, commit) and the
        # commit alone (append + commit), each one graph replay after an L2 flush
        cyc = CycleSet(sets[0], proj, device, S)
        for name, fn in (("spec_cycle", cyc.cycle), ("commit", cyc.commit)):
            with torch.cuda.stream(stream):
                fn(S, stream)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                fn(S, stream)
            ctx_a = int(cyc.ctx.item())
            evs = []
            with torch.cuda.stream(stream):
                for i in range(n_rep):
                    flush.zero_()
                    e_a, e_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e_a.record(stream)
                    g.replay()
                    e_b.record(stream)
                    evs.append((e_a, e_b))
            torch.cuda.synchronize()
            del g
            per = sum(a.elapsed_time(b) for a, b in evs[3:]) / 1e3 / (n_rep - 3)
            grown = int(cyc.ctx.item()) - ctx_a
            kernels[name] = {"us_per_call": per * 1e6, "calls_per_step": 0,
                             "kernel_launches_per_call": cyc.launches if name == "spec_cycle" else 2,
                             "tokens_committed_per_call": grown / n_rep}
        assert S.sd_fault_word() == 0, "device guard fired in the cycle measurement"
        kc_ = kernels["spec_cycle"]
        kc_["committed_tokens_per_s"] = kc_["tokens_committed_per_call"] / (kc_["us_per_call"] * 1e-6)
        kc_["note"] = ("one speculative cycle in one CUDA graph: 4 drafter layers, target verify, greedy "
                       "acceptance, drafter-context append of the committed rows, commit (ctx_len, tokens, "
                       "anchor); no host round trip; the context grows by the committed tokens every replay")
        kernels["commit"]["note"] = ("the device-side commit alone: projector append of the committed rows "
                                     "(weights read once) + token / length update")
        del cyc, proj
        # the SpecFLASH latent compressor (three launches), one graph replay after an L2 flush
        from serving_sd_verify_gb300 import workloads as W
        lq, lf = W.latent_inputs(frames=LC_FRAMES, N=LC_N, Cq=LC_C, d=LC_D, seed=16)
        lq, lf = lq.to(device), lf.to(device)
        lout = torch.empty(LC_FRAMES, LC_C, LC_D, dtype=torch.bfloat16, device=device)
        lws = S.workspace(S.sd_latent_compress_workspace_size(LC_FRAMES, LC_N, LC_C, LC_D), device)
        with torch.cuda.stream(stream):
            S.sd_latent_compress(lq, lf, lout, lws, stream)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            S.sd_latent_compress(lq, lf, lout, lws, stream)
        evs = []
        with torch.cuda.stream(stream):
            for i in range(n_rep):
                flush.zero_()
                e_a, e_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e_a.record(stream)
                g.replay()
                e_b.record(stream)
                evs.append((e_a, e_b))
        torch.cuda.synchronize()
        del g, lq, lf, lout, lws
        per = sum(a.elapsed_time(b) for a, b in evs[3:]) / 1e3 / (n_rep - 3)
        kernels["latent_compress"] = {
            "us_per_call": per * 1e6, "calls_per_step": 0, "kernel_launches_per_call": 3,
            "algorithmic_bytes_per_call": LC_BYTES, "GBps": LC_BYTES / per / 1e9,
            "TFLOPs": LC_FLOPS / per / 1e12,
            "note": (f"SpecFLASH latent compressor softmax(Q.F^T).F: {LC_FRAMES} frames x {LC_N} visual features "
                     f"(d {LC_D}, LLaVA-1.5-7B) -> {LC_C} latents each; scores, softmax and output kernels; "
                     "features read from HBM once, re-read from L2; not part of the step")}
        # acceptance at the batched workloads -- greedy over the ragged batch's
        # logits (B 8) and the sampled rule of the 72B-shaped workload (B 4) --
        # issued back to back in one graph over 4 input copies (more than L2)
        acceptance = {}
        g8 = W.greedy_inputs(B=8, T=T, V=V, seed=103)
        s4 = W.sample_inputs(B=4, T=T, V=V, seed=105, draft_seed=1235)
        g1 = W.greedy_inputs(B=1, T=T, V=V, seed=101)
        s1 = W.sample_inputs(B=1, T=T, V=V, seed=106, draft_seed=1236)
        for name, Bn, n_copies, make, call, nbytes in (
                ("greedy_b8", 8, 4,
                 lambda: (g8["draft"].to(device), g8["logits"].to(device),
                          S.workspace(S.sd_accept_greedy_workspace_size(8, T, V), device)),
                 lambda c, n_, x_: S.sd_accept_greedy(c[0], c[1], n_, x_, c[2], stream),
                 8 * (T * V * 2 + (T - 1) * 4 + 8)),
                ("sample_b4", 4, 4,
                 lambda: (s4["draft"].to(device), s4["q"].to(device), s4["logits"].to(device),
                          S.workspace(S.sd_accept_sample_workspace_size(4, T, V), device)),
                 lambda c, n_, x_: S.sd_accept_sample(c[0], c[1], c[2], 1.0, 1234, 0, n_, x_, c[3], stream),
                 4 * (T * V * 2 + V * 2 + V * 4 + (T - 1) * 8 + 8)),
                # one sequence: 32 input copies, so that the copies exceed L2
                ("greedy_b1", 1, 32,
                 lambda: (g1["draft"].to(device), g1["logits"].to(device),
                          S.workspace(S.sd_accept_greedy_workspace_size(1, T, V), device)),
                 lambda c, n_, x_: S.sd_accept_greedy(c[0], c[1], n_, x_, c[2], stream),
                 1 * (T * V * 2 + (T - 1) * 4 + 8)),
                ("sample_b1", 1, 32,
                 lambda: (s1["draft"].to(device), s1["q"].to(device), s1["logits"].to(device),
                          S.workspace(S.sd_accept_sample_workspace_size(1, T, V), device)),
                 lambda c, n_, x_: S.sd_accept_sample(c[0], c[1], c[2], 1.0, 1234, 0, n_, x_, c[3], stream),
                 1 * (T * V * 2 + V * 2 + V * 4 + (T - 1) * 8 + 8))):
            cps = [make() for _ in range(n_copies)]
            n_ = torch.zeros(Bn, dtype=torch.int32, device=device)
            x_ = torch.zeros(Bn, dtype=torch.int32, device=device)
            with torch.cuda.stream(stream):
                for c in cps:
                    call(c, n_, x_)
            torch.cuda.synchronize()
            ga = torch.cuda.CUDAGraph()
            with torch.cuda.graph(ga, stream=stream):
                for i in range(2 * n_copies):
                    call(cps[i % n_copies], n_, x_)
            reps_a = 25
            with torch.cuda.stream(stream):
                for _ in range(3):
                    ga.replay()
                e_a, e_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e_a.record(stream)
                for _ in range(reps_a):
                    ga.replay()
                e_b.record(stream)
            torch.cuda.synchronize()
            del ga, cps
            per = e_a.elapsed_time(e_b) / 1e3 / (reps_a * 2 * n_copies)
            acceptance[name] = {"us_per_call": per * 1e6, "algorithmic_bytes_per_call": nbytes,
                                "GBps": nbytes / per / 1e9}
        del g8, s4, g1, s1
        # verify attention of the ragged batch and of the 72B-shaped batch at
        # full size, and the drafter's layers split into the HBM-cold first one
        # and the L2-resident rest
        per_config = {}
        for n in (3, 5):
            per_config[n] = config_verify_pass(S, device, stream, n)
        per_config["draft"] = drafter_layer_pass(S, sets[0], stream, flush)
        # the four layers back to back in one graph, as inside the step (the
        # projected context stays in L2 after the first layer)
        ds0 = sets[0]
        per_config["draft_b2b"] = time_back_to_back(
            [(lambda L=L, li=li: S.sd_draft_block_attention(L[0], ds0.kc, ds0.vc, ds0.nctx, CTX, L[1], L[2],
                                                            ds0.dout[li], 1.0, ds0.ws_d, stream))
             for li, L in enumerate(ds0.layers)], LAYERS, stream)
        per_config["tree60"] = tree60_pass(S, device, stream)
        tpk, tsrc = bf16_peak(sustained=False)
        kp = kernels["project_prefill"]
        kp["TFLOPs"] = PROJ_PREFILL_FLOPS / (kp["us_per_call"] * 1e-6) / 1e12
        kp["frac_of_bf16_peak"] = kp["TFLOPs"] / tpk
        kp["peak_source"] = tsrc
        kp["note"] = (f"drafter K/V projector over the whole {CTX}-row context ({HD} -> 2 x {HKV * D}), "
                      "tensor cores; a prefill-time call, not part of the step")
        ka = kernels["project_append"]
        ka["algorithmic_bytes_per_call"] = BYTES["project_append"]
        ka["GBps"] = BYTES["project_append"] / (ka["us_per_call"] * 1e-6) / 1e9
        ka["note"] = f"the {APPEND} rows one cycle commits, appended to the drafter's context; not part of the step"
        del flush
        kernels["draft_attention"]["note"] = ("average over the 4 layers of one step; they share one projected "
                                              "context, so layers 2-4 read it from L2 and only the first call "
                                              "is HBM-bound")
        for name in ("verify_tree_attention", "accept_tree_greedy"):
            kernels[name]["note"] = ("tree verification (a seeded 16-node draft tree), timed alone; not part of "
                                     "the step, which uses the chain calls")
        for name, nl in (("draft_attention", ATTN_LAUNCHES["draft"]), ("verify_attention", ATTN_LAUNCHES["verify"]),
                         ("accept_greedy", 1),
                         ("accept_sample", ATTN_LAUNCHES["sample"]), ("verify_tree_attention", ATTN_LAUNCHES["verify"]),
                         ("accept_tree_greedy", 1)):
            kernels[name]["kernel_launches_per_call"] = nl

    # ---- the verify attention back to back, as in the step: one graph of
    # 2 x copies calls rotating over the input copies (their K/V together
    # exceed L2, so every call streams its cache from HBM); events around
    # the replays, average over the calls ----
    if kernels:
        n_calls = 2 * len(sets)
        gv = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gv, stream=stream):
            for i in range(n_calls):
                run_step(S, sets[i % len(sets)], stream, ("verify",))
        reps_v = 25
        with torch.cuda.stream(stream):
            for _ in range(3):
                gv.replay()
            e_a, e_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e_a.record(stream)
            for _ in range(reps_v):
                gv.replay()
            e_b.record(stream)
        torch.cuda.synchronize()
        del gv
        per = e_a.elapsed_time(e_b) / 1e3 / (reps_v * n_calls)
        kv = kernels["verify_attention"]
        kv["us_per_call_back_to_back"] = per * 1e6
        kv["GBps_back_to_back"] = BYTES["verify_attention"] / per / 1e9
        kv["note"] = ("us_per_call: one call after an L2 flush (cold, launch latency included); "
                      "us_per_call_back_to_back: average over calls issued back to back in one graph, inputs "
                      f"rotating over {len(sets)} copies ({len(sets) * 52} MB of K/V, more than L2)")

    # ---- roofline: the verify attention (the headline kernel) ----
    roofline = None
    if kernels:
        peak, peak_src = hbm_peak(sustained=False)
        k = kernels["verify_attention"]
        achieved = k["GBps_back_to_back"]
        traffic = ncu_traffic("verify_attention")
        roofline = {"kernel": "verify attention (one sd_verify_attention call: split pass with the "
                              "log-sum-exp merge inside the same kernel); traffic is that kernel's DRAM "
                              "bytes per launch",
                    "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                    "frac": achieved / peak, "peak_source": peak_src,
                    "timing": "average duration of calls issued back to back in one CUDA graph with inputs "
                              "larger than L2 (as inside the timed step); the cold single-call figure is "
                              "kernels.verify_attention.GBps",
                    "frac_cold_single_call": k["GBps"] / peak,
                    "traffic": traffic,
                    "algorithmic_bytes_per_launch": BYTES["verify_attention"],
                    "units_per_launch": f"{CTX + T - 1} keys x {HKV} kv heads (K and V bf16, D {D}) + Q + out"}
        for name, kk in kernels.items():
            if "GBps" in kk:
                kk["frac_of_peak"] = kk["GBps"] / peak
        for name, kk in acceptance.items():
            kk["frac_of_peak"] = kk["GBps"] / peak
        # short scalar keys, one figure each, per workload
        t3, b3 = per_config[3]
        t5, b5 = per_config[5]
        tg8 = acceptance["greedy_b8"]["us_per_call"] * 1e-6
        ts4 = acceptance["sample_b4"]["us_per_call"] * 1e-6
        t_l1, t_l234 = per_config["draft"]
        draft_flops = 2 * 2 * T * HQ * (CTX + T) * D
        tpk_, _ = bf16_peak(sustained=False)
        roofline.update({
            "cfg2_verify_us": k["us_per_call_back_to_back"],
            "cfg3_verify_us": t3 * 1e6, "cfg3_verify_GBps": b3 / t3 / 1e9, "cfg3_verify_frac": b3 / t3 / 1e9 / peak,
            "cfg3_verify_bytes": b3,
            "cfg5_verify_us": t5 * 1e6, "cfg5_verify_GBps": b5 / t5 / 1e9, "cfg5_verify_frac": b5 / t5 / 1e9 / peak,
            "cfg5_verify_bytes": b5,
            "accept_greedy_b8_us": tg8 * 1e6, "accept_greedy_b8_frac": acceptance["greedy_b8"]["frac_of_peak"],
            "accept_sample_b4_us": ts4 * 1e6, "accept_sample_b4_frac": acceptance["sample_b4"]["frac_of_peak"],
            "accept_greedy_b1_us": kernels["accept_greedy"]["us_per_call"],
            "accept_sample_b1_us": kernels["accept_sample"]["us_per_call"],
            "accept_greedy_b1_us_back_to_back": acceptance["greedy_b1"]["us_per_call"],
            "accept_sample_b1_us_back_to_back": acceptance["sample_b1"]["us_per_call"],
            "cfg3_blocks_per_s": 8 / (t3 + tg8),
            "cfg5_blocks_per_s": 4 / (t5 + ts4),
            "draft_l1_us": t_l1 * 1e6, "draft_l1_frac": BYTES["draft_attention"] / t_l1 / 1e9 / peak,
            "draft_l234_us": t_l234 * 1e6,
            "draft_l234_tensor_frac": draft_flops / t_l234 / 1e12 / tpk_,
            "draft_layer_us_back_to_back": per_config["draft_b2b"] * 1e6,
            "draft_layer_tensor_frac_back_to_back": draft_flops / per_config["draft_b2b"] / 1e12 / tpk_,
            "cfg4_draft_blocks_per_s": 1.0 / (t_l1 + (LAYERS - 1) * t_l234),
        })
        t_tv, t_ta, b_tv, b_ta = per_config["tree60"]
        roofline.update({
            "tree60_verify_us": t_tv * 1e6, "tree60_verify_frac": b_tv / t_tv / 1e9 / peak,
            "tree60_accept_us": t_ta * 1e6, "tree60_accept_frac": b_ta / t_ta / 1e9 / peak,
            "tree60_blocks_per_s": 1.0 / (t_tv + t_ta),
            "chain16_blocks_per_s": 1.0 / (k["us_per_call_back_to_back"] * 1e-6 +
                                           kernels["accept_greedy"]["us_per_call"] * 1e-6),
        })
        # the same per-call times in SM cycles at the median clock sampled
        # during the timed step, so that a change can be judged when the
        # clock differs between runs
        if clocks and clocks.get("sm_mhz"):
            mhz = float(clocks["sm_mhz"])
            roofline["kcycles_at_sampled_clock"] = {
                "sm_mhz": mhz,
                "step": ms_per_step * 1e3 * mhz / 1e3,
                "cfg2_verify": k["us_per_call_back_to_back"] * mhz / 1e3,
                "cfg5_verify": t5 * 1e6 * mhz / 1e3,
                "draft_l234": t_l234 * 1e6 * mhz / 1e3,
                "accept_greedy_b8": tg8 * 1e6 * mhz / 1e3,
                "accept_sample_b4": ts4 * 1e6 * mhz / 1e3,
            }
        roofline["acceptance_back_to_back"] = dict(acceptance, note=(
            "acceptance kernels at the batched workloads (greedy over 8 sequences' logits, the sampled rule "
            "over 4; 4 input copies) and for one sequence (32 copies), calls issued back to back in one "
            "graph over input copies larger than L2"))

    # ---- end to end: host buffers, copies inside the timed region ----
    e2e = None
    if not args.skip_extras:
        e2e = e2e_pass(S, host, sets[0], device, stream, max(20, min(200, args.steps // 10)))

    # ---- CPU baseline (rank 0, N = 1 only) ----
    cpu = None
    if rank == 0 and world == 1 and not args.skip_cpu_baseline:
        try:
            cpu = cpu_baseline_leg(host, args)
        except Exception as exc:  # the GPU figures are still reported
            cpu = {"value": None, "unit": "blocks/s", "cores": host_cores(), "kind": "oracle",
                   "sample": f"failed: {type(exc).__name__}: {exc}"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "blocks/s", "n_gpus": world, "steps": steps_done,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": WORKLOAD, "global_batch": world, "seq_len": CTX,
                       "parallelism": "replicas" if world > 1 else "none",
                       "l2": f"inputs rotate over {len(sets)} copies ({resident / 1e6:.0f} MB > 2x L2)",
                       "graph": graph is not None},
            "roofline": roofline,
            "kernels": kernels,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": steps_done * kernels_per_step(),
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def cpu_baseline_leg(host, args):
    """The oracle on a bounded sample of the step, on one thread and on every host core."""
    import oracle
    oracle.build()
    cores = host_cores()
    legs = {}
    for threads, rows_per_call in ((1, args.cpu_rows), (cores, min(T * HQ, args.cpu_rows * cores))):
        n_s, total, work = 0, 0.0, 0.0
        while work < 6.0 and n_s < 20:
            st, w = cpu_step_sample(host, rows_per_call, threads)
            total += st
            work += w
            n_s += 1
        legs[threads] = (n_s / total, n_s, work, rows_per_call)
    v_all, n_all, w_all, r_all = legs[cores]
    v_one, n_one, w_one, r_one = legs[1]
    cpu = {"value": v_all, "unit": "blocks/s", "cores": cores, "kind": "oracle",
           "value_1_thread": v_one,
           "sample": f"{n_all} steps on {cores} threads (attention rows sliced over them), per step "
                     f"{r_all} of {T * HQ} query rows per attention call scaled by {T * HQ}/{r_all}, "
                     f"acceptance in full on one thread, {w_all:.1f} s wall; value_1_thread: {n_one} steps "
                     f"of {r_one} rows per call on one thread, {w_one:.1f} s"}
    return cpu


def e2e_pass(S, host, ds, device, stream, steps):
    """Blocks/s through the public binding with the per-step inputs in pinned
    host memory: each step copies them in, runs the step, and reads the results
    back.  The long-context K/V (target cache, projected drafter context) is
    resident state built at prefill and is not re-sent per block; the block's
    own new K/V slots are written into the cache each step.  The per-block
    inputs sit in two packed pinned buffers (what the attention calls read;
    what the acceptance calls read) mirrored by two device buffers whose views
    the calls take, so a block costs a handful of copies, not one per tensor."""
    import types
    import torch
    a, g, d, s = host["attn"], host["greedy"], host["drafter"], host["sample"]

    def packed(tensors):
        offs, n = [], 0
        for t in tensors:
            offs.append(n)
            n += (t.numel() * t.element_size() + 255) // 256 * 256
        hbuf = torch.empty(n, dtype=torch.uint8).pin_memory()
        dbuf = torch.empty(n, dtype=torch.uint8, device=device)
        views = []
        for t, o in zip(tensors, offs):
            nb = t.numel() * t.element_size()
            hbuf[o:o + nb].view(t.dtype).view(t.shape).copy_(t)
            views.append(dbuf[o:o + nb].view(t.dtype).view(t.shape))
        return hbuf, dbuf, views

    att_in = [a["q"].contiguous()] + [x.contiguous() for L in d["layers"] for x in (L["q"], L["kb"], L["vb"])]
    acc_in = [g["logits"].contiguous(), g["draft"].contiguous(), s["q"].contiguous(), s["draft"].contiguous()]
    h_att, d_att, v_att = packed(att_in)
    h_acc, d_acc, v_acc = packed(acc_in)
    h_blk_k = a["k"][:, CTX - 1:CTX + T - 1].contiguous().pin_memory()
    h_blk_v = a["v"][:, CTX - 1:CTX + T - 1].contiguous().pin_memory()
    # the step's results -- verify output and the four accept ids -- side by
    # side in one device buffer, stored into pinned host memory by one
    # sd_store_to_host call (the GPU's own stores: for these 229 KB sooner
    # done than a copy-engine transfer)
    out_bytes = 1 * T * HQ * D * 4
    d_outres = torch.zeros(out_bytes + 256, dtype=torch.uint8, device=device)
    h_outres = torch.empty(out_bytes + 256, dtype=torch.uint8).pin_memory()
    res = d_outres[out_bytes:out_bytes + 16].view(torch.int32)
    e2 = types.SimpleNamespace(**vars(ds))
    e2.out = d_outres[:out_bytes].view(torch.float32).view(1, T, HQ, D)
    e2.q = v_att[0]
    e2.layers = [tuple(v_att[1 + 3 * li: 4 + 3 * li]) for li in range(LAYERS)]
    e2.logits, e2.draft, e2.sq, e2.sdraft = v_acc
    e2.n, e2.c, e2.sn, e2.snx = res[0:1], res[1:2], res[2:3], res[3:4]
    h2d = h_att.numel() + h_acc.numel() + h_blk_k.numel() * 2 + h_blk_v.numel() * 2
    d2h = out_bytes + 16
    side = torch.cuda.Stream(device)

    def body():
        cur = torch.cuda.current_stream()
        # what the attention calls read goes first, alone, on the main stream;
        # then the block's own K/V slots (read from the verify on) and the
        # acceptance inputs (target logits, draft ids and probabilities: 14.6
        # of the 15.3 MB) travel on a side stream while the drafter layers
        # run, and join before the verify call.  The side copies start after
        # the first one: started together, they slow it down
        d_att.copy_(h_att, non_blocking=True)
        side.wait_stream(cur)
        with torch.cuda.stream(side):
            ds.k[:, CTX - 1:CTX + T - 1].copy_(h_blk_k, non_blocking=True)
            ds.v[:, CTX - 1:CTX + T - 1].copy_(h_blk_v, non_blocking=True)
            d_acc.copy_(h_acc, non_blocking=True)
        run_step(S, e2, stream, ("draft",))
        cur.wait_stream(side)
        run_step(S, e2, stream, ("verify", "greedy", "sample"))
        S.sd_store_to_host(h_outres[:d2h], d_outres[:d2h], cur)

    def one():
        body()
        torch.cuda.current_stream().synchronize()

    def timed(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(steps):
            fn()
        return time.perf_counter() - t0

    with torch.cuda.stream(stream):
        sec_eager = timed(one)
        # the same step -- copies in, the C-ABI calls, results out -- captured
        # once into a CUDA graph and replayed per block, the host waiting for
        # each block's results before the next (as a serving loop that refills
        # the pinned input buffers between blocks would)
        body()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            body()

        def replay():
            g.replay()
            stream.synchronize()
        sec = timed(replay)
        del g
    return {"value": steps / sec, "unit": "blocks/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": steps, "eager_value": steps / sec_eager,
            "note": "per-block inputs from pinned host memory (two packed buffers plus the block's K/V slots), "
                    "results stored into pinned host memory every step by one sd_store_to_host call (SM "
                    "stores), the host waiting for them; the block's K/V "
                    "slots and the acceptance inputs copied on a side stream while the drafter layers run, "
                    "after the attention inputs' copy; "
                    "the step (copies and C-ABI calls) replayed "
                    "from one CUDA graph (eager_value: the same step issued call by call from Python); context "
                    "K/V resident"}


if __name__ == "__main__":
    sys.exit(main())
