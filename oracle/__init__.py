"""fp64 CPU oracle for block verification -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The GPU library neither imports nor
links it, and the two share no code: the only thing both sides see are the
seeded inputs from ``serving_sd_verify_gb300.workloads``.

The arithmetic lives in ``sd_oracle.c`` (plain C99, fp64, single thread);
this module only marshals numpy arrays through ctypes.  See that file's
header for the passages each routine follows.

Pins (tests/test_oracle_*.py) fix every routine to something other than
itself: Philox known-answer vectors, textbook decode attention, closed forms
(constant keys, one key), brute force on tiny shapes, the worked cycle of the
VFlash-FM project page, the autoregressive-equivalence invariant, a
chi-square test of the sampled rule, and for the latent compressor closed
forms (equal features, zero queries, a one-hot limit), a hand example and
the library's scaled-dot-product attention.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sd_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_sd_oracle.so")
_lock = threading.Lock()
_lib = None

_dp = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")
_ip = np.ctypeslib.ndpointer(dtype=np.int32, flags="C_CONTIGUOUS")
_lp = np.ctypeslib.ndpointer(dtype=np.int64, flags="C_CONTIGUOUS")
_up = np.ctypeslib.ndpointer(dtype=np.uint32, flags="C_CONTIGUOUS")
_u64p = np.ctypeslib.ndpointer(dtype=np.uint64, flags="C_CONTIGUOUS")


def build(force: bool = False) -> str:
    """Compile sd_oracle.c into _sd_oracle.so beside it (gcc, no fast-math)."""
    with _lock:
        if (not force and os.path.exists(_LIB_PATH)
                and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
            return _LIB_PATH
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-ffp-contract=off",
               "-fno-fast-math", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
        return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB_PATH)
    lib.oracle_philox4x32_10_batch.argtypes = [_up, _up, _up, ctypes.c_long]
    lib.oracle_philox4x32_10_batch.restype = None
    lib.oracle_uniform.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint32,
                                   ctypes.c_uint32, ctypes.c_uint32]
    lib.oracle_uniform.restype = ctypes.c_double
    lib.oracle_attention_rows.argtypes = [
        _dp, _dp, _dp, ctypes.c_void_p, ctypes.c_void_p, _ip, ctypes.c_int,
        ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        ctypes.c_double, ctypes.c_long, ctypes.c_long, ctypes.c_void_p, ctypes.c_long,
        _dp, ctypes.c_void_p]
    lib.oracle_attention_rows.restype = ctypes.c_int
    lib.oracle_lse_merge.argtypes = [_dp, _dp, ctypes.c_int, ctypes.c_int, _dp]
    lib.oracle_lse_merge.restype = ctypes.c_double
    lib.oracle_accept_greedy.argtypes = [_ip, _dp, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                         _ip, _ip, ctypes.c_void_p]
    lib.oracle_accept_greedy.restype = ctypes.c_int
    lib.oracle_accept_sample.argtypes = [_ip, _dp, _dp, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_double, ctypes.c_uint64, ctypes.c_uint32,
                                         _ip, _ip, ctypes.c_void_p]
    lib.oracle_accept_sample.restype = ctypes.c_int
    _up32 = np.ctypeslib.ndpointer(dtype=np.uint32, flags="C_CONTIGUOUS")
    lib.oracle_tree_attention_rows.argtypes = [
        _dp, _dp, _dp, _ip, _u64p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_void_p, ctypes.c_long, _dp]
    lib.oracle_tree_attention_rows.restype = ctypes.c_int
    lib.oracle_accept_tree_greedy.argtypes = [_ip, _ip, _dp, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                              _ip, _ip, _ip, _ip]
    lib.oracle_accept_tree_greedy.restype = ctypes.c_int
    lib.oracle_project_rows.argtypes = [_dp, _dp, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                        ctypes.c_long, _dp]
    lib.oracle_project_rows.restype = ctypes.c_int
    lib.oracle_commit_tokens.argtypes = [_ip, ctypes.c_int, ctypes.c_void_p, _ip, _ip, ctypes.c_int, ctypes.c_int,
                                         _ip, ctypes.c_int, ctypes.c_void_p, _ip, _ip, ctypes.c_int, _ip, _ip]
    lib.oracle_commit_tokens.restype = ctypes.c_int
    _u8 = np.ctypeslib.ndpointer(dtype=np.uint8, flags="C_CONTIGUOUS")
    lib.oracle_compact_tree_kv.argtypes = [_u8, _u8, ctypes.c_long, ctypes.c_long, ctypes.c_long, ctypes.c_int,
                                           _ip, _ip, _ip, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_int, _ip]
    lib.oracle_compact_tree_kv.restype = ctypes.c_int
    lib.oracle_latent_compress.argtypes = [_dp, _dp, _dp, ctypes.c_int, ctypes.c_int, ctypes.c_int, _dp]
    lib.oracle_latent_compress.restype = ctypes.c_int
    _lib = lib
    return lib


def _f64(x) -> np.ndarray:
    """Exact fp64 copy of a numpy array or a CPU torch tensor (bf16 / fp32 values)."""
    if hasattr(x, "detach"):  # torch tensor: widen on the CPU, exactly
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(x, dtype=np.float64)


def _i32(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").numpy()
    return np.ascontiguousarray(x, dtype=np.int32)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


# --------------------------------------------------------------------------
# Philox4x32-10
# --------------------------------------------------------------------------

def philox4x32_10(counters, key) -> np.ndarray:
    """counters [n, 4] uint32, key [2] uint32 -> [n, 4] uint32."""
    ctr = np.ascontiguousarray(counters, dtype=np.uint32).reshape(-1, 4)
    k = np.ascontiguousarray(key, dtype=np.uint32).reshape(2)
    out = np.empty_like(ctr)
    _load().oracle_philox4x32_10_batch(ctr, k, out, ctr.shape[0])
    return out


def uniform(seed: int, row: int, batch: int, stream: int, offset: int) -> float:
    return _load().oracle_uniform(seed, row, batch, stream, offset)


# --------------------------------------------------------------------------
# Attention
# --------------------------------------------------------------------------

def attention_rows(q, k, v, nctx, scale, *, mode=0, kb=None, vb=None, rows=None,
                   key_range=None, return_lse=False):
    """Exact fp64 attention for the selected flat rows (b*T + j)*Hq + h.

    q [B,T,Hq,D]; k, v [B,Sc,Hkv,D]; nctx [B]; mode 0 = target verify (row j
    sees cache keys [0, nctx+j)), mode 1 = drafter (cache keys [0, nctx) then
    the T block keys kb, vb [B,T,Hkv,D]).  Returns out [n_rows, D] (and lse).
    """
    qd, kd, vd = _f64(q), _f64(k), _f64(v)
    B, T, Hq, D = qd.shape
    _, Sc, Hkv, _ = kd.shape
    n = _i32(nctx).reshape(B)
    kbd = _f64(kb) if kb is not None else None
    vbd = _f64(vb) if vb is not None else None
    rows_a = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64).reshape(-1)
    n_rows = B * T * Hq if rows_a is None else rows_a.size
    out = np.zeros((n_rows, D), dtype=np.float64)
    lse = np.zeros(n_rows, dtype=np.float64)
    lo, hi = (-1, -1) if key_range is None else key_range
    rc = _load().oracle_attention_rows(qd, kd, vd, _ptr(kbd), _ptr(vbd), n, int(mode),
                                       B, T, Hq, Hkv, D, Sc, float(scale), int(lo), int(hi),
                                       _ptr(rows_a), n_rows, out, _ptr(lse))
    if rc != 0:
        raise ValueError("oracle_attention_rows rejected its arguments")
    return (out, lse) if return_lse else out


def tree_attention_rows(q, k, v, nctx, tree_mask, scale, *, rows=None):
    """Exact fp64 tree-verify attention for the selected flat rows (b*T + j)*Hq + h.

    Node j of sequence b attends to cache keys [0, nctx-1) and to the block
    slots k (cache slot nctx-1+k) whose bit is set in tree_mask[b, j].
    q [B,T,Hq,D] (T <= 64); k, v [B,Sc,Hkv,D]; tree_mask [B,T] (bit k of a 64-bit
    word per node).  Returns out [n_rows, D].
    """
    qd, kd, vd = _f64(q), _f64(k), _f64(v)
    B, T, Hq, D = qd.shape
    _, Sc, Hkv, _ = kd.shape
    n = _i32(nctx).reshape(B)
    m = np.ascontiguousarray(np.asarray(tree_mask).astype(np.uint64).reshape(B * T))
    rows_a = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64).reshape(-1)
    n_rows = B * T * Hq if rows_a is None else rows_a.size
    out = np.zeros((n_rows, D), dtype=np.float64)
    rc = _load().oracle_tree_attention_rows(qd, kd, vd, n, m, B, T, Hq, Hkv, D, Sc, float(scale),
                                            _ptr(rows_a), n_rows, out)
    if rc != 0:
        raise ValueError("oracle_tree_attention_rows rejected its arguments")
    return out


def project_rows(hidden, weight, rows=None):
    """Exact fp64 linear map of the selected rows: hidden [N, Hd], weight [Dout, Hd]
    -> out [n_rows, Dout] = hidden[rows] @ weight^T."""
    h = _f64(hidden)
    w = _f64(weight)
    N, Hd = h.shape
    Dout = w.shape[0]
    rows_a = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64).reshape(-1)
    n_rows = N if rows_a is None else rows_a.size
    out = np.zeros((n_rows, Dout), dtype=np.float64)
    rc = _load().oracle_project_rows(h, w, N, Hd, Dout, _ptr(rows_a), n_rows, out)
    if rc != 0:
        raise ValueError("oracle_project_rows rejected its arguments")
    return out


def commit_tokens(proposals, n_accepted, next_token, ctx_len, out_tokens, out_len, ctx_cap, path=None):
    """Commit of a verified block on copies of the state.  proposals [B, P]
    (chain: the T-1 drafts; tree: the T node tokens, with path [B, T] the kept
    nodes by depth); n_accepted, next_token, ctx_len, out_len [B];
    out_tokens [B, out_cap].  Returns a dict with the new ctx_len, draft_ctx
    (= ctx_len - 1), out_tokens, out_len, anchor and status (1 = rejected, left
    unchanged)."""
    prop = np.ascontiguousarray(_i32(proposals))
    B = prop.shape[0]
    ps = prop.shape[1] if prop.ndim == 2 else 0
    prop = prop.reshape(-1) if prop.size else np.zeros(1, dtype=np.int32)
    n = np.ascontiguousarray(_i32(n_accepted).reshape(B))
    nx = np.ascontiguousarray(_i32(next_token).reshape(B))
    ctx = np.array(_i32(ctx_len).reshape(B), dtype=np.int32)
    toks = np.array(_i32(out_tokens), dtype=np.int32)
    out_cap = toks.shape[1]
    olen = np.array(_i32(out_len).reshape(B), dtype=np.int32)
    dctx = np.array(ctx - 1, dtype=np.int32)
    anchor = np.full(B, -1, dtype=np.int32)
    status = np.zeros(B, dtype=np.int32)
    if path is not None:
        pa = np.ascontiguousarray(_i32(path))
        T = pa.shape[1]
        pth = _ptr(pa.reshape(-1))
    else:
        pa, T, pth = None, ps + 1, None
    rc = _load().oracle_commit_tokens(prop, ps, pth, n, nx, B, T, ctx, int(ctx_cap), _ptr(dctx), toks, olen,
                                      out_cap, anchor, status)
    if rc != 0:
        raise ValueError("oracle_commit_tokens rejected its arguments")
    return {"ctx_len": ctx, "draft_ctx": dctx, "out_tokens": toks, "out_len": olen, "anchor": anchor,
            "status": status}


def compact_tree_kv(k_cache, v_cache, ctx_len, path, n_accepted):
    """Tree commit of the target's K/V cache on copies: k_cache, v_cache
    [B, S, Hkv, D] numpy arrays of any element type (moved as raw bytes);
    ctx_len (before the commit), n_accepted [B]; path [B, T].  Returns
    (k, v, status)."""
    k = np.array(k_cache, copy=True, order="C")
    v = np.array(v_cache, copy=True, order="C")
    B, S, Hkv, D = k.shape
    pa = np.ascontiguousarray(_i32(path))
    T = pa.shape[1]
    status = np.zeros(B, dtype=np.int32)
    kb, vb = k.view(np.uint8).reshape(-1), v.view(np.uint8).reshape(-1)
    rc = _load().oracle_compact_tree_kv(kb, vb, S * Hkv * D, Hkv * D, D, k.itemsize,
                                        np.ascontiguousarray(_i32(ctx_len).reshape(B)), pa.reshape(-1),
                                        np.ascontiguousarray(_i32(n_accepted).reshape(B)), B, T, S, Hkv, D, status)
    if rc != 0:
        raise ValueError("oracle_compact_tree_kv rejected its arguments")
    return k, v, status


def latent_compress(queries, features, values=None):
    """SpecFLASH latent compressor, exact fp64: queries [Cq, d], features
    [..., N, d] (a leading frame axis is allowed) -> [..., Cq, d] =
    softmax(queries . features^T) . values, values defaulting to features."""
    qv = _f64(queries)
    f = _f64(features)
    v = f if values is None else _f64(values)
    lead = f.shape[:-2]
    N, d = f.shape[-2:]
    Cq = qv.shape[0]
    f2 = f.reshape(-1, N, d)
    v2 = v.reshape(-1, N, d)
    out = np.zeros((f2.shape[0], Cq, d))
    for i in range(f2.shape[0]):
        o = np.zeros((Cq, d))
        rc = _load().oracle_latent_compress(qv, np.ascontiguousarray(f2[i]), np.ascontiguousarray(v2[i]),
                                            Cq, N, d, o)
        if rc != 0:
            raise ValueError("oracle_latent_compress rejected its arguments")
        out[i] = o
    return out.reshape(*lead, Cq, d)


def lse_merge(o_parts, lse_parts):
    """o_parts [S, D], lse_parts [S] -> (out [D], merged lse)."""
    o = _f64(o_parts)
    l = _f64(lse_parts).reshape(-1)
    S, D = o.shape
    out = np.zeros(D, dtype=np.float64)
    m = _load().oracle_lse_merge(o, l, S, D, out)
    return out, m


# --------------------------------------------------------------------------
# Acceptance
# --------------------------------------------------------------------------

def accept_greedy(draft_ids, logits, return_argmax=False):
    """draft [B,T-1] int, logits [B,T,V] -> (n_accepted [B], correction [B])."""
    lg = _f64(logits)
    B, T, V = lg.shape
    d = _i32(draft_ids).reshape(B, max(T - 1, 0))
    d = np.ascontiguousarray(d) if d.size else np.zeros(1, dtype=np.int32)
    n = np.zeros(B, dtype=np.int32)
    c = np.zeros(B, dtype=np.int32)
    am = np.zeros((B, T), dtype=np.int32)
    rc = _load().oracle_accept_greedy(d, lg, B, T, V, n, c, _ptr(am))
    if rc != 0:
        raise ValueError("oracle_accept_greedy rejected its arguments")
    return (n, c, am) if return_argmax else (n, c)


def accept_tree_greedy(tokens, parents, logits):
    """Greedy acceptance over a draft tree: tokens, parents [B,T] (parents[:,0] = -1,
    parents[:,j] < j), logits [B,T,V] -> (n_accepted [B], correction [B], best node [B],
    path [B,T] (accepted nodes at depth 1..n, then -1))."""
    lg = _f64(logits)
    B, T, V = lg.shape
    tk = np.ascontiguousarray(_i32(tokens).reshape(B, T))
    pa = np.ascontiguousarray(_i32(parents).reshape(B, T))
    n = np.zeros(B, dtype=np.int32)
    c = np.zeros(B, dtype=np.int32)
    best = np.zeros(B, dtype=np.int32)
    path = np.zeros((B, T), dtype=np.int32)
    rc = _load().oracle_accept_tree_greedy(tk, pa, lg, B, T, V, n, c, best, path)
    if rc != 0:
        raise ValueError("oracle_accept_tree_greedy rejected its arguments")
    return n, c, best, path


def accept_sample(draft_ids, draft_probs, logits, temperature, seed, offset=0,
                  return_diag=False):
    """Speculative accept / residual resample; returns (n_accepted, next_id[, diag])."""
    lg = _f64(logits)
    B, T, V = lg.shape
    q = _f64(draft_probs).reshape(B, T, V)
    d = _i32(draft_ids).reshape(B, max(T - 1, 0))
    d = np.ascontiguousarray(d) if d.size else np.zeros(1, dtype=np.int32)
    n = np.zeros(B, dtype=np.int32)
    nx = np.zeros(B, dtype=np.int32)
    diag = np.zeros((B, 2 * (T - 1) + 6), dtype=np.float64)
    rc = _load().oracle_accept_sample(d, q, lg, B, T, V, float(temperature), int(seed),
                                      int(offset), n, nx, _ptr(diag))
    if rc != 0:
        raise ValueError("oracle_accept_sample rejected its arguments")
    return (n, nx, diag) if return_diag else (n, nx)


def split_diag(diag, T):
    """Name the columns of accept_sample's diag array."""
    t1 = T - 1
    return {
        "u": diag[:, :t1], "ratio": diag[:, t1:2 * t1],
        "x": diag[:, 2 * t1], "S": diag[:, 2 * t1 + 1], "c_prev": diag[:, 2 * t1 + 2],
        "c_at": diag[:, 2 * t1 + 3], "mode": diag[:, 2 * t1 + 4], "u2": diag[:, 2 * t1 + 5],
    }
