"""Thin Python binding of libsdverify.so (ctypes).

Argument marshalling only: every function reads shapes, strides and device
pointers off torch tensors and calls the C entry point of the same name (see
include/sd_verify.h for what each computes and its contract).  Every step of
the computation runs in the library's CUDA kernels; there is no fallback.  If
the shared library has not been built, loading fails loudly.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsdverify.so")

SD_OK, SD_ERR_INVALID_ARG, SD_ERR_UNSUPPORTED, SD_ERR_WORKSPACE, SD_ERR_CUDA = range(5)
SD_BF16, SD_FP32 = 0, 1

# exported symbols, in header order
SYMBOLS = [
    "sd_verify_attention", "sd_verify_attention_workspace_size",
    "sd_draft_block_attention", "sd_draft_block_attention_workspace_size",
    "sd_accept_greedy", "sd_accept_greedy_workspace_size",
    "sd_verify_tree_attention", "sd_verify_tree_attention_workspace_size",
    "sd_accept_tree_greedy", "sd_accept_tree_greedy_workspace_size",
    "sd_accept_sample", "sd_accept_sample_workspace_size", "sd_accept_greedy_noalloc",
    "sd_philox4x32_10", "sd_status_string", "sd_last_error", "sd_version",
    "sd_fault_word", "sd_set_attention_path", "sd_last_attention_path", "sd_last_attention_launches",
    "sd_project_kv", "sd_set_projector_path", "sd_last_projector_path",
    "sd_set_sample_path", "sd_last_sample_path", "sd_set_wait_test",
    "sd_commit_tokens", "sd_compact_tree_kv", "sd_store_to_host", "sd_project_kv_commit",
    "sd_latent_compress", "sd_latent_compress_workspace_size",
]


class SdError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{_status_name(status)}: {msg}")
        self.status = status


class Strides(ctypes.Structure):
    _fields_ = [("b", ctypes.c_int64), ("s", ctypes.c_int64), ("h", ctypes.c_int64)]


_lib = None
_vp, _i, _sz, _f = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_float


def load():
    """Load the shared library (raises if it is missing: build it with build.build())."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: run serving_sd_verify_gb300.build.build() "
                           "(nvcc, sm_103a) first; there is no CPU fallback")
    lib = ctypes.CDLL(LIB_PATH)
    lib.sd_verify_attention.argtypes = [_vp, _vp, _vp, Strides, _vp, _i, _vp, _i, _i, _i, _i, _i, _i,
                                        _f, _vp, _sz, _vp]
    lib.sd_verify_attention.restype = _i
    lib.sd_verify_attention_workspace_size.argtypes = [_i] * 7
    lib.sd_verify_attention_workspace_size.restype = _sz
    lib.sd_draft_block_attention.argtypes = [_vp, _vp, _vp, Strides, _vp, _i, _vp, _vp, _vp,
                                             _i, _i, _i, _i, _i, _i, _f, _vp, _sz, _vp]
    lib.sd_draft_block_attention.restype = _i
    lib.sd_draft_block_attention_workspace_size.argtypes = [_i] * 7
    lib.sd_draft_block_attention_workspace_size.restype = _sz
    lib.sd_accept_greedy.argtypes = [_vp, _vp, _i, _i, _i, _i, _vp, _vp, _vp, _sz, _vp]
    lib.sd_accept_greedy.restype = _i
    lib.sd_verify_tree_attention.argtypes = [_vp, _vp, _vp, Strides, _vp, _i, _vp, _vp, _i, _i, _i, _i, _i, _i,
                                             ctypes.c_float, _vp, _sz, _vp]
    lib.sd_verify_tree_attention.restype = _i
    lib.sd_verify_tree_attention_workspace_size.argtypes = [_i] * 7
    lib.sd_verify_tree_attention_workspace_size.restype = _sz
    lib.sd_accept_tree_greedy.argtypes = [_vp, _vp, _vp, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _sz, _vp]
    lib.sd_accept_tree_greedy.restype = _i
    lib.sd_accept_tree_greedy_workspace_size.argtypes = [_i] * 4
    lib.sd_accept_tree_greedy_workspace_size.restype = _sz
    lib.sd_accept_greedy_workspace_size.argtypes = [_i] * 4
    lib.sd_accept_greedy_workspace_size.restype = _sz
    lib.sd_accept_sample.argtypes = [_vp, _vp, _vp, _i, _i, _i, _i, _f, ctypes.c_uint64,
                                     ctypes.c_uint32, _vp, _vp, _vp, _sz, _vp]
    lib.sd_accept_sample.restype = _i
    lib.sd_accept_sample_workspace_size.argtypes = [_i] * 4
    lib.sd_accept_sample_workspace_size.restype = _sz
    lib.sd_accept_greedy_noalloc.argtypes = [_vp, _vp, _i, _i, _i, _i, _vp, _vp, _vp]
    lib.sd_accept_greedy_noalloc.restype = _i
    lib.sd_philox4x32_10.argtypes = [_vp, ctypes.c_uint64, _vp, ctypes.c_int64, _vp]
    lib.sd_philox4x32_10.restype = _i
    lib.sd_status_string.argtypes = [_i]
    lib.sd_status_string.restype = ctypes.c_char_p
    lib.sd_last_error.argtypes = []
    lib.sd_last_error.restype = ctypes.c_char_p
    lib.sd_version.argtypes = []
    lib.sd_version.restype = _i
    lib.sd_fault_word.argtypes = [ctypes.POINTER(ctypes.c_uint32), _i]
    lib.sd_fault_word.restype = _i
    lib.sd_set_attention_path.argtypes = [_i]
    lib.sd_set_attention_path.restype = _i
    lib.sd_last_attention_path.argtypes = [ctypes.POINTER(_i)]
    lib.sd_last_attention_path.restype = _i
    lib.sd_last_attention_launches.argtypes = []
    lib.sd_last_attention_launches.restype = _i
    lib.sd_project_kv.argtypes = [_vp, ctypes.c_int64, _vp, _vp, _i, _i, _i, _vp, _vp, ctypes.c_int64, _i, _vp]
    lib.sd_project_kv.restype = _i
    lib.sd_commit_tokens.argtypes = [_vp, _i, _vp, _vp, _vp, _i, _i, _vp, _i, _vp, _vp, _vp, _i, _vp, _vp, _vp]
    lib.sd_commit_tokens.restype = _i
    lib.sd_compact_tree_kv.argtypes = [_vp, _vp, Strides, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp]
    lib.sd_compact_tree_kv.restype = _i
    lib.sd_store_to_host.argtypes = [_vp, _vp, ctypes.c_int64, _vp]
    lib.sd_store_to_host.restype = _i
    _i64 = ctypes.c_int64
    lib.sd_project_kv_commit.argtypes = [_vp, _i64, _i64, _vp, _vp, _i, _i, _vp, _vp, _vp, _i, _i, _vp, _vp,
                                         _i64, _i64, _i, _i, _vp]
    lib.sd_project_kv_commit.restype = _i
    lib.sd_latent_compress.argtypes = [_vp, _vp, _i64, _i64, _i, _i, _i, _i, _vp, _i64, _i64, _i, _vp, _sz, _vp]
    lib.sd_latent_compress.restype = _i
    lib.sd_latent_compress_workspace_size.argtypes = [_i] * 4
    lib.sd_latent_compress_workspace_size.restype = _sz
    lib.sd_set_projector_path.argtypes = [_i]
    lib.sd_set_projector_path.restype = _i
    lib.sd_set_wait_test.argtypes = [ctypes.c_uint32, ctypes.c_uint64]
    lib.sd_set_wait_test.restype = _i
    lib.sd_set_sample_path.argtypes = [_i]
    lib.sd_set_sample_path.restype = _i
    lib.sd_last_sample_path.argtypes = []
    lib.sd_last_sample_path.restype = _i
    lib.sd_last_projector_path.argtypes = []
    lib.sd_last_projector_path.restype = _i
    _lib = lib
    return lib


def _status_name(s: int) -> str:
    try:
        return load().sd_status_string(s).decode()
    except Exception:  # library not loadable: still name the code
        return f"status {s}"


def _check(status: int):
    if status != SD_OK:
        raise SdError(status, load().sd_last_error().decode())


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return SD_BF16
    if t.dtype == torch.float32:
        return SD_FP32
    raise TypeError(f"unsupported dtype {t.dtype} (bf16 or fp32)")


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _p(t):
    return None if t is None else t.data_ptr()


def _need_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("all tensors must be CUDA tensors (device memory)")


def _kv_strides(k: torch.Tensor) -> Strides:
    if k.stride(3) != 1:
        raise ValueError("the D axis of the cache must be contiguous")
    return Strides(k.stride(0), k.stride(1), k.stride(2))


# --------------------------------------------------------------------------
# workspace sizes
# --------------------------------------------------------------------------

def sd_verify_attention_workspace_size(B, T, Hq, Hkv, D, max_ctx, dtype=SD_BF16) -> int:
    return load().sd_verify_attention_workspace_size(B, T, Hq, Hkv, D, max_ctx, dtype)


def sd_draft_block_attention_workspace_size(B, T, Hq, Hkv, D, max_ctx, dtype=SD_BF16) -> int:
    return load().sd_draft_block_attention_workspace_size(B, T, Hq, Hkv, D, max_ctx, dtype)


def sd_accept_greedy_workspace_size(B, T, V, dtype=SD_BF16) -> int:
    return load().sd_accept_greedy_workspace_size(B, T, V, dtype)


def sd_accept_sample_workspace_size(B, T, V, dtype=SD_BF16) -> int:
    return load().sd_accept_sample_workspace_size(B, T, V, dtype)


def workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """Zero-filled device workspace (the acceptance calls need the first 256 bytes zero)."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)


# --------------------------------------------------------------------------
# entry points
# --------------------------------------------------------------------------

def sd_verify_attention(q, k_cache, v_cache, ctx_len, max_ctx, out, scale, ws, stream=None):
    """q [B,T,Hq,D]; k_cache/v_cache [B,S,Hkv,D]; ctx_len int32 [B]; out fp32 [B,T,Hq,D]."""
    _need_cuda(q, k_cache, v_cache, ctx_len, out, ws)
    B, T, Hq, D = q.shape
    Hkv = k_cache.shape[2]
    if not q.is_contiguous() or not out.is_contiguous() or out.dtype != torch.float32:
        raise ValueError("q and out must be contiguous; out fp32")
    if ctx_len.dtype != torch.int32 or k_cache.dtype != q.dtype or v_cache.dtype != q.dtype:
        raise ValueError("ctx_len int32; q, k_cache, v_cache of one dtype")
    if k_cache.stride() != v_cache.stride():
        raise ValueError("k_cache and v_cache must share strides")
    _check(load().sd_verify_attention(_p(q), _p(k_cache), _p(v_cache), _kv_strides(k_cache), _p(ctx_len),
                                      int(max_ctx), _p(out), B, T, Hq, Hkv, D, _dt(q), float(scale),
                                      _p(ws), ws.numel() * ws.element_size(), _stream(stream)))


def sd_draft_block_attention(q, k_ctx, v_ctx, n_ctx, max_ctx, k_blk, v_blk, out, scale, ws,
                             stream=None):
    """q [B,T,Hq,D]; k_ctx/v_ctx [B,S,Hkv,D]; n_ctx int32 [B]; k_blk/v_blk [B,T,Hkv,D]."""
    _need_cuda(q, k_ctx, v_ctx, n_ctx, k_blk, v_blk, out, ws)
    B, T, Hq, D = q.shape
    Hkv = k_ctx.shape[2]
    if not (q.is_contiguous() and out.is_contiguous() and k_blk.is_contiguous() and v_blk.is_contiguous()):
        raise ValueError("q, out, k_blk, v_blk must be contiguous")
    if out.dtype != torch.float32 or n_ctx.dtype != torch.int32:
        raise ValueError("out fp32, n_ctx int32")
    if k_ctx.stride() != v_ctx.stride():
        raise ValueError("k_ctx and v_ctx must share strides")
    _check(load().sd_draft_block_attention(_p(q), _p(k_ctx), _p(v_ctx), _kv_strides(k_ctx), _p(n_ctx),
                                           int(max_ctx), _p(k_blk), _p(v_blk), _p(out), B, T, Hq, Hkv,
                                           D, _dt(q), float(scale), _p(ws), ws.numel() * ws.element_size(),
                                           _stream(stream)))


def sd_verify_tree_attention_workspace_size(B, T, Hq, Hkv, D, max_ctx, dtype=SD_BF16) -> int:
    return load().sd_verify_tree_attention_workspace_size(B, T, Hq, Hkv, D, max_ctx, dtype)


def sd_accept_tree_greedy_workspace_size(B, T, V, dtype=SD_BF16) -> int:
    return load().sd_accept_tree_greedy_workspace_size(B, T, V, dtype)


def sd_verify_tree_attention(q, k_cache, v_cache, ctx_len, max_ctx, tree_mask, out, scale, ws, stream=None):
    """As sd_verify_attention, plus tree_mask int64 [B,T] (bit k of node j's 64-bit word: node j
    sees block slot k); T <= 64."""
    _need_cuda(q, k_cache, v_cache, ctx_len, tree_mask, out, ws)
    B, T, Hq, D = q.shape
    Hkv = k_cache.shape[2]
    if not q.is_contiguous() or not out.is_contiguous() or out.dtype != torch.float32:
        raise ValueError("q and out must be contiguous; out fp32")
    if ctx_len.dtype != torch.int32 or k_cache.dtype != q.dtype or v_cache.dtype != q.dtype:
        raise ValueError("ctx_len int32; q, k_cache, v_cache of one dtype")
    if tree_mask.dtype != torch.int64 or tree_mask.numel() != B * T or not tree_mask.is_contiguous():
        raise ValueError("tree_mask: contiguous int64 [B, T] (one 64-bit mask word per node)")
    if k_cache.stride() != v_cache.stride():
        raise ValueError("k_cache and v_cache must share strides")
    _check(load().sd_verify_tree_attention(_p(q), _p(k_cache), _p(v_cache), _kv_strides(k_cache), _p(ctx_len),
                                           int(max_ctx), _p(tree_mask), _p(out), B, T, Hq, Hkv, D, _dt(q),
                                           float(scale), _p(ws), ws.numel() * ws.element_size(), _stream(stream)))


def sd_accept_tree_greedy(tokens, parents, target_logits, n_accepted, correction_id, path, ws, stream=None):
    """tokens, parents int32 [B,T]; target_logits [B,T,V]; n_accepted, correction_id int32 [B];
    path int32 [B,T]."""
    _need_cuda(tokens, parents, target_logits, n_accepted, correction_id, path, ws)
    B, T, V = target_logits.shape
    for t in (tokens, parents, path):
        if t.dtype != torch.int32 or not t.is_contiguous() or t.numel() != B * T:
            raise ValueError("tokens, parents and path are contiguous int32 [B, T]")
    if not target_logits.is_contiguous():
        raise ValueError("logits must be contiguous")
    if n_accepted.dtype != torch.int32 or correction_id.dtype != torch.int32:
        raise ValueError("ids are int32")
    _check(load().sd_accept_tree_greedy(_p(tokens), _p(parents), _p(target_logits), B, T, V, _dt(target_logits),
                                        _p(n_accepted), _p(correction_id), _p(path), _p(ws),
                                        ws.numel() * ws.element_size(), _stream(stream)))


def sd_accept_greedy(draft_ids, target_logits, n_accepted, correction_id, ws, stream=None):
    """draft_ids int32 [B,T-1]; target_logits [B,T,V]; outputs int32 [B]."""
    _need_cuda(draft_ids, target_logits, n_accepted, correction_id, ws)
    B, T, V = target_logits.shape
    if not target_logits.is_contiguous() or not draft_ids.is_contiguous():
        raise ValueError("logits and draft ids must be contiguous")
    if draft_ids.dtype != torch.int32 or n_accepted.dtype != torch.int32 or correction_id.dtype != torch.int32:
        raise ValueError("ids are int32")
    _check(load().sd_accept_greedy(_p(draft_ids), _p(target_logits), B, T, V, _dt(target_logits),
                                   _p(n_accepted), _p(correction_id), _p(ws), ws.numel() * ws.element_size(),
                                   _stream(stream)))


def sd_accept_sample(draft_ids, draft_probs, target_logits, temperature, philox_seed, philox_offset,
                     n_accepted, next_id, ws, stream=None):
    """draft_ids int32 [B,T-1]; draft_probs fp32 [B,T,V]; target_logits [B,T,V]."""
    _need_cuda(draft_ids, draft_probs, target_logits, n_accepted, next_id, ws)
    B, T, V = target_logits.shape
    if not (target_logits.is_contiguous() and draft_ids.is_contiguous() and draft_probs.is_contiguous()):
        raise ValueError("inputs must be contiguous")
    if draft_probs.dtype != torch.float32 or draft_ids.dtype != torch.int32:
        raise ValueError("draft_probs fp32, draft_ids int32")
    _check(load().sd_accept_sample(_p(draft_ids), _p(draft_probs), _p(target_logits), B, T, V,
                                   _dt(target_logits), float(temperature), int(philox_seed),
                                   int(philox_offset), _p(n_accepted), _p(next_id), _p(ws),
                                   ws.numel() * ws.element_size(), _stream(stream)))


def sd_project_kv(hidden, w_k, w_v, k_out, v_out, stream=None):
    """hidden bf16 [N, Hd] (rows may be strided); w_k, w_v bf16 [Dout, Hd]
    contiguous; k_out, v_out bf16 [N, Dout] (rows may be strided, e.g. a slice
    of a [S, Hkv * D] cache view)."""
    _need_cuda(hidden, w_k, w_v, k_out, v_out)
    N, Hd = hidden.shape
    Dout = w_k.shape[0]
    if w_k.shape != (Dout, Hd) or w_v.shape != (Dout, Hd) or not (w_k.is_contiguous() and w_v.is_contiguous()):
        raise ValueError("w_k and w_v are contiguous [Dout, Hd]")
    if k_out.shape != (N, Dout) or v_out.shape != (N, Dout) or k_out.stride() != v_out.stride():
        raise ValueError("k_out and v_out are [N, Dout] with equal strides")
    if hidden.stride(1) != 1 or k_out.stride(1) != 1:
        raise ValueError("the last axis must be contiguous")
    dt = _dt(hidden)
    _check(load().sd_project_kv(_p(hidden), hidden.stride(0), _p(w_k), _p(w_v), N, Hd, Dout, _p(k_out), _p(v_out),
                                k_out.stride(0), dt, _stream(stream)))


def _i32_cuda(*ts):
    for t in ts:
        if t is not None and (t.dtype != torch.int32 or not t.is_contiguous()):
            raise ValueError("index tensors are contiguous int32")


def sd_commit_tokens(proposals, n_accepted, next_token, ctx_len, out_tokens, out_len, anchor, ctx_cap,
                     path=None, draft_ctx=None, status=None, stream=None):
    """proposals int32 [B, P] (chain drafts, or tree node tokens with path
    [B, T]); out_tokens int32 [B, out_cap]; the rest int32 [B], updated in
    place on the device."""
    _need_cuda(proposals, n_accepted, next_token, ctx_len, out_tokens, out_len, anchor, path, draft_ctx, status)
    _i32_cuda(proposals, n_accepted, next_token, ctx_len, out_tokens, out_len, anchor, path, draft_ctx, status)
    B, P = proposals.shape
    T = path.shape[1] if path is not None else P + 1
    _check(load().sd_commit_tokens(_p(proposals), P, _p(path), _p(n_accepted), _p(next_token), B, T,
                                   _p(ctx_len), int(ctx_cap), _p(draft_ctx), _p(out_tokens), _p(out_len),
                                   out_tokens.shape[1], _p(anchor), _p(status), _stream(stream)))


def sd_compact_tree_kv(k_cache, v_cache, ctx_len, path, n_accepted, stream=None):
    """k_cache, v_cache [B, S, Hkv, D] (D contiguous, equal strides); path int32 [B, T]."""
    _need_cuda(k_cache, v_cache, ctx_len, path, n_accepted)
    _i32_cuda(ctx_len, path, n_accepted)
    if k_cache.stride() != v_cache.stride() or k_cache.shape != v_cache.shape:
        raise ValueError("K and V caches must share shape and strides")
    B, S, Hkv, D = k_cache.shape
    T = path.shape[1]
    _check(load().sd_compact_tree_kv(_p(k_cache), _p(v_cache), _kv_strides(k_cache), _p(ctx_len), _p(path),
                                     _p(n_accepted), B, T, S, Hkv, D, _dt(k_cache), _stream(stream)))


def sd_store_to_host(host_dst, src, stream=None):
    """host_dst: a pinned CPU tensor; src: a CUDA tensor of the same byte size
    (both contiguous, a multiple of 16 bytes).  Enqueued on the stream; read
    host_dst after synchronising with it."""
    if host_dst.is_cuda or not host_dst.is_pinned():
        raise ValueError("host_dst must be a pinned CPU tensor")
    _need_cuda(src)
    if not (host_dst.is_contiguous() and src.is_contiguous()):
        raise ValueError("both tensors must be contiguous")
    nb = src.numel() * src.element_size()
    if host_dst.numel() * host_dst.element_size() != nb:
        raise ValueError("host_dst and src must hold the same number of bytes")
    _check(load().sd_store_to_host(_p(host_dst), _p(src), nb, _stream(stream)))


def sd_project_kv_commit(hidden_block, w_k, w_v, n_accepted, draft_ctx, k_ctx, v_ctx, path=None, stream=None):
    """hidden_block bf16 [B, T, Hd] (last axis contiguous); w_k, w_v bf16
    [Dout, Hd]; k_ctx, v_ctx bf16 [B, S, Dout] (last axis contiguous, equal
    strides); n_accepted, draft_ctx int32 [B]; path int32 [B, T] for a tree."""
    _need_cuda(hidden_block, w_k, w_v, n_accepted, draft_ctx, k_ctx, v_ctx, path)
    _i32_cuda(n_accepted, draft_ctx, path)
    B, T, Hd = hidden_block.shape
    Dout = w_k.shape[0]
    if w_k.shape != (Dout, Hd) or w_v.shape != (Dout, Hd) or not (w_k.is_contiguous() and w_v.is_contiguous()):
        raise ValueError("w_k and w_v are contiguous [Dout, Hd]")
    if k_ctx.shape != v_ctx.shape or k_ctx.stride() != v_ctx.stride() or k_ctx.shape[2] != Dout:
        raise ValueError("k_ctx and v_ctx are [B, S, Dout] with equal strides")
    if hidden_block.stride(2) != 1 or k_ctx.stride(2) != 1:
        raise ValueError("the last axis must be contiguous")
    _check(load().sd_project_kv_commit(_p(hidden_block), hidden_block.stride(1), hidden_block.stride(0), _p(w_k),
                                       _p(w_v), Hd, Dout, _p(n_accepted), _p(path), _p(draft_ctx), B, T,
                                       _p(k_ctx), _p(v_ctx), k_ctx.stride(0), k_ctx.stride(1), k_ctx.shape[1],
                                       _dt(hidden_block), _stream(stream)))


def sd_latent_compress_workspace_size(frames, N, Cq, d) -> int:
    return int(load().sd_latent_compress_workspace_size(frames, N, Cq, d))


def sd_latent_compress(queries, features, out, ws, stream=None):
    """queries bf16 [Cq, d] contiguous; features bf16 [F, N, d] (last axis
    contiguous); out bf16 [F, Cq, d] (last axis contiguous)."""
    _need_cuda(queries, features, out, ws)
    F, N, d = features.shape
    Cq = queries.shape[0]
    if queries.shape != (Cq, d) or not queries.is_contiguous():
        raise ValueError("queries are contiguous [Cq, d]")
    if out.shape != (F, Cq, d) or out.stride(2) != 1 or features.stride(2) != 1:
        raise ValueError("out is [F, Cq, d]; the last axes must be contiguous")
    _check(load().sd_latent_compress(_p(queries), _p(features), features.stride(1), features.stride(0), F, N, Cq, d,
                                     _p(out), out.stride(1), out.stride(0), _dt(features), _p(ws),
                                     ws.numel() * ws.element_size(), _stream(stream)))


def sd_set_projector_path(path: int) -> int:
    return load().sd_set_projector_path(int(path))


def sd_last_projector_path() -> int:
    return int(load().sd_last_projector_path())


def sd_set_wait_test(extra_arrivals: int, limit_ns: int = 0) -> None:
    _check(load().sd_set_wait_test(int(extra_arrivals), int(limit_ns)))


def sd_set_sample_path(path: int) -> int:
    return load().sd_set_sample_path(int(path))


def sd_last_sample_path() -> int:
    return int(load().sd_last_sample_path())


def sd_philox4x32_10(counters, key, out, stream=None):
    """counters uint32-as-int32 [n,4] device, out same shape."""
    _need_cuda(counters, out)
    n = counters.shape[0]
    _check(load().sd_philox4x32_10(_p(counters), int(key), _p(out), n, _stream(stream)))


def sd_fault_word(clear: bool = True) -> int:
    v = ctypes.c_uint32(0)
    _check(load().sd_fault_word(ctypes.byref(v), 1 if clear else 0))
    return v.value


def sd_set_attention_path(path: int) -> int:
    return load().sd_set_attention_path(int(path))


def sd_last_attention_launches() -> int:
    """Kernels the last attention call on this thread launched (1 or 2)."""
    return int(load().sd_last_attention_launches())


def sd_last_attention_path():
    n = ctypes.c_int(0)
    path = load().sd_last_attention_path(ctypes.byref(n))
    return path, n.value
