// C-ABI layer of libsdverify: argument validation on the host, workspace
// layout, kernel selection and launch.  Declarations and the passages each
// call follows are in include/sd_verify.h.
#include <cuda_runtime.h>

#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <atomic>

#include "internal.h"

// device fault word, set by kernel guards (never a trap)
__device__ unsigned int g_sd_fault_word;

namespace sdv {

namespace {

thread_local char g_err[512] = "";
thread_local int g_last_path = 0;
thread_local int g_last_splits = 0;
thread_local int g_last_launches = 0;
std::atomic<int> g_force_path{0};
std::atomic<int> g_force_proj_path{0};
thread_local int g_last_proj_path = 0;
std::atomic<int> g_force_sample_path{0};
std::atomic<unsigned int> g_wait_extra{0};
std::atomic<unsigned long long> g_wait_ns{kBarrierWaitNs};
thread_local int g_last_sample_path = 0;

constexpr size_t kHeader = 256;  // counters; zero between calls

sd_status fail(sd_status s, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return s;
}

sd_status cuda_fail(cudaError_t e, const char *what) {
    return fail(SD_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// device address of the fault word, looked up once per device (the lookup is
// idempotent, so threads that race on a first call store the same value)
unsigned int *fault_ptr() {
    static std::atomic<unsigned int *> ptrs[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    unsigned int *f = ptrs[dev].load(std::memory_order_acquire);
    if (!f) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_sd_fault_word) != cudaSuccess) return nullptr;
        f = static_cast<unsigned int *>(p);
        ptrs[dev].store(f, std::memory_order_release);
    }
    return f;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t esize(sd_dtype dt) { return dt == SD_BF16 ? 2 : 4; }

// ----------------------------------------------------------------------------
// attention planning
// ----------------------------------------------------------------------------
struct AttnPlan {
    int path;           // 1 CUDA-core, 2 tensor-core
    int n_splits, keys_per_split;
    int n_mblk, mblk_nodes;   // tensor-core row blocks per kv head and block rows in each
};

// row blocks of the tensor-core kernel: whole block rows, at most 128 query rows each
void row_blocks(int G, int T, int *n_mblk, int *mblk_nodes) {
    const int nodes = std::max(1, std::min(T, 128 / std::max(1, G)));
    *mblk_nodes = nodes;
    *n_mblk = (T + nodes - 1) / nodes;
}

// keys of the longest sequence's key space
int max_keys(int mode, int max_ctx, int T) { return mode == 1 ? max_ctx + T : max_ctx + T - 1; }

AttnPlan plan_attention(const AttnParams &p, int path) {
    const int sms = device_sm_count();
    const int N = max_keys(p.mode, p.max_ctx, p.T);
    AttnPlan pl;
    pl.path = path;
    pl.n_mblk = 1;
    pl.mblk_nodes = p.T;
    if (path >= 2) {
        // tensor cores: one CTA per work slot, at most one per SM when the units
        // fit (the kernel spreads the slots over the units by their sequences'
        // lengths, read on the device), else one per unit
        row_blocks(p.Hq / p.Hkv, p.T, &pl.n_mblk, &pl.mblk_nodes);
        const long units = (long)p.B * p.Hkv * pl.n_mblk;
        // tiles of the longest unit: its cache keys, plus the drafter's block tile
        const long cache_keys = p.mode == 1 ? p.max_ctx : (long)p.max_ctx + p.T - 1;
        const long max_tiles = (cache_keys + kTcTileKeys - 1) / kTcTileKeys + (p.mode == 1 ? 1 : 0);
        if (units > sms) {
            pl.n_splits = (int)units;
        } else if (p.B == 1) {
            // one sequence: every unit has max_tiles; the fewest splits per unit
            // that reach the smallest load of any split count fitting the SMs
            const long per = std::max(1L, std::min<long>(sms / units, max_tiles));
            const long load = (max_tiles + per - 1) / per;
            pl.n_splits = (int)(units * ((max_tiles + load - 1) / load));
        } else {
            // several sequences: the kernel spreads up to one CTA per SM over the
            // units by their lengths
            pl.n_splits = (int)std::min<long>(sms, units * max_tiles);
        }
        pl.keys_per_split = 0;
        return pl;
    }
    const int units = p.B * p.Hkv * pl.n_mblk;
    int ctas_per_sm, min_keys, gran;
    if (path >= 2) { ctas_per_sm = 1; min_keys = 2 * kTcTileKeys; gran = kTcTileKeys; }
    else { ctas_per_sm = 2; min_keys = 128; gran = 32; }
    const int target = std::max(1, sms * ctas_per_sm);
    // the tensor-core grid stays within one CTA per SM, so that the splits of
    // a (sequence, kv head) can merge inside the kernel
    int splits = path >= 2 ? std::max(1, target / units) : (target + units - 1) / units;
    splits = std::max(1, std::min(splits, (N + min_keys - 1) / min_keys));
    int kps = (N + splits - 1) / splits;
    kps = (kps + gran - 1) / gran * gran;
    pl.keys_per_split = kps;
    pl.n_splits = (N + kps - 1) / kps;
    return pl;
}

// attention workspace: [header][merge counters, B * Hkv * n_mblk][o_part][lse_part]
size_t attn_counters_bytes(int B, int Hkv, int n_mblk) {
    return align_up((size_t)B * Hkv * n_mblk * sizeof(unsigned int), 256);
}
// partial rows: CUDA-core kernel [n_splits][B*T*Hq] rows; tensor-core kernel one
// slot of 128 rows per CTA
size_t attn_partial_rows(int path, int B, int T, int Hq, int n_splits) {
    return path >= 2 ? (size_t)n_splits * 128 : (size_t)n_splits * B * T * Hq;
}
size_t attn_workspace(int path, int B, int T, int Hq, int Hkv, int D, int n_splits, int n_mblk) {
    const size_t rows = attn_partial_rows(path, B, T, Hq, n_splits);
    return kHeader + attn_counters_bytes(B, Hkv, n_mblk) + align_up(rows * D * sizeof(float), 256) +
           align_up(rows * sizeof(float), 256);
}

sd_status validate_attention(const AttnParams &p) {
    if (!p.q || !p.kc || !p.vc || !p.nctx || !p.out)
        return fail(SD_ERR_INVALID_ARG, "null tensor pointer");
    if (p.mode == 1 && (!p.kb || !p.vb)) return fail(SD_ERR_INVALID_ARG, "null block key/value pointer");
    if (p.mode == 2 && !p.tree_mask) return fail(SD_ERR_INVALID_ARG, "null tree mask");
    if (p.mode == 2 && (reinterpret_cast<uintptr_t>(p.tree_mask) & 7u))
        return fail(SD_ERR_INVALID_ARG, "tree mask must be 8-byte aligned");
    if (p.mode == 2) {
        if (p.B < 1 || p.T < 1 || p.T > kMaxTreeT) return fail(SD_ERR_INVALID_ARG, "need B >= 1 and T in [1, 64]");
    } else if (p.B < 1 || p.T < 1 || p.T > kMaxT) {
        return fail(SD_ERR_INVALID_ARG, "need B >= 1 and T in [1, 16]");
    }
    if (p.Hq < 1 || p.Hkv < 1 || p.Hq % p.Hkv) return fail(SD_ERR_INVALID_ARG, "Hq must be a multiple of Hkv");
    if (p.Hq > 4096) return fail(SD_ERR_UNSUPPORTED, "Hq must be <= 4096");
    if (p.D != 64 && p.D != 128) return fail(SD_ERR_UNSUPPORTED, "D must be 64 or 128");
    if (p.dt != SD_BF16 && p.dt != SD_FP32) return fail(SD_ERR_INVALID_ARG, "unknown dtype");
    if (p.max_ctx < 1) return fail(SD_ERR_INVALID_ARG, "max_ctx must be >= 1");
    if (!(p.scale == p.scale)) return fail(SD_ERR_INVALID_ARG, "scale is NaN");
    const size_t es = esize(p.dt);
    if (!aligned16(p.q) || !aligned16(p.kc) || !aligned16(p.vc) || !aligned16(p.out) ||
        (p.mode == 1 && (!aligned16(p.kb) || !aligned16(p.vb))))
        return fail(SD_ERR_INVALID_ARG, "tensor base addresses must be 16-byte aligned");
    if (p.kv.s < p.D || p.kv.h < p.D || p.kv.b < 1)
        return fail(SD_ERR_INVALID_ARG, "cache strides must not overlap the D axis");
    if (((size_t)p.kv.b * es) % 16 || ((size_t)p.kv.s * es) % 16 || ((size_t)p.kv.h * es) % 16)
        return fail(SD_ERR_INVALID_ARG, "cache strides must be multiples of 16 bytes");
    return SD_OK;
}

sd_status run_attention(AttnParams &p, void *ws, size_t ws_bytes, cudaStream_t st) {
    sd_status v = validate_attention(p);
    if (v != SD_OK) return v;
    if (!p.fault) return fail(SD_ERR_CUDA, "no CUDA device / fault word unavailable");
    const int force = g_force_path.load();
    int path;
    if (force == 1) path = 1;
    else if (attn_tc_supported(p)) path = 2;
    else if (force >= 2) return fail(SD_ERR_UNSUPPORTED, "tensor-core attention does not cover this shape");
    else path = 1;
    for (;;) {
        AttnPlan pl = plan_attention(p, path);
        const size_t need = attn_workspace(path, p.B, p.T, p.Hq, p.Hkv, p.D, pl.n_splits, pl.n_mblk);
        if (!ws || ws_bytes < need)
            return fail(SD_ERR_WORKSPACE, "attention workspace too small: need %zu bytes, got %zu", need, ws_bytes);
        if (!aligned16(ws)) return fail(SD_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
        const size_t rows = attn_partial_rows(path, p.B, p.T, p.Hq, pl.n_splits);
        p.merge_ctr = reinterpret_cast<unsigned int *>(static_cast<char *>(ws) + kHeader);
        char *w = static_cast<char *>(ws) + kHeader + attn_counters_bytes(p.B, p.Hkv, pl.n_mblk);
        p.o_part = reinterpret_cast<float *>(w);
        p.lse_part = reinterpret_cast<float *>(w + align_up(rows * p.D * sizeof(float), 256));
        p.n_splits = pl.n_splits;
        p.keys_per_split = pl.keys_per_split;
        p.n_mblk = pl.n_mblk;
        p.mblk_nodes = pl.mblk_nodes;
        // one sequence: a (splits, units) grid, every unit as long as the others
        p.plan_static = path == 2 && p.B == 1 && (long)p.Hkv * pl.n_mblk <= device_sm_count() ? 1 : 0;
        // tensor-core path: the splits of a unit merge inside the kernel (its grid
        // has at most one CTA per SM whenever a unit has several splits), and a
        // unit's only split writes the output itself; the CUDA-core path merges
        // in the merge kernel
        p.merge = path == 2 ? 1 : 0;
        p.wt = wait_test();
        cudaError_t e = path == 2 ? launch_attn_tc(p, st) : launch_attn_generic(p, st);
        if (e == cudaErrorCooperativeLaunchTooLarge && path == 2) {
            // the device cannot hold the whole grid at once (a partitioned one):
            // the CUDA-core kernel and the merge kernel, whose CTAs never wait
            (void)cudaGetLastError();
            if (force >= 2) return fail(SD_ERR_UNSUPPORTED, "the device cannot hold the tensor-core grid at once");
            path = 1;
            continue;
        }
        if (e != cudaSuccess) return cuda_fail(e, "attention split kernel launch");
        if (p.merge == 0) {
            e = launch_lse_merge(p, st);
            if (e != cudaSuccess) return cuda_fail(e, "attention merge kernel launch");
        }
        g_last_path = path;
        g_last_splits = pl.n_splits;
        g_last_launches = p.merge == 0 ? 2 : 1;
        return SD_OK;
    }
}

size_t attention_ws_size(int mode, int B, int T, int Hq, int Hkv, int D, int max_ctx, sd_dtype dt) {
    if (B < 1 || T < 1 || T > (mode == 2 ? kMaxTreeT : kMaxT) || Hq < 1 || Hkv < 1 || Hq % Hkv || Hq > 4096 ||
        max_ctx < 1 || (D != 64 && D != 128))
        return 0;
    AttnParams p = {};
    p.mode = mode; p.B = B; p.T = T; p.Hq = Hq; p.Hkv = Hkv; p.D = D; p.dt = dt; p.max_ctx = max_ctx;
    const AttnPlan p1 = plan_attention(p, 1), p2 = plan_attention(p, 2);
    return std::max(attn_workspace(1, B, T, Hq, Hkv, D, p1.n_splits, p1.n_mblk),
                    attn_workspace(2, B, T, Hq, Hkv, D, p2.n_splits, p2.n_mblk));
}

// ----------------------------------------------------------------------------
// acceptance planning
// ----------------------------------------------------------------------------
// chunk length of the acceptance pass-1 kernels: every row is cut into
// floor(per_sm * SMs / rows) chunks (at least one), so the grid fits in one
// wave of per_sm CTAs per SM (greedy streams its chunk: 3 per SM for 64 rows
// and more, 2 below, where larger chunks mean fewer partials and tickets; the
// sampled pass 1 holds its chunk in registers: 2 per SM)
int accept_chunk(int rows, int V, int cap, int per_sm) {
    const long slots = (long)per_sm * device_sm_count();
    const long per_row = std::max(1L, slots / std::max(1, rows));
    long chunk = (V + per_row - 1) / per_row;
    chunk = std::max(2048L, std::min(chunk, (long)cap));
    chunk = (chunk + 7) / 8 * 8;
    return (int)std::min<long>(chunk, (long)V);
}

// the greedy pass streams its chunk, so its chunks are sized only by the grid;
// the sampled pass 1 holds its chunk in registers: at most 8 vectors per thread
int greedy_cap(sd_dtype) { return 1 << 30; }
int greedy_per_sm(int rows) { return rows >= 64 ? 3 : 2; }
int sample_cap(sd_dtype dt) { return dt == SD_BF16 ? 8 * 8 * 256 : 8 * 4 * 256; }

// greedy workspace: [header: CTAs-finished counter][pval][pidx]
struct GreedyLayout {
    size_t pval, pidx, total;
};
GreedyLayout greedy_layout(int B, int T, int V, int chunk) {
    const size_t R = (size_t)B * T, parts = R * ((V + chunk - 1) / chunk);
    GreedyLayout l;
    l.pval = kHeader;
    l.pidx = l.pval + align_up(parts * 4, 256);
    l.total = l.pidx + align_up(parts * 4, 256);
    return l;
}

// chunk of the sampled rule's second pass (the deciding row of each sequence):
// the largest chunk the in-chunk search covers, so the chunk sums are few
int draw_chunk_for(int B, int V) {
    (void)B;
    return std::min(V, kDrawChunkMax);
}

// sample workspace: [header: counters][per-sequence counters]
// [pm][pz][row_stats][state][rs] for the two-kernel form, then [pp][fs] for
// the one-launch form (sized for a grid of kSampleFusedPerSm CTAs per SM)
struct SampleLayout {
    size_t row_ctr, pm, pz, row_stats, state, rs, pp, fs, total;
};
SampleLayout sample_layout(int B, int T, int V, int chunk, int draw_chunk) {
    const size_t R = (size_t)B * T, nc = (V + chunk - 1) / chunk, parts = R * nc;
    const size_t nd = (V + draw_chunk - 1) / draw_chunk;
    const size_t cmax = (size_t)kSampleFusedPerSm * device_sm_count();
    SampleLayout l;
    l.row_ctr = kHeader;
    l.pm = l.row_ctr + align_up((size_t)B * 8, 256);
    l.pz = l.pm + align_up(parts * 4, 256);
    l.row_stats = l.pz + align_up(parts * 8, 256);
    l.state = l.row_stats + align_up(R * 8, 256);
    l.rs = l.state + align_up((size_t)B * 16, 256);
    l.pp = l.rs + align_up((size_t)B * nd * 8, 256);
    l.fs = l.pp + align_up(cmax * 2 * 16, 256);
    l.total = l.fs + align_up(cmax * 16, 256);
    return l;
}

// The one-launch form of the sampled rule, where its grid fits on the device at
// once (kSampleFusedPerSm CTAs per SM): segments of the B*T*V logits, at least
// 2048 elements, a multiple of 8, no longer than a row, one per CTA; chunks of
// the deciding row, at least 2048 elements, as many per sequence as the grid
// holds, each within 4 vectors per thread.
struct FusedPlan {
    int grid, seg, n_segs, fchunk, n_fchunks;
};
bool plan_sample_fused(int B, int T, int V, sd_dtype dt, FusedPlan &f) {
    const long R = (long)B * T;
    const int sms = device_sm_count();
    const int C = kSampleFusedPerSm * sms;
    if (R > C || B > C) return false;
    const int nb = std::max(1, std::min(C / B, (V + 2047) / 2048));
    long fchunk = (V + nb - 1) / nb;
    fchunk = (fchunk + 7) / 8 * 8;
    f.fchunk = (int)std::min<long>(fchunk, V);
    f.n_fchunks = (V + f.fchunk - 1) / f.fchunk;
    const int nv = sample_vec_per_thread(dt, f.fchunk);
    if (nv > 4) return false;   // (1, 2, 4 vectors per thread cover the chunk; 8 is the cap)
    if (sample_fused_per_sm(dt, nv) < kSampleFusedPerSm) return false;
    const long n = R * V;
    long seg = (n + C - 1) / C;
    seg = std::max(2048L, (seg + 7) / 8 * 8);
    f.seg = (int)std::min<long>(seg, V);
    f.n_segs = (int)((n + f.seg - 1) / f.seg);
    f.grid = std::max(f.n_segs, B * f.n_fchunks);
    return f.grid <= C;
}

}  // namespace

WaitTest wait_test() {
    WaitTest w;
    w.extra = g_wait_extra.load();
    w.limit_ns = g_wait_ns.load();
    return w;
}

int device_sm_count() {
    static std::atomic<int> cache[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
    int n = cache[dev].load(std::memory_order_relaxed);
    if (!n) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) n = 148;
        cache[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

sd_status report_error(sd_status s, const char *msg) { return fail(s, "%s", msg); }

}  // namespace sdv

using namespace sdv;

extern "C" {

const char *sd_status_string(sd_status s) {
    switch (s) {
        case SD_OK: return "SD_OK";
        case SD_ERR_INVALID_ARG: return "SD_ERR_INVALID_ARG";
        case SD_ERR_UNSUPPORTED: return "SD_ERR_UNSUPPORTED";
        case SD_ERR_WORKSPACE: return "SD_ERR_WORKSPACE";
        case SD_ERR_CUDA: return "SD_ERR_CUDA";
    }
    return "SD_ERR_UNKNOWN";
}

const char *sd_last_error(void) { return g_err; }

int sd_version(void) { return 100; }

int sd_set_attention_path(int path) {
    if (path < 0 || path > 2) path = 0;
    return g_force_path.exchange(path);
}

int sd_last_attention_path(int *n_splits) {
    if (n_splits) *n_splits = g_last_splits;
    return g_last_path;
}

int sd_last_attention_launches(void) {
    return g_last_launches;
}

sd_status sd_fault_word(uint32_t *out, int clear) {
    if (!out) return fail(SD_ERR_INVALID_ARG, "null output pointer");
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
    unsigned int v = 0;
    e = cudaMemcpyFromSymbol(&v, g_sd_fault_word, sizeof v);
    if (e != cudaSuccess) return cuda_fail(e, "reading the fault word");
    *out = v;
    if (clear) {
        const unsigned int z = 0;
        e = cudaMemcpyToSymbol(g_sd_fault_word, &z, sizeof z);
        if (e != cudaSuccess) return cuda_fail(e, "clearing the fault word");
    }
    return SD_OK;
}

sd_status sd_verify_attention(const void *q, const void *k_cache, const void *v_cache, sd_strides kv,
                              const int32_t *ctx_len, int max_ctx, float *out, int B, int T, int Hq,
                              int Hkv, int D, sd_dtype dtype, float scale, void *workspace,
                              size_t workspace_bytes, void *stream) {
    AttnParams p = {};
    p.q = q; p.kc = k_cache; p.vc = v_cache; p.kv = kv; p.nctx = ctx_len; p.mode = 0;
    p.out = out; p.B = B; p.T = T; p.Hq = Hq; p.Hkv = Hkv; p.D = D; p.dt = dtype; p.scale = scale;
    p.max_ctx = max_ctx;
    p.fault = fault_ptr();
    return run_attention(p, workspace, workspace_bytes, static_cast<cudaStream_t>(stream));
}

size_t sd_verify_attention_workspace_size(int B, int T, int Hq, int Hkv, int D, int max_ctx, sd_dtype dtype) {
    return attention_ws_size(0, B, T, Hq, Hkv, D, max_ctx, dtype);
}

sd_status sd_draft_block_attention(const void *q, const void *k_ctx, const void *v_ctx, sd_strides ctx,
                                   const int32_t *n_ctx, int max_ctx, const void *k_blk, const void *v_blk,
                                   float *out, int B, int T, int Hq, int Hkv, int D, sd_dtype dtype,
                                   float scale, void *workspace, size_t workspace_bytes, void *stream) {
    AttnParams p = {};
    p.q = q; p.kc = k_ctx; p.vc = v_ctx; p.kv = ctx; p.nctx = n_ctx; p.mode = 1;
    p.kb = k_blk; p.vb = v_blk;
    p.out = out; p.B = B; p.T = T; p.Hq = Hq; p.Hkv = Hkv; p.D = D; p.dt = dtype; p.scale = scale;
    p.max_ctx = max_ctx;
    p.fault = fault_ptr();
    return run_attention(p, workspace, workspace_bytes, static_cast<cudaStream_t>(stream));
}

size_t sd_draft_block_attention_workspace_size(int B, int T, int Hq, int Hkv, int D, int max_ctx,
                                               sd_dtype dtype) {
    return attention_ws_size(1, B, T, Hq, Hkv, D, max_ctx, dtype);
}

sd_status sd_verify_tree_attention(const void *q, const void *k_cache, const void *v_cache, sd_strides kv,
                                   const int32_t *ctx_len, int max_ctx, const uint64_t *tree_mask, float *out,
                                   int B, int T, int Hq, int Hkv, int D, sd_dtype dtype, float scale,
                                   void *workspace, size_t workspace_bytes, void *stream) {
    AttnParams p = {};
    p.q = q; p.kc = k_cache; p.vc = v_cache; p.kv = kv; p.nctx = ctx_len; p.mode = 2;
    p.tree_mask = tree_mask;
    p.out = out; p.B = B; p.T = T; p.Hq = Hq; p.Hkv = Hkv; p.D = D; p.dt = dtype; p.scale = scale;
    p.max_ctx = max_ctx;
    p.fault = fault_ptr();
    return run_attention(p, workspace, workspace_bytes, static_cast<cudaStream_t>(stream));
}

size_t sd_verify_tree_attention_workspace_size(int B, int T, int Hq, int Hkv, int D, int max_ctx,
                                               sd_dtype dtype) {
    return attention_ws_size(2, B, T, Hq, Hkv, D, max_ctx, dtype);
}

size_t sd_accept_greedy_workspace_size(int B, int T, int V, sd_dtype dtype) {
    if (B < 1 || T < 1 || T > kMaxT || V < 1) return 0;
    return greedy_layout(B, T, V, accept_chunk(B * T, V, greedy_cap(dtype), greedy_per_sm(B * T))).total;
}

sd_status sd_accept_greedy(const int32_t *draft_ids, const void *target_logits, int B, int T, int V,
                           sd_dtype dtype, int32_t *n_accepted, int32_t *correction_id, void *workspace,
                           size_t workspace_bytes, void *stream) {
    if (B < 1 || T < 1 || T > kMaxT || V < 1) return fail(SD_ERR_INVALID_ARG, "need B >= 1, T in [1, 16], V >= 1");
    if (!target_logits || !n_accepted || !correction_id || (T > 1 && !draft_ids))
        return fail(SD_ERR_INVALID_ARG, "null tensor pointer");
    if (dtype != SD_BF16 && dtype != SD_FP32) return fail(SD_ERR_INVALID_ARG, "unknown dtype");
    if ((reinterpret_cast<uintptr_t>(target_logits) % esize(dtype)) != 0)
        return fail(SD_ERR_INVALID_ARG, "logits pointer not aligned to its element size");
    GreedyParams p = {};
    p.draft = draft_ids; p.logits = target_logits; p.B = B; p.T = T; p.V = V; p.dt = dtype;
    p.n_acc = n_accepted; p.corr = correction_id;
    p.chunk = accept_chunk(B * T, V, greedy_cap(dtype), greedy_per_sm(B * T));
    p.n_chunks = (V + p.chunk - 1) / p.chunk;
    const GreedyLayout gl = greedy_layout(B, T, V, p.chunk);
    if (!workspace || workspace_bytes < gl.total)
        return fail(SD_ERR_WORKSPACE, "greedy workspace too small: need %zu bytes, got %zu", gl.total, workspace_bytes);
    if (!aligned16(workspace)) return fail(SD_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
    char *w = static_cast<char *>(workspace);
    p.counter = reinterpret_cast<unsigned int *>(w);
    p.pval = reinterpret_cast<float *>(w + gl.pval);
    p.pidx = reinterpret_cast<int *>(w + gl.pidx);
    p.fault = fault_ptr();
    if (!p.fault) return fail(SD_ERR_CUDA, "no CUDA device / fault word unavailable");
    cudaError_t e = launch_accept_greedy(p, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "greedy accept launch");
    return SD_OK;
}

size_t sd_accept_tree_greedy_workspace_size(int B, int T, int V, sd_dtype dtype) {
    if (B < 1 || T < 1 || T > kMaxTreeT || V < 1) return 0;
    return greedy_layout(B, T, V, accept_chunk(B * T, V, greedy_cap(dtype), greedy_per_sm(B * T))).total;
}

sd_status sd_accept_tree_greedy(const int32_t *tokens, const int32_t *parents, const void *target_logits, int B,
                                int T, int V, sd_dtype dtype, int32_t *n_accepted, int32_t *correction_id,
                                int32_t *path, void *workspace, size_t workspace_bytes, void *stream) {
    if (B < 1 || T < 1 || T > kMaxTreeT || V < 1)
        return fail(SD_ERR_INVALID_ARG, "need B >= 1, T in [1, 64], V >= 1");
    if (!target_logits || !n_accepted || !correction_id || !tokens || !parents || !path)
        return fail(SD_ERR_INVALID_ARG, "null tensor pointer");
    if (dtype != SD_BF16 && dtype != SD_FP32) return fail(SD_ERR_INVALID_ARG, "unknown dtype");
    if ((reinterpret_cast<uintptr_t>(target_logits) % esize(dtype)) != 0)
        return fail(SD_ERR_INVALID_ARG, "logits pointer not aligned to its element size");
    GreedyParams p = {};
    p.draft = tokens; p.parents = parents; p.path = path;
    p.logits = target_logits; p.B = B; p.T = T; p.V = V; p.dt = dtype;
    p.n_acc = n_accepted; p.corr = correction_id;
    p.chunk = accept_chunk(B * T, V, greedy_cap(dtype), greedy_per_sm(B * T));
    p.n_chunks = (V + p.chunk - 1) / p.chunk;
    const GreedyLayout gl = greedy_layout(B, T, V, p.chunk);
    if (!workspace || workspace_bytes < gl.total)
        return fail(SD_ERR_WORKSPACE, "tree greedy workspace too small: need %zu bytes, got %zu", gl.total,
                    workspace_bytes);
    if (!aligned16(workspace)) return fail(SD_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
    char *w = static_cast<char *>(workspace);
    p.counter = reinterpret_cast<unsigned int *>(w);
    p.pval = reinterpret_cast<float *>(w + gl.pval);
    p.pidx = reinterpret_cast<int *>(w + gl.pidx);
    p.fault = fault_ptr();
    if (!p.fault) return fail(SD_ERR_CUDA, "no CUDA device / fault word unavailable");
    cudaError_t e = launch_accept_greedy(p, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "tree greedy accept launch");
    return SD_OK;
}

size_t sd_accept_sample_workspace_size(int B, int T, int V, sd_dtype dtype) {
    (void)dtype;
    if (B < 1 || T < 1 || T > kMaxT || V < 1) return 0;
    return sample_layout(B, T, V, accept_chunk(B * T, V, sample_cap(dtype), 2), draw_chunk_for(B, V)).total;
}

sd_status sd_accept_sample(const int32_t *draft_ids, const float *draft_probs, const void *target_logits,
                           int B, int T, int V, sd_dtype dtype, float temperature, uint64_t philox_seed,
                           uint32_t philox_offset, int32_t *n_accepted, int32_t *next_id, void *workspace,
                           size_t workspace_bytes, void *stream) {
    if (B < 1 || T < 1 || T > kMaxT || V < 1) return fail(SD_ERR_INVALID_ARG, "need B >= 1, T in [1, 16], V >= 1");
    if (!target_logits || !draft_probs || !n_accepted || !next_id || (T > 1 && !draft_ids))
        return fail(SD_ERR_INVALID_ARG, "null tensor pointer");
    if (dtype != SD_BF16 && dtype != SD_FP32) return fail(SD_ERR_INVALID_ARG, "unknown dtype");
    if (!(temperature > 0.f) || temperature == INFINITY)
        return fail(SD_ERR_INVALID_ARG, "temperature must be finite and > 0 (use sd_accept_greedy for 0)");
    if ((reinterpret_cast<uintptr_t>(target_logits) % esize(dtype)) != 0 ||
        (reinterpret_cast<uintptr_t>(draft_probs) % 4) != 0)
        return fail(SD_ERR_INVALID_ARG, "tensor pointer not aligned to its element size");
    SampleParams p = {};
    p.draft = draft_ids; p.q = draft_probs; p.logits = target_logits; p.B = B; p.T = T; p.V = V;
    p.dt = dtype; p.inv_tau = 1.0f / temperature; p.seed = philox_seed; p.offset = philox_offset;
    p.n_acc = n_accepted; p.next_id = next_id;
    p.chunk = accept_chunk(B * T, V, sample_cap(dtype), 2);
    p.n_chunks = (V + p.chunk - 1) / p.chunk;
    p.draw_chunk = draw_chunk_for(B, V);
    p.n_draw_chunks = (V + p.draw_chunk - 1) / p.draw_chunk;
    const SampleLayout sl = sample_layout(B, T, V, p.chunk, p.draw_chunk);
    if (!workspace || workspace_bytes < sl.total)
        return fail(SD_ERR_WORKSPACE, "sample workspace too small: need %zu bytes, got %zu", sl.total, workspace_bytes);
    if (!aligned16(workspace)) return fail(SD_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
    char *w = static_cast<char *>(workspace);
    p.counters = reinterpret_cast<unsigned int *>(w);
    p.row_counter = reinterpret_cast<unsigned int *>(w + sl.row_ctr);
    p.pm = reinterpret_cast<float *>(w + sl.pm);
    p.pz = reinterpret_cast<float2 *>(w + sl.pz);
    p.row_stats = reinterpret_cast<float2 *>(w + sl.row_stats);
    p.state = reinterpret_cast<float4 *>(w + sl.state);
    p.rs = reinterpret_cast<float2 *>(w + sl.rs);
    p.pp = reinterpret_cast<float4 *>(w + sl.pp);
    p.fs = reinterpret_cast<float4 *>(w + sl.fs);
    p.fault = fault_ptr();
    if (!p.fault) return fail(SD_ERR_CUDA, "no CUDA device / fault word unavailable");
    p.wt = wait_test();
    const int force = g_force_sample_path.load();
    FusedPlan fp = {};
    const bool fused = force != 1 && aligned16(target_logits) && plan_sample_fused(B, T, V, dtype, fp);
    if (force == 2 && !fused) return fail(SD_ERR_UNSUPPORTED, "the one-launch sampled rule does not fit this call");
    cudaError_t e;
    if (fused) {
        p.seg = fp.seg; p.n_segs = fp.n_segs; p.fchunk = fp.fchunk; p.n_fchunks = fp.n_fchunks;
        e = launch_accept_sample_fused(p, fp.grid, static_cast<cudaStream_t>(stream));
        if (e == cudaSuccess) {
            g_last_sample_path = 2;
            return SD_OK;
        }
        if (e != cudaErrorCooperativeLaunchTooLarge || force == 2) return cuda_fail(e, "sampled accept launch");
        (void)cudaGetLastError();   // the device is shared more than planned: two kernels instead
    }
    e = launch_accept_sample(p, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "sampled accept launch");
    g_last_sample_path = 1;
    return SD_OK;
}

sd_status sd_set_wait_test(uint32_t extra_arrivals, uint64_t limit_ns) {
    if (extra_arrivals > 1024) return fail(SD_ERR_INVALID_ARG, "extra_arrivals must be <= 1024");
    g_wait_ns.store(limit_ns == 0 || limit_ns > kBarrierWaitNs ? kBarrierWaitNs : (unsigned long long)limit_ns);
    g_wait_extra.store(extra_arrivals);
    return SD_OK;
}

int sd_set_sample_path(int path) {
    if (path < 0 || path > 2) path = 0;
    return g_force_sample_path.exchange(path);
}

int sd_last_sample_path(void) { return g_last_sample_path; }

sd_status sd_project_kv(const void *hidden, int64_t ld_hidden, const void *w_k, const void *w_v, int N, int Hd,
                        int Dout, void *k_out, void *v_out, int64_t ld_out, sd_dtype dtype, void *stream) {
    g_last_proj_path = 0;
    if (dtype == SD_FP32) return fail(SD_ERR_UNSUPPORTED, "the projector takes bf16 tensors only");
    if (dtype != SD_BF16) return fail(SD_ERR_INVALID_ARG, "unknown dtype");
    if (N < 0 || N > (1 << 21)) return fail(SD_ERR_INVALID_ARG, "need 0 <= N <= 2^21");
    if (Hd < 8 || Hd % 8 != 0 || Hd > (1 << 20)) return fail(SD_ERR_INVALID_ARG, "need Hd a positive multiple of 8");
    if (Dout < 32 || Dout % 32 != 0 || Dout > (1 << 20))
        return fail(SD_ERR_INVALID_ARG, "need Dout a positive multiple of 32");
    if (ld_hidden < Hd || ld_hidden % 8 != 0 || ld_out < Dout || ld_out % 8 != 0)
        return fail(SD_ERR_INVALID_ARG, "row strides must cover a row and be multiples of 8 elements");
    if (N == 0) return SD_OK;
    if (!hidden || !w_k || !w_v || !k_out || !v_out) return fail(SD_ERR_INVALID_ARG, "null tensor pointer");
    if (!aligned16(hidden) || !aligned16(w_k) || !aligned16(w_v) || !aligned16(k_out) || !aligned16(v_out))
        return fail(SD_ERR_INVALID_ARG, "tensor base addresses must be 16-byte aligned");
    ProjParams p = {};
    p.h = static_cast<const __nv_bfloat16 *>(hidden);
    p.wk = static_cast<const __nv_bfloat16 *>(w_k);
    p.wv = static_cast<const __nv_bfloat16 *>(w_v);
    p.k_out = static_cast<__nv_bfloat16 *>(k_out);
    p.v_out = static_cast<__nv_bfloat16 *>(v_out);
    p.ld_h = (long)ld_hidden; p.ld_out = (long)ld_out;
    p.N = N; p.Hd = Hd; p.Dout = Dout;
    p.fault = fault_ptr();
    if (!p.fault) return fail(SD_ERR_CUDA, "no CUDA device / fault word unavailable");
    const int force = g_force_proj_path.load();
    const bool small_ok = project_small_supported(8, Hd);   // 16 rows per CTA where they fit, else 8
    int path = N <= kProjSmallRows && small_ok ? 1 : 2;
    if (force == 1) path = 1;
    if (force == 2) path = 2;
    if (path == 2 && !project_tc_supported()) {
        if (force == 2) return fail(SD_ERR_UNSUPPORTED, "tensor-core projector needs sm_103 and 200 KB shared memory");
        path = 1;
    }
    if (path == 1 && !small_ok)
        return fail(SD_ERR_UNSUPPORTED, "CUDA-core projector stages 8 rows of Hd in 200 KB: Hd too large");
    cudaError_t e = launch_project(p, path, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "projector launch");
    g_last_proj_path = path;
    return SD_OK;
}

sd_status sd_project_kv_commit(const void *hidden_block, int64_t ld_hidden, int64_t hidden_bstride, const void *w_k,
                               const void *w_v, int Hd, int Dout, const int32_t *n_accepted, const int32_t *path,
                               const int32_t *draft_ctx, int B, int T, void *k_ctx, void *v_ctx,
                               int64_t ctx_bstride, int64_t ld_out, int max_rows, sd_dtype dtype, void *stream) {
    if (dtype == SD_FP32) return fail(SD_ERR_UNSUPPORTED, "the projector takes bf16 tensors only");
    if (dtype != SD_BF16) return fail(SD_ERR_INVALID_ARG, "unknown dtype");
    if (B < 1 || T < 1 || T > kMaxTreeT) return fail(SD_ERR_INVALID_ARG, "need B >= 1 and T in [1, 64]");
    if (Hd < 8 || Hd % 8 != 0 || Hd > (1 << 20)) return fail(SD_ERR_INVALID_ARG, "need Hd a positive multiple of 8");
    if (Dout < 32 || Dout % 32 != 0 || Dout > (1 << 20))
        return fail(SD_ERR_INVALID_ARG, "need Dout a positive multiple of 32");
    if (ld_hidden < Hd || ld_hidden % 8 != 0 || hidden_bstride < (int64_t)T * ld_hidden || hidden_bstride % 8 != 0)
        return fail(SD_ERR_INVALID_ARG, "hidden strides must cover a block and be multiples of 8 elements");
    if (max_rows < 1 || ld_out < Dout || ctx_bstride < (int64_t)max_rows * ld_out)
        return fail(SD_ERR_INVALID_ARG, "output strides must cover max_rows rows of Dout elements");
    if (!hidden_block || !w_k || !w_v || !k_ctx || !v_ctx || !n_accepted || !draft_ctx)
        return fail(SD_ERR_INVALID_ARG, "null tensor pointer");
    if (!aligned16(hidden_block) || !aligned16(w_k) || !aligned16(w_v))
        return fail(SD_ERR_INVALID_ARG, "hidden states and weights must be 16-byte aligned");
    if (!project_small_supported(kMaxT, Hd))
        return fail(SD_ERR_UNSUPPORTED, "the append stages 16 rows of Hd in 200 KB of shared memory: Hd <= 6400");
    if ((reinterpret_cast<uintptr_t>(k_ctx) | reinterpret_cast<uintptr_t>(v_ctx)) % 2 != 0)
        return fail(SD_ERR_INVALID_ARG, "outputs must be 2-byte aligned");
    ProjParams p = {};
    p.h = static_cast<const __nv_bfloat16 *>(hidden_block);
    p.wk = static_cast<const __nv_bfloat16 *>(w_k);
    p.wv = static_cast<const __nv_bfloat16 *>(w_v);
    p.k_out = static_cast<__nv_bfloat16 *>(k_ctx);
    p.v_out = static_cast<__nv_bfloat16 *>(v_ctx);
    p.ld_h = (long)ld_hidden; p.ld_out = (long)ld_out;
    p.h_bstride = (long)hidden_bstride; p.out_bstride = (long)ctx_bstride;
    p.N = T; p.Hd = Hd; p.Dout = Dout;
    p.n_acc = n_accepted; p.path = path; p.dst_row0 = draft_ctx;
    p.B = B; p.T = T; p.max_rows = max_rows;
    p.fault = fault_ptr();
    if (!p.fault) return fail(SD_ERR_CUDA, "no CUDA device / fault word unavailable");
    cudaError_t e = launch_project_commit(p, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "projector append launch");
    return SD_OK;
}

sd_status sd_commit_tokens(const int32_t *proposals, int proposal_stride, const int32_t *path,
                           const int32_t *n_accepted, const int32_t *next_token, int B, int T, int32_t *ctx_len,
                           int ctx_cap, int32_t *draft_ctx, int32_t *out_tokens, int32_t *out_len, int out_cap,
                           int32_t *anchor, int32_t *status, void *stream) {
    if (B < 1 || T < 1 || T > kMaxTreeT) return fail(SD_ERR_INVALID_ARG, "need B >= 1 and T in [1, 64]");
    if (proposal_stride < (path ? T : T - 1)) return fail(SD_ERR_INVALID_ARG, "proposal_stride too small");
    if (ctx_cap < 1 || out_cap < 1) return fail(SD_ERR_INVALID_ARG, "need ctx_cap >= 1 and out_cap >= 1");
    if ((T > 1 && !proposals) || !n_accepted || !next_token || !ctx_len || !out_tokens || !out_len || !anchor)
        return fail(SD_ERR_INVALID_ARG, "null tensor pointer");
    CommitParams p = {};
    p.prop = proposals; p.ps = proposal_stride; p.path = path;
    p.n_acc = n_accepted; p.next_tok = next_token; p.B = B; p.T = T;
    p.ctx_len = ctx_len; p.ctx_cap = ctx_cap; p.draft_ctx = draft_ctx;
    p.out_tokens = out_tokens; p.out_len = out_len; p.out_cap = out_cap;
    p.anchor = anchor; p.status = status;
    p.fault = fault_ptr();
    if (!p.fault) return fail(SD_ERR_CUDA, "no CUDA device / fault word unavailable");
    cudaError_t e = launch_commit_tokens(p, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "commit launch");
    return SD_OK;
}

sd_status sd_compact_tree_kv(void *k_cache, void *v_cache, sd_strides kv, const int32_t *ctx_len,
                             const int32_t *path, const int32_t *n_accepted, int B, int T, int max_slots, int Hkv,
                             int D, sd_dtype dtype, void *stream) {
    if (B < 1 || T < 1 || T > kMaxTreeT || Hkv < 1 || D < 1 || max_slots < T)
        return fail(SD_ERR_INVALID_ARG, "need B, Hkv, D >= 1, T in [1, 64] and max_slots >= T");
    if (dtype != SD_BF16 && dtype != SD_FP32) return fail(SD_ERR_INVALID_ARG, "unknown dtype");
    const int es = (int)esize(dtype);
    if ((D * es) % 16 != 0 || D * es > kMaxHeadBytes)
        return fail(SD_ERR_UNSUPPORTED, "a (position, head) row must be a multiple of 16 bytes, at most 512");
    if (kv.s < (int64_t)Hkv * D && kv.h < (int64_t)D)
        return fail(SD_ERR_INVALID_ARG, "cache strides overlap");
    if ((kv.b * es) % 16 != 0 || (kv.s * es) % 16 != 0 || (kv.h * es) % 16 != 0)
        return fail(SD_ERR_INVALID_ARG, "cache strides must be multiples of 16 bytes");
    if (!k_cache || !v_cache || !ctx_len || !path || !n_accepted) return fail(SD_ERR_INVALID_ARG, "null tensor pointer");
    if (!aligned16(k_cache) || !aligned16(v_cache)) return fail(SD_ERR_INVALID_ARG, "caches must be 16-byte aligned");
    CompactParams p = {};
    p.kc = k_cache; p.vc = v_cache; p.kv = kv; p.es = es;
    p.ctx_len = ctx_len; p.path = path; p.n_acc = n_accepted;
    p.B = B; p.T = T; p.S = max_slots; p.Hkv = Hkv; p.D = D;
    p.fault = fault_ptr();
    if (!p.fault) return fail(SD_ERR_CUDA, "no CUDA device / fault word unavailable");
    cudaError_t e = launch_compact_tree_kv(p, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "tree compaction launch");
    return SD_OK;
}

sd_status sd_store_to_host(void *host_dst, const void *src, int64_t bytes, void *stream) {
    if (bytes < 0) return fail(SD_ERR_INVALID_ARG, "bytes must be >= 0");
    if (bytes == 0) return SD_OK;
    if (!host_dst || !src) return fail(SD_ERR_INVALID_ARG, "null pointer");
    if (bytes % 16 != 0 || !aligned16(host_dst) || !aligned16(src))
        return fail(SD_ERR_INVALID_ARG, "bytes and both addresses must be multiples of 16");
    cudaPointerAttributes ad = {}, as = {};
    if (cudaPointerGetAttributes(&ad, host_dst) != cudaSuccess || ad.type != cudaMemoryTypeHost ||
        !ad.devicePointer) {
        (void)cudaGetLastError();
        return fail(SD_ERR_INVALID_ARG, "host_dst must be pinned host memory (cudaHostAlloc / cudaHostRegister)");
    }
    if (cudaPointerGetAttributes(&as, src) != cudaSuccess ||
        (as.type != cudaMemoryTypeDevice && as.type != cudaMemoryTypeManaged)) {
        (void)cudaGetLastError();
        return fail(SD_ERR_INVALID_ARG, "src must be device memory");
    }
    HostStoreParams p = {};
    p.src = static_cast<const uint4 *>(src);
    p.dst = static_cast<uint4 *>(ad.devicePointer);
    p.n16 = bytes / 16;
    cudaError_t e = launch_store_to_host(p, device_sm_count(), static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "host store launch");
    return SD_OK;
}

namespace {
struct LatentLayout {
    int n_splits, ksteps;
    size_t scores, probs, total;
};
// slices of d for the scores kernel: enough CTAs for every SM, at least 2
// stages of kLatentStageD per slice
LatentLayout latent_layout(int frames, int N, int Cq, int d) {
    LatentLayout l;
    const long ctas = (long)frames * ((N + 127) / 128);
    const int steps = (d + kLatentStageD - 1) / kLatentStageD;
    int splits = (int)std::min<long>((device_sm_count() + ctas - 1) / ctas, std::max(1, steps / 2));
    splits = std::max(1, std::min(splits, 16));
    l.ksteps = (steps + splits - 1) / splits;
    l.n_splits = (steps + l.ksteps - 1) / l.ksteps;
    const size_t ld_s = (size_t)((N + 127) / 128) * 128;
    const size_t ld_p = align_up((size_t)N, 8);
    l.scores = 0;
    l.probs = align_up((size_t)l.n_splits * frames * kLatentMaxQueries * ld_s * sizeof(float), 256);
    l.total = l.probs + align_up((size_t)frames * Cq * ld_p * 2, 256);
    return l;
}
bool latent_shape_ok(int frames, int N, int Cq, int d) {
    return frames >= 1 && frames <= 65535 && N >= 1 && N <= (1 << 20) && Cq >= 1 && Cq <= kLatentMaxQueries &&
           d >= 64 && d % 64 == 0 && d <= (1 << 16);
}
}  // namespace

size_t sd_latent_compress_workspace_size(int frames, int N, int Cq, int d) {
    if (!latent_shape_ok(frames, N, Cq, d)) return 0;
    return latent_layout(frames, N, Cq, d).total;
}

sd_status sd_latent_compress(const void *queries, const void *features, int64_t ld_features, int64_t frame_stride,
                             int frames, int N, int Cq, int d, void *out, int64_t ld_out, int64_t out_frame_stride,
                             sd_dtype dtype, void *workspace, size_t workspace_bytes, void *stream) {
    if (dtype == SD_FP32) return fail(SD_ERR_UNSUPPORTED, "the latent compressor takes bf16 tensors only");
    if (dtype != SD_BF16) return fail(SD_ERR_INVALID_ARG, "unknown dtype");
    if (!latent_shape_ok(frames, N, Cq, d))
        return fail(SD_ERR_INVALID_ARG, "need frames in [1, 65535], N >= 1, Cq in [1, 64], d a multiple of 64");
    if (ld_features < d || ld_features % 8 != 0 || frame_stride < (int64_t)N * ld_features || frame_stride % 8 != 0)
        return fail(SD_ERR_INVALID_ARG, "feature strides must cover a frame and be multiples of 8 elements");
    if (ld_out < d || ld_out % 8 != 0 || out_frame_stride < (int64_t)Cq * ld_out || out_frame_stride % 8 != 0)
        return fail(SD_ERR_INVALID_ARG, "output strides must cover a frame and be multiples of 8 elements");
    if (!queries || !features || !out) return fail(SD_ERR_INVALID_ARG, "null tensor pointer");
    if (!aligned16(queries) || !aligned16(features) || !aligned16(out))
        return fail(SD_ERR_INVALID_ARG, "tensor base addresses must be 16-byte aligned");
    const LatentLayout ll = latent_layout(frames, N, Cq, d);
    if (!workspace || workspace_bytes < ll.total)
        return fail(SD_ERR_WORKSPACE, "latent workspace too small: need %zu bytes, got %zu", ll.total, workspace_bytes);
    if (!aligned16(workspace)) return fail(SD_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
    if (!latent_supported()) return fail(SD_ERR_UNSUPPORTED, "the latent compressor needs sm_103 and 200 KB shared memory");
    char *w = static_cast<char *>(workspace);
    LatentParams p = {};
    p.q = static_cast<const __nv_bfloat16 *>(queries);
    p.f = static_cast<const __nv_bfloat16 *>(features);
    p.ld_f = (long)ld_features; p.f_fstride = (long)frame_stride;
    p.out = static_cast<__nv_bfloat16 *>(out);
    p.ld_out = (long)ld_out; p.out_fstride = (long)out_frame_stride;
    p.frames = frames; p.N = N; p.Cq = Cq; p.d = d;
    p.n_tiles = (N + 127) / 128;
    p.n_splits = ll.n_splits;
    p.ksteps_per_split = ll.ksteps;
    p.scores = reinterpret_cast<float *>(w + ll.scores);
    p.ld_s = (long)p.n_tiles * 128;
    p.probs = reinterpret_cast<__nv_bfloat16 *>(w + ll.probs);
    p.ld_p = (long)align_up((size_t)N, 8);
    p.fault = fault_ptr();
    if (!p.fault) return fail(SD_ERR_CUDA, "no CUDA device / fault word unavailable");
    cudaError_t e = launch_latent(p, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "latent compressor launch");
    return SD_OK;
}

int sd_set_projector_path(int path) {
    if (path < 0 || path > 2) path = 0;
    return g_force_proj_path.exchange(path);
}

int sd_last_projector_path(void) { return g_last_proj_path; }

sd_status sd_philox4x32_10(const uint32_t *counters, uint64_t key, uint32_t *out, int64_t n, void *stream) {
    if (n < 0) return fail(SD_ERR_INVALID_ARG, "n must be >= 0");
    if (n == 0) return SD_OK;
    if (!counters || !out) return fail(SD_ERR_INVALID_ARG, "null tensor pointer");
    if (!aligned16(counters) || !aligned16(out)) return fail(SD_ERR_INVALID_ARG, "buffers must be 16-byte aligned");
    if (n > (int64_t)1 << 40) return fail(SD_ERR_INVALID_ARG, "n too large");
    cudaError_t e = launch_philox(counters, key, out, n, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "philox launch");
    return SD_OK;
}

}  // extern "C"
