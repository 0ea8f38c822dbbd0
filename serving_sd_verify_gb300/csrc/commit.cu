// Commit of a verified block, on the device, so a whole speculative cycle
// (draft, verify, accept, append, commit) runs back to back with no host
// round trip.
//
// Source: "VFlash-FM" project page, "How VFlash-FM works", the worked cycle:
// the accepted prefix and the target's own token at the first disagreement
// are committed, the rest of the block is dropped, and the next cycle starts
// from that token as its anchor.  With the cache laid out as [context |
// block], dropping needs no copy for a chain: the next block simply
// overwrites the rejected slots once ctx_len has moved past the kept ones.
// A tree keeps a root path whose nodes sit at scattered block slots, so
// their K/V rows are first moved to consecutive positions.
#include <algorithm>

#include "common.cuh"

namespace sdv {

namespace {

constexpr int kCommitWarps = 8;
constexpr int kCompactThreads = 128;

// one warp per sequence
__global__ void __launch_bounds__(kCommitWarps * 32) commit_tokens_kernel(const CommitParams p) {
#if __CUDA_ARCH__ >= 900
    asm volatile("griddepcontrol.wait;" ::: "memory");
#endif
    const int lane = threadIdx.x & 31;
    const int b = blockIdx.x * kCommitWarps + (threadIdx.x >> 5);
    if (b >= p.B) return;
    const int n = p.n_acc[b];
    const int c = p.ctx_len[b];
    const int ol = p.out_len[b];
    bool ok = n >= 0 && n <= p.T - 1;
    // committed token i (i <= n, at most 64): kept proposal i, then the next token;
    // lane l takes tokens l and l + 32
    int tok[2] = {0, 0};
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int i = lane + 32 * k;
        if (ok && i < n) {
            int src = i;
            if (p.path) {
                const int node = p.path[(long)b * p.T + i];
                ok = node >= 1 && node < p.T;
                src = node;
            }
            if (ok) tok[k] = p.prop[(long)b * p.ps + src];
        }
        if (i == n) tok[k] = p.next_tok[b];
    }
    ok = __all_sync(0xffffffffu, ok);
    ok = ok && (long)c + n + 1 <= p.ctx_cap && ol >= 0 && (long)ol + n + 1 <= p.out_cap && c >= 1;
    if (!ok) {
        if (lane == 0) {
            if (p.status) p.status[b] = 1;
            set_fault(p.fault, FAULT_BAD_COMMIT);
        }
        return;
    }
#pragma unroll
    for (int k = 0; k < 2; ++k)
        if (lane + 32 * k <= n) p.out_tokens[(long)b * p.out_cap + ol + lane + 32 * k] = tok[k];
    if (lane == 0) {
        p.out_len[b] = ol + n + 1;
        p.ctx_len[b] = c + n + 1;
        if (p.draft_ctx) p.draft_ctx[b] = c + n;
        p.anchor[b] = p.next_tok[b];
        if (p.status) p.status[b] = 0;
    }
}

// CTA (b, h): moves the rows of the kept nodes of sequence b, kv head h, to
// positions ctx-1+1 .. ctx-1+n, K then V.  Every kept row of a cache is read
// into shared memory before any is written: a destination may be another
// depth's source.
__global__ void __launch_bounds__(kCompactThreads) compact_tree_kv_kernel(const CompactParams p) {
#if __CUDA_ARCH__ >= 900
    asm volatile("griddepcontrol.wait;" ::: "memory");
#endif
    __shared__ uint4 stage[kMaxTreeT - 1][kMaxHeadBytes / 16];
    const int b = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
    const int n = p.n_acc[b], c = p.ctx_len[b];
    bool ok = n >= 0 && n <= p.T - 1 && c >= 1 && (long)c - 1 + p.T <= p.S;
    for (int d = 1; ok && d <= n; ++d) {
        const int node = p.path[(long)b * p.T + d - 1];
        ok = node >= 1 && node < p.T;
    }
    if (!ok) {
        if (h == 0 && tid == 0) set_fault(p.fault, FAULT_BAD_COMMIT);
        return;
    }
    const int vec = p.D * p.es / 16;              // 16-byte words per row
    const long es = p.es;
    const long base = ((long)b * p.kv.b + (long)h * p.kv.h) * es;
    for (int kv = 0; kv < 2; ++kv) {
        char *cache = static_cast<char *>(kv ? p.vc : p.kc);
        for (int i = tid; i < n * vec; i += kCompactThreads) {
            const int d = i / vec, x = i % vec;
            const int node = p.path[(long)b * p.T + d];
            stage[d][x] = reinterpret_cast<const uint4 *>(cache + base + (long)(c - 1 + node) * p.kv.s * es)[x];
        }
        __syncthreads();
        for (int i = tid; i < n * vec; i += kCompactThreads) {
            const int d = i / vec, x = i % vec;
            reinterpret_cast<uint4 *>(cache + base + (long)(c + d) * p.kv.s * es)[x] = stage[d][x];
        }
        __syncthreads();   // the stage is reused by the next cache
    }
}

// A grid-stride copy of 16-byte vectors.  The stores cross the chip-to-host
// link one by one, so a handful of CTAs per SM keep enough of them in flight;
// for the few hundred KB of a step's results this ends sooner than a
// copy-engine transfer, whose set-up dominates at that size.
constexpr int kStoreThreads = 256;
constexpr int kStoreCtasPerSm = 4;
__global__ void __launch_bounds__(kStoreThreads) store_to_host_kernel(const HostStoreParams p) {
#if __CUDA_ARCH__ >= 900
    asm volatile("griddepcontrol.wait;" ::: "memory");   // the results of the kernels before
#endif
    const int64_t stride = (int64_t)gridDim.x * kStoreThreads;
    for (int64_t i = (int64_t)blockIdx.x * kStoreThreads + threadIdx.x; i < p.n16; i += stride)
        p.dst[i] = __ldcg(p.src + i);
}

template <typename K, typename P>
cudaError_t launch_pdl_cm(K kern, dim3 grid, dim3 block, cudaStream_t st, const P &args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args);
}

}  // namespace

cudaError_t launch_commit_tokens(const CommitParams &p, cudaStream_t st) {
    const dim3 grid((unsigned)((p.B + kCommitWarps - 1) / kCommitWarps));
    return launch_pdl_cm(commit_tokens_kernel, grid, dim3(kCommitWarps * 32), st, p);
}

cudaError_t launch_store_to_host(const HostStoreParams &p, int sm_count, cudaStream_t st) {
    const int64_t need = (p.n16 + kStoreThreads - 1) / kStoreThreads;
    const int64_t cap = (int64_t)std::max(1, sm_count) * kStoreCtasPerSm;
    return launch_pdl_cm(store_to_host_kernel, dim3((unsigned)std::min(need, cap)), dim3(kStoreThreads), st, p);
}

cudaError_t launch_compact_tree_kv(const CompactParams &p, cudaStream_t st) {
    return launch_pdl_cm(compact_tree_kv_kernel, dim3((unsigned)p.B, (unsigned)p.Hkv), dim3(kCompactThreads), st, p);
}

}  // namespace sdv
