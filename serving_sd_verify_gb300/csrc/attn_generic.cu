// CUDA-core split-KV attention (any supported shape, fp32 or bf16 storage)
// and the log-sum-exp merge shared by both attention kernels.
//
// Target verify: "VFlash-FM" project page, "How VFlash-FM works" -- the
// target scores the 16 block slots in one forward with grouped-query
// attention over its KV cache; slot j only sees keys before slot j+1.
// Drafter: same page -- block queries see every projected context key and
// every block key.
//
// One CTA owns one (split, kv head, sequence) and loops over all G*T query
// rows that read this kv head, so each K/V tile is read from HBM once and used
// by every row.  Per tile of 32 keys a warp handles one row: lane = key for the
// dot products, a warp-shuffle max / sum for the online softmax (log2 domain),
// and lane = output dimension for the P.V update.  Per-row state (O, m, l)
// lives in shared memory.
#include "common.cuh"

#include <math.h>
#include <atomic>

namespace sdv {

namespace {

constexpr int kGenThreads = 128;
constexpr int kGenTile = 32;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// rows per pass so that Q and O of the pass take at most 64 KB of shared memory
template <int D> struct RowsPerPass { static constexpr int value = 8192 / D; };

template <typename Tin, int D>
__global__ void __launch_bounds__(kGenThreads)
attn_split_generic_kernel(const AttnParams p) {
    constexpr int RC = RowsPerPass<D>::value;
    constexpr int KS = D + 1;  // padded K row: lane-indexed reads hit distinct banks
    constexpr int VPR = D / Elem<Tin>::kPerVec;  // 16-byte vectors per key row
    extern __shared__ float smem[];
    float *Ks = smem;                    // [32][D+1]
    float *Vs = Ks + kGenTile * KS;      // [32][D]
    float *Qs = Vs + kGenTile * D;       // [RC][D], pre-multiplied by scale*log2(e)
    float *Os = Qs + RC * D;             // [RC][D]
    float *Ms = Os + RC * D;             // [RC] running max (log2 units)
    float *Ls = Ms + RC;                 // [RC] running sum

    const int s = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int T = p.T, G = p.Hq / p.Hkv, R = G * T;

    int nb = p.nctx[b];
    if (nb < 1 || nb > p.max_ctx) {
        if (tid == 0) set_fault(p.fault, FAULT_BAD_CTX);
        nb = max(1, min(nb, p.max_ctx));
    }
    const int N_b = p.mode == 1 ? nb + T : nb + T - 1;
    const int k0 = s * p.keys_per_split;
    const int k1 = min(N_b, k0 + p.keys_per_split);
    const float qscale = p.scale * kLog2e;
    const Tin *q = static_cast<const Tin *>(p.q);
    const Tin *kc = static_cast<const Tin *>(p.kc);
    const Tin *vc = static_cast<const Tin *>(p.vc);
    const Tin *kb = static_cast<const Tin *>(p.kb);
    const Tin *vb = static_cast<const Tin *>(p.vb);
    const long rows_total = (long)p.B * T * p.Hq;

    for (int rc0 = 0; rc0 < R; rc0 += RC) {
        const int nr = min(RC, R - rc0);
        __syncthreads();
        // row r of the pass = (j, h) with r + rc0 = j*G + hl, h = g*G + hl
        for (int idx = tid; idx < nr * D; idx += kGenThreads) {
            const int r = idx / D, d = idx % D;
            const int row = rc0 + r, j = row / G, h = g * G + row % G;
            Qs[idx] = Elem<Tin>::load(q + (((long)b * T + j) * p.Hq + h) * D + d) * qscale;
            Os[idx] = 0.f;
        }
        for (int r = tid; r < nr; r += kGenThreads) { Ms[r] = -INFINITY; Ls[r] = 0.f; }

        for (int kt = k0; kt < k1; kt += kGenTile) {
            __syncthreads();
            for (int idx = tid; idx < kGenTile * VPR; idx += kGenThreads) {
                const int kk = idx / VPR, vv = idx % VPR, key = kt + kk;
                float kf[Elem<Tin>::kPerVec], vf[Elem<Tin>::kPerVec];
                if (key < k1) {
                    const Tin *kp, *vp;
                    if (p.mode == 1 && key >= nb) {
                        const long off = (((long)b * T + (key - nb)) * p.Hkv + g) * D;
                        kp = kb + off; vp = vb + off;
                    } else {
                        const long off = (long)b * p.kv.b + (long)key * p.kv.s + (long)g * p.kv.h;
                        kp = kc + off; vp = vc + off;
                    }
                    Elem<Tin>::load_vec(kp + vv * Elem<Tin>::kPerVec, kf);
                    Elem<Tin>::load_vec(vp + vv * Elem<Tin>::kPerVec, vf);
                } else {
#pragma unroll
                    for (int e = 0; e < Elem<Tin>::kPerVec; ++e) { kf[e] = 0.f; vf[e] = 0.f; }
                }
#pragma unroll
                for (int e = 0; e < Elem<Tin>::kPerVec; ++e) {
                    Ks[kk * KS + vv * Elem<Tin>::kPerVec + e] = kf[e];
                    Vs[kk * D + vv * Elem<Tin>::kPerVec + e] = vf[e];
                }
            }
            __syncthreads();
            for (int r = warp; r < nr; r += kGenThreads / 32) {
                const int row = rc0 + r, j = row / G;
                const int key = kt + lane;
                bool valid;
                if (p.mode == 2) {
                    // tree: the context before the anchor, then the slots of the node's mask
                    const int slot = key - (nb - 1);
                    valid = key < k1 && (slot < 0 || (slot < T && ((p.tree_mask[(long)b * T + j] >> slot) & 1ull)));
                } else {
                    valid = key < min(k1, p.mode == 0 ? nb + j : N_b);
                }
                float sc = 0.f;
                const float *qr = Qs + r * D;
                const float *kr = Ks + lane * KS;
#pragma unroll 8
                for (int d = 0; d < D; ++d) sc = fmaf(qr[d], kr[d], sc);
                sc = valid ? sc : -INFINITY;
                const float tmax = warp_max(sc);
                const float m_old = Ms[r];
                const float m_new = fmaxf(m_old, tmax);
                if (m_new == -INFINITY) continue;  // warp-uniform: no valid key yet
                const float pv = valid ? exp2f(sc - m_new) : 0.f;
                const float psum = warp_sum(pv);
                const float alpha = exp2f(m_old - m_new);  // 0 when m_old = -inf
                float acc[D / 32];
#pragma unroll
                for (int c = 0; c < D / 32; ++c) acc[c] = Os[r * D + lane + 32 * c] * alpha;
#pragma unroll 4
                for (int kk = 0; kk < kGenTile; ++kk) {
                    const float pk = __shfl_sync(0xffffffffu, pv, kk);
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) acc[c] = fmaf(pk, Vs[kk * D + lane + 32 * c], acc[c]);
                }
#pragma unroll
                for (int c = 0; c < D / 32; ++c) Os[r * D + lane + 32 * c] = acc[c];
                __syncwarp();
                if (lane == 0) { Ms[r] = m_new; Ls[r] = Ls[r] * alpha + psum; }
                __syncwarp();
            }
        }
        __syncthreads();
        // partial output (normalised) and its log-sum-exp, natural log
        for (int r = warp; r < nr; r += kGenThreads / 32) {
            const int row = rc0 + r, j = row / G, h = g * G + row % G;
            const long frow = ((long)b * T + j) * p.Hq + h;
            const float l = Ls[r];
            const float inv = l > 0.f ? 1.f / l : 0.f;
            float *dst = p.o_part + ((long)s * rows_total + frow) * D;
            for (int d = lane; d < D; d += 32) dst[d] = Os[r * D + d] * inv;
            if (lane == 0)
                p.lse_part[(long)s * rows_total + frow] = l > 0.f ? Ms[r] * kLn2 + logf(l) : -INFINITY;
        }
    }
}

// Log-sum-exp merge of the split partials, one CTA of 4 warps per output row:
//   out = sum_s exp(lse_s - M) O_s / sum_s exp(lse_s - M),  M = max_s lse_s.
// Warp w takes splits w, w+4, ...; each lane owns D/32 output columns.  Empty
// splits carry lse = -inf and a zero partial, so the sums need no branch and
// the loads of four splits are in flight together.
template <int D>
__global__ void __launch_bounds__(128) lse_merge_kernel(const float *__restrict__ o_part,
                                                        const float *__restrict__ lse_part,
                                                        float *__restrict__ out, long rows, int n_splits) {
#if __CUDA_ARCH__ >= 900
    asm volatile("griddepcontrol.wait;" ::: "memory");
#endif
    constexpr int VW = D / 32;  // floats per lane
    __shared__ float s_max[4];
    __shared__ float s_wsum[4];
    __shared__ float s_acc[4][D];
    const long row = blockIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float M = -INFINITY;
    for (int sp = threadIdx.x; sp < n_splits; sp += 128) M = fmaxf(M, __ldcg(lse_part + (long)sp * rows + row));
    M = warp_max(M);
    if (lane == 0) s_max[warp] = M;
    __syncthreads();
    M = fmaxf(fmaxf(s_max[0], s_max[1]), fmaxf(s_max[2], s_max[3]));
    float acc[VW];
#pragma unroll
    for (int e = 0; e < VW; ++e) acc[e] = 0.f;
    float wsum = 0.f;
    if (M != -INFINITY) {
        int sp = warp;
        for (; sp + 12 < n_splits; sp += 16) {
            float w[4], v[4][VW];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const long ss = sp + 4 * u;
                const float l = __ldcg(lse_part + ss * rows + row);
                w[u] = __expf(l - M);  // 0 for an empty split (l = -inf)
                const float *src = o_part + (ss * rows + row) * D + lane * VW;
                if constexpr (VW == 4) {
                    const float4 t4 = __ldcg(reinterpret_cast<const float4 *>(src));
                    v[u][0] = t4.x; v[u][1] = t4.y; v[u][2] = t4.z; v[u][3] = t4.w;
                } else {
                    const float2 t2 = __ldcg(reinterpret_cast<const float2 *>(src));
                    v[u][0] = t2.x; v[u][1] = t2.y;
                }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                wsum += w[u];
#pragma unroll
                for (int e = 0; e < VW; ++e) acc[e] = fmaf(w[u], v[u][e], acc[e]);
            }
        }
        for (; sp < n_splits; sp += 4) {
            const float l = __ldcg(lse_part + (long)sp * rows + row);
            const float w = __expf(l - M);
            const float *src = o_part + ((long)sp * rows + row) * D + lane * VW;
            wsum += w;
#pragma unroll
            for (int e = 0; e < VW; ++e) acc[e] = fmaf(w, __ldcg(src + e), acc[e]);
        }
    }
    if (lane == 0) s_wsum[warp] = wsum;
#pragma unroll
    for (int e = 0; e < VW; ++e) s_acc[warp][lane * VW + e] = acc[e];
    __syncthreads();
    const float wt = (s_wsum[0] + s_wsum[1]) + (s_wsum[2] + s_wsum[3]);
    const float inv = wt > 0.f ? 1.f / wt : 0.f;
    for (int d = threadIdx.x; d < D; d += 128)
        out[row * D + d] = ((s_acc[0][d] + s_acc[1][d]) + (s_acc[2][d] + s_acc[3][d])) * inv;
}

template <typename Tin, int D>
cudaError_t launch_generic_t(const AttnParams &p, cudaStream_t st) {
    constexpr int RC = RowsPerPass<D>::value;
    const size_t smem = sizeof(float) * (kGenTile * (D + 1) + kGenTile * D + 2 * RC * D + 2 * RC);
    auto kern = attn_split_generic_kernel<Tin, D>;
    // the shared-memory opt-in is set once per device, before any graph capture
    static std::atomic<bool> opted_in[64];  // per device: shared-memory limit raised
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !opted_in[dev].load(std::memory_order_acquire)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) opted_in[dev].store(true, std::memory_order_release);
    }
    dim3 grid(p.n_splits, p.Hkv, p.B);
    kern<<<grid, kGenThreads, smem, st>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_generic(const AttnParams &p, cudaStream_t st) {
    if (p.dt == SD_BF16) {
        return p.D == 128 ? launch_generic_t<__nv_bfloat16, 128>(p, st)
                          : launch_generic_t<__nv_bfloat16, 64>(p, st);
    }
    return p.D == 128 ? launch_generic_t<float, 128>(p, st) : launch_generic_t<float, 64>(p, st);
}

cudaError_t launch_lse_merge(const AttnParams &p, cudaStream_t st) {
    const long rows = (long)p.B * p.T * p.Hq;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)rows);
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (p.D == 128)
        return cudaLaunchKernelEx(&cfg, lse_merge_kernel<128>, (const float *)p.o_part, (const float *)p.lse_part,
                                  p.out, rows, p.n_splits);
    return cudaLaunchKernelEx(&cfg, lse_merge_kernel<64>, (const float *)p.o_part, (const float *)p.lse_part,
                              p.out, rows, p.n_splits);
}

}  // namespace sdv
