// Acceptance kernels: greedy first-mismatch prefix + correction, and the
// lossless sampled accept / residual resample, plus Philox4x32-10.
//
// Greedy: "VFlash-FM" project page, worked cycle -- proposals equal to the
// target's greedy picks are kept up to the first mismatch, where the target's
// own pick is committed.  Sampled: "SpecFLASH" README, inference section --
// the standard speculative accept/reject rule.  Philox: Salmon et al., SC'11,
// section 3.2.
//
// Both reductions are vocabulary-wide over B*T rows: a grid of (chunk, row)
// CTAs reads each row once with 16-byte loads, reduces within warps by
// shuffles and across warps through shared memory, writes one partial per CTA,
// and the last CTA to finish (a ticket counter in the workspace, returned to
// zero by that CTA) combines the partials and runs the per-sequence scan.  No
// CTA ever waits for another.
#include "common.cuh"

#include <float.h>
#include <limits.h>
#include <math.h>

namespace sdv {

namespace {

constexpr int kAccThreads = 256;

// ----------------------------------------------------------------------------
// Philox4x32-10
// ----------------------------------------------------------------------------
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
        const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
        c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return c;
}

// U(seed; row, batch, stream, offset) = (word0 >> 8) * 2^-24
__device__ __forceinline__ float philox_uniform(uint64_t seed, uint32_t row, uint32_t batch,
                                                uint32_t stream, uint32_t offset) {
    const uint4 w = philox4x32_10(make_uint4(row, batch, stream, offset), (uint32_t)seed,
                                  (uint32_t)(seed >> 32));
    return (float)(w.x >> 8) * (1.0f / 16777216.0f);
}

__global__ void philox_kernel(const uint4 *__restrict__ ctr, uint64_t key, uint4 *__restrict__ out,
                              int64_t n) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) out[i] = philox4x32_10(ctr[i], (uint32_t)key, (uint32_t)(key >> 32));
}

// ----------------------------------------------------------------------------
// chunk traversal: calls f(index, value) for every element of [lo, hi) of a row,
// in ascending index order per thread, 16-byte loads where aligned
// ----------------------------------------------------------------------------
template <typename Tin, typename F>
__device__ __forceinline__ void for_chunk(const Tin *row, int lo, int hi, F &&f) {
    constexpr int PV = Elem<Tin>::kPerVec;
    // first index >= lo whose address is 16-byte aligned
    const uintptr_t base = reinterpret_cast<uintptr_t>(row);
    int a0 = lo;
    while (a0 < hi && ((base + (uintptr_t)a0 * sizeof(Tin)) & 15u)) ++a0;
    const int nvec = (hi - a0) / PV;
    const int a1 = a0 + nvec * PV;
    for (int i = lo + (int)threadIdx.x; i < a0; i += kAccThreads) f(i, Elem<Tin>::load(row + i));
    for (int v = threadIdx.x; v < nvec; v += kAccThreads) {
        float x[PV];
        Elem<Tin>::load_vec(row + a0 + v * PV, x);
#pragma unroll
        for (int e = 0; e < PV; ++e) f(a0 + v * PV + e, x[e]);
    }
    for (int i = a1 + (int)threadIdx.x; i < hi; i += kAccThreads) f(i, Elem<Tin>::load(row + i));
}

__device__ __forceinline__ void warp_argmax(float &v, int &i) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, v, o);
        const int oi = __shfl_xor_sync(0xffffffffu, i, o);
        if (argmax_better(ov, oi, v, i)) { v = ov; i = oi; }
    }
}

// block-wide (value, index) argmax; result valid in every thread
__device__ __forceinline__ void block_argmax(float &v, int &i) {
    __shared__ float sv[kAccThreads / 32];
    __shared__ int si[kAccThreads / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    warp_argmax(v, i);
    __syncthreads();
    if (lane == 0) { sv[warp] = v; si[warp] = i; }
    __syncthreads();
    v = sv[0]; i = si[0];
    for (int w = 1; w < kAccThreads / 32; ++w)
        if (argmax_better(sv[w], si[w], v, i)) { v = sv[w]; i = si[w]; }
}

template <typename T>
__device__ __forceinline__ T block_sum(T x) {
    __shared__ T sh[kAccThreads / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    __syncthreads();
    if (lane == 0) sh[warp] = x;
    __syncthreads();
    T t = sh[0];
    for (int w = 1; w < kAccThreads / 32; ++w) t += sh[w];
    return t;
}

__device__ __forceinline__ float block_max(float x) {
    __shared__ float sh[kAccThreads / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    __syncthreads();
    if (lane == 0) sh[warp] = x;
    __syncthreads();
    float t = sh[0];
    for (int w = 1; w < kAccThreads / 32; ++w) t = fmaxf(t, sh[w]);
    return t;
}

// last-CTA election: true in every thread of the CTA that finished last
__device__ __forceinline__ bool last_cta_done(unsigned int *counter, unsigned int total) {
    __shared__ bool is_last;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) is_last = atomicAdd(counter, 1u) == total - 1;
    __syncthreads();
    if (is_last) __threadfence();
    return is_last;
}

// ----------------------------------------------------------------------------
// greedy acceptance
// ----------------------------------------------------------------------------
template <typename Tin>
__global__ void __launch_bounds__(kAccThreads) greedy_kernel(const GreedyParams p) {
    const int c = blockIdx.x, row = blockIdx.y;
    const int lo = c * p.chunk, hi = min(p.V, lo + p.chunk);
    const Tin *lg = static_cast<const Tin *>(p.logits) + (long)row * p.V;
    float bv = -INFINITY;
    int bi = INT_MAX;
    for_chunk<Tin>(lg, lo, hi, [&](int i, float x) {
        if (argmax_better(x, i, bv, bi)) { bv = x; bi = i; }
    });
    block_argmax(bv, bi);
    if (threadIdx.x == 0) {
        p.pval[(long)row * p.n_chunks + c] = bv;
        p.pidx[(long)row * p.n_chunks + c] = bi;
    }
    const unsigned int total = gridDim.x * gridDim.y;
    if (!last_cta_done(p.counter, total)) return;

    // finisher: per-row argmax over the chunk partials, then the prefix scan,
    // over windows holding whole sequences (W rows, a multiple of T)
    __shared__ int amax[kAccThreads];
    const int R = p.B * p.T;
    const int W = (kAccThreads / p.T) * p.T;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int r0 = 0; r0 < R; r0 += W) {
        for (int r = r0 + warp; r < min(R, r0 + W); r += kAccThreads / 32) {
            float v = -INFINITY;
            int i = INT_MAX;
            for (int k = lane; k < p.n_chunks; k += 32) {
                const float pv = __ldcg(p.pval + (long)r * p.n_chunks + k);
                const int pi = __ldcg(p.pidx + (long)r * p.n_chunks + k);
                if (argmax_better(pv, pi, v, i)) { v = pv; i = pi; }
            }
            warp_argmax(v, i);
            if (lane == 0) {
                if (i == INT_MAX) { set_fault(p.fault, FAULT_NAN_ROW); i = 0; }
                amax[r - r0] = i;
            }
        }
        __syncthreads();
        const int b0 = r0 / p.T, nbw = min(p.B - b0, W / p.T);
        for (int bl = threadIdx.x; bl < nbw; bl += kAccThreads) {
            const int b = b0 + bl, rb = bl * p.T;
            int n = p.T - 1;
            for (int j = 0; j < p.T - 1; ++j) {
                if (p.draft[(long)b * (p.T - 1) + j] != amax[rb + j]) { n = j; break; }
            }
            p.n_acc[b] = n;
            p.corr[b] = amax[rb + n];
        }
        __syncthreads();
    }
    if (threadIdx.x == 0) *p.counter = 0u;
}

// ----------------------------------------------------------------------------
// sampled acceptance, pass 1: per-row max and sum of exp over chunks, then the
// accept scan (last CTA)
// ----------------------------------------------------------------------------
template <typename Tin>
__global__ void __launch_bounds__(kAccThreads) sample_stats_kernel(const SampleParams p) {
    const int c = blockIdx.x, row = blockIdx.y;
    const int lo = c * p.chunk, hi = min(p.V, lo + p.chunk);
    const Tin *lg = static_cast<const Tin *>(p.logits) + (long)row * p.V;
    const float it = p.inv_tau;
    float m = -INFINITY;
    for_chunk<Tin>(lg, lo, hi, [&](int, float x) { m = fmaxf(m, x * it); });
    m = block_max(m);
    float z = 0.f;
    if (m != -INFINITY) for_chunk<Tin>(lg, lo, hi, [&](int, float x) { z += expf(x * it - m); });
    const double zs = block_sum<double>((double)z);
    if (threadIdx.x == 0) {
        p.pm[(long)row * p.n_chunks + c] = m;
        p.pz[(long)row * p.n_chunks + c] = (float)zs;
    }
    const unsigned int total = gridDim.x * gridDim.y;
    if (!last_cta_done(p.counters, total)) return;

    // finisher: per-row max / normaliser from the chunk partials (a warp per
    // row), then one thread per sequence scans its rows in order; windows of
    // W rows hold whole sequences
    __shared__ float rowM[kAccThreads];
    __shared__ float rowZ[kAccThreads];
    const int R = p.B * p.T;
    const int W = (kAccThreads / p.T) * p.T;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int r0 = 0; r0 < R; r0 += W) {
        for (int r = r0 + warp; r < min(R, r0 + W); r += kAccThreads / 32) {
            float M = -INFINITY;
            for (int k = lane; k < p.n_chunks; k += 32) M = fmaxf(M, __ldcg(p.pm + (long)r * p.n_chunks + k));
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
            double Z = 0.0;
            for (int k = lane; k < p.n_chunks; k += 32) {
                const float mk = __ldcg(p.pm + (long)r * p.n_chunks + k);
                if (mk != -INFINITY)
                    Z += (double)__ldcg(p.pz + (long)r * p.n_chunks + k) * (double)expf(mk - M);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) Z += __shfl_xor_sync(0xffffffffu, Z, o);
            if (lane == 0) { rowM[r - r0] = M; rowZ[r - r0] = (float)Z; }
        }
        __syncthreads();
        const int b0 = r0 / p.T, nbw = min(p.B - b0, W / p.T);
        for (int bl = threadIdx.x; bl < nbw; bl += kAccThreads) {
            const int b = b0 + bl;
            int n = p.T - 1;
            for (int j = 0; j < p.T - 1; ++j) {
                const long r = (long)b * p.T + j;
                const float M = rowM[bl * p.T + j], Zr = rowZ[bl * p.T + j];
                const int d = p.draft[(long)b * (p.T - 1) + j];
                float pd = 0.f, qd = 0.f;
                if (d >= 0 && d < p.V) {
                    const Tin *lgr = static_cast<const Tin *>(p.logits) + r * p.V;
                    pd = expf(Elem<Tin>::load(lgr + d) * it - M) / Zr;
                    qd = __ldg(p.q + r * p.V + d);
                } else {
                    set_fault(p.fault, FAULT_BAD_DRAFT_ID);
                }
                const float u = philox_uniform(p.seed, (uint32_t)j, (uint32_t)b, 0u, p.offset);
                if (!(u * qd < pd)) { n = j; break; }
            }
            p.n_acc[b] = n;
            p.state[b] = make_float4(__int_as_float(n), rowM[bl * p.T + n], rowZ[bl * p.T + n], 0.f);
        }
        __syncthreads();
    }
    if (threadIdx.x == 0) *p.counters = 0u;
}

// ----------------------------------------------------------------------------
// sampled acceptance, pass 2: chunk sums of the residual (and of p) on the
// row that decides the next token, then the inverse-cdf draw (last CTA)
// ----------------------------------------------------------------------------
template <typename Tin>
__device__ __forceinline__ float draw_weight(const SampleParams &p, const Tin *lg, const float *qn,
                                             bool residual, float M, float Z, int i, float x) {
    const float pi = expf(x * p.inv_tau - M) / Z;
    if (!residual) return pi;
    const float r = pi - __ldg(qn + i);
    return r > 0.f ? r : 0.f;
}

template <typename Tin>
__global__ void __launch_bounds__(kAccThreads) sample_draw_kernel(const SampleParams p) {
    const int c = blockIdx.x, b = blockIdx.y;
    const float4 st = p.state[b];
    const int n = __float_as_int(st.x);
    const float M = st.y, Z = st.z;
    const bool rejected = n < p.T - 1;
    const long r = (long)b * p.T + n;
    const Tin *lg = static_cast<const Tin *>(p.logits) + r * p.V;
    const float *qn = p.q + r * p.V;
    const int lo = c * p.chunk, hi = min(p.V, lo + p.chunk);
    double sr = 0.0, sp = 0.0;
    for_chunk<Tin>(lg, lo, hi, [&](int i, float x) {
        const float pi = expf(x * p.inv_tau - M) / Z;
        sp += pi;
        if (rejected) {
            const float rr = pi - __ldg(qn + i);
            sr += rr > 0.f ? rr : 0.f;
        }
    });
    sr = block_sum<double>(sr);
    sp = block_sum<double>(sp);
    if (threadIdx.x == 0) {
        p.rs[(long)b * p.n_chunks + c] = sr;
        p.ps[(long)b * p.n_chunks + c] = sp;
    }
    const unsigned int total = gridDim.x * gridDim.y;
    if (!last_cta_done(p.counters + 1, total)) return;

    __shared__ double tsum[kAccThreads];
    __shared__ int sel_chunk;
    __shared__ double sel_base, sel_x;
    __shared__ int sel_res;
    for (int bb = 0; bb < p.B; ++bb) {
        const float4 s2 = __ldcg(&p.state[bb]);
        const int nb = __float_as_int(s2.x);
        const float Mb = s2.y, Zb = s2.z;
        const bool rej = nb < p.T - 1;
        if (threadIdx.x == 0) {
            double Sr = 0.0, Sp = 0.0;
            for (int k = 0; k < p.n_chunks; ++k) {
                Sr += __ldcg(p.rs + (long)bb * p.n_chunks + k);
                Sp += __ldcg(p.ps + (long)bb * p.n_chunks + k);
            }
            const bool use_r = rej && Sr > 0.0;
            const double* cs = use_r ? p.rs : p.ps;
            const double S = use_r ? Sr : Sp;
            const float u2 = philox_uniform(p.seed, (uint32_t)nb, (uint32_t)bb, 1u, p.offset);
            const double x = (double)u2 * S;
            double base = 0.0;
            int ck = -1, last_pos = 0;
            for (int k = 0; k < p.n_chunks; ++k) {
                const double v = __ldcg(cs + (long)bb * p.n_chunks + k);
                if (v > 0.0) last_pos = k;
                if (ck < 0 && base + v > x) { ck = k; break; }
                base += v;
            }
            if (ck < 0) {  // x reached the total through rounding: last non-empty chunk
                ck = last_pos;
                base = 0.0;
                for (int k = 0; k < ck; ++k) base += __ldcg(cs + (long)bb * p.n_chunks + k);
            }
            sel_chunk = ck; sel_base = base; sel_x = x; sel_res = use_r ? 1 : 0;
        }
        __syncthreads();
        // inclusive scan of the selected chunk, in index order: each thread owns a
        // contiguous run, runs are combined by an exclusive scan over threads
        const long rr = (long)bb * p.T + nb;
        const Tin *lgb = static_cast<const Tin *>(p.logits) + rr * p.V;
        const float *qb = p.q + rr * p.V;
        const int clo = sel_chunk * p.chunk, chi = min(p.V, clo + p.chunk);
        const int per = (chi - clo + kAccThreads - 1) / kAccThreads;
        const int tlo = min(chi, clo + (int)threadIdx.x * per), thi = min(chi, tlo + per);
        double run = 0.0;
        for (int i = tlo; i < thi; ++i)
            run += draw_weight<Tin>(p, lgb, qb, sel_res != 0, Mb, Zb, i, Elem<Tin>::load(lgb + i));
        tsum[threadIdx.x] = run;
        __syncthreads();
        if (threadIdx.x == 0) {
            // find the thread whose run crosses x, then the element
            double acc = sel_base;
            int owner = -1;
            for (int t = 0; t < kAccThreads; ++t) {
                if (acc + tsum[t] > sel_x) { owner = t; break; }
                acc += tsum[t];
            }
            int id = -1, last_pos = -1;
            if (owner >= 0) {
                const int olo = min(chi, clo + owner * per), ohi = min(chi, olo + per);
                for (int i = olo; i < ohi; ++i) {
                    const float w = draw_weight<Tin>(p, lgb, qb, sel_res != 0, Mb, Zb, i,
                                                     Elem<Tin>::load(lgb + i));
                    if (w > 0.f) last_pos = i;
                    acc += w;
                    if (acc > sel_x) { id = i; break; }
                }
            }
            if (id < 0) {  // rounding: the last positive-weight index of the chunk
                for (int i = chi - 1; i >= clo; --i) {
                    if (draw_weight<Tin>(p, lgb, qb, sel_res != 0, Mb, Zb, i,
                                         Elem<Tin>::load(lgb + i)) > 0.f) { last_pos = i; break; }
                }
                id = last_pos >= 0 ? last_pos : clo;
            }
            p.next_id[bb] = id;
        }
        __syncthreads();
    }
    if (threadIdx.x == 0) p.counters[1] = 0u;
}

}  // namespace

cudaError_t launch_accept_greedy(const GreedyParams &p, cudaStream_t st) {
    dim3 grid(p.n_chunks, p.B * p.T);
    if (p.dt == SD_BF16) greedy_kernel<__nv_bfloat16><<<grid, kAccThreads, 0, st>>>(p);
    else greedy_kernel<float><<<grid, kAccThreads, 0, st>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_accept_sample(const SampleParams &p, cudaStream_t st) {
    dim3 g1(p.n_chunks, p.B * p.T), g2(p.n_chunks, p.B);
    if (p.dt == SD_BF16) {
        sample_stats_kernel<__nv_bfloat16><<<g1, kAccThreads, 0, st>>>(p);
        sample_draw_kernel<__nv_bfloat16><<<g2, kAccThreads, 0, st>>>(p);
    } else {
        sample_stats_kernel<float><<<g1, kAccThreads, 0, st>>>(p);
        sample_draw_kernel<float><<<g2, kAccThreads, 0, st>>>(p);
    }
    return cudaGetLastError();
}

cudaError_t launch_philox(const uint32_t *ctr, uint64_t key, uint32_t *out, int64_t n,
                          cudaStream_t st) {
    const int threads = 256;
    const int64_t blocks = (n + threads - 1) / threads;
    philox_kernel<<<(unsigned)blocks, threads, 0, st>>>(reinterpret_cast<const uint4 *>(ctr), key,
                                                        reinterpret_cast<uint4 *>(out), n);
    return cudaGetLastError();
}

}  // namespace sdv
