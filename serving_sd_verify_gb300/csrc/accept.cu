// Acceptance kernels: greedy first-mismatch prefix + correction, and the
// lossless sampled accept / residual resample, plus Philox4x32-10.
//
// Greedy: "VFlash-FM" project page, worked cycle -- proposals equal to the
// target's greedy picks are kept up to the first mismatch, where the target's
// own pick is committed.  Sampled: "SpecFLASH" README, inference section --
// the standard speculative accept/reject rule.  Philox: Salmon et al., SC'11,
// section 3.2.
//
// Both are vocabulary-wide reductions over B*T rows.  A grid of (chunk, row)
// CTAs reads every row once: each thread pulls its share of the chunk into
// registers with 16-byte loads issued together, reduces it, and the CTA
// reduces across warps (shuffles, then shared memory) into one partial.  The
// last CTA of a row to finish (a per-row ticket counter) combines that row's
// partials; the last row to finish (a second counter) runs the per-sequence
// scan.  Every counter is returned to zero by the CTA that read it last, so a
// zero-filled workspace stays reusable.  No CTA ever waits for another.
#include "common.cuh"

#include <float.h>
#include <limits.h>
#include <math.h>

namespace sdv {

namespace {

constexpr int kAccThreads = 256;
constexpr int kArgChains = 4;     // independent argmax chains per thread in the greedy stream
constexpr int kGreedyBatch = 4;   // 16-byte vectors per thread per batch of the pass-1 streams
constexpr int kFinRows = 4;       // rows per warp whose chunk partials a finisher loads together
constexpr int kFinStaged = 1024;  // chunk partials the greedy finisher stages in shared memory at once
constexpr int kDrawChunksStaged = 512;  // chunk sums the draw finisher stages in shared memory

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
// a chunk [lo, hi) of one row, pulled into registers: vector v (< NV) of this
// thread holds elements a0 + (tid + v * kAccThreads) * PV + e; the unaligned
// head [lo, a0) and tail [a1, hi) are read element by element
// ----------------------------------------------------------------------------
template <typename Tin, int NV>
struct ChunkRegs {
    static constexpr int PV = Elem<Tin>::kPerVec;
    float x[NV][PV];
    int a0, a1, nvec;

    __device__ __forceinline__ void load(const Tin *row, int lo, int hi, float fill) {
        const uintptr_t base = reinterpret_cast<uintptr_t>(row);
        int s = lo;
        while (s < hi && ((base + (uintptr_t)s * sizeof(Tin)) & 15u)) ++s;
        a0 = s;
        nvec = (hi - a0) / PV;
        a1 = a0 + nvec * PV;
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            const int vi = threadIdx.x + v * kAccThreads;
            if (vi < nvec) {
                Elem<Tin>::load_vec(row + a0 + vi * PV, x[v]);
            } else {
#pragma unroll
                for (int e = 0; e < PV; ++e) x[v][e] = fill;
            }
        }
    }
    __device__ __forceinline__ int index(int v, int e) const { return a0 + ((int)threadIdx.x + v * kAccThreads) * PV + e; }
    __device__ __forceinline__ bool valid(int v) const { return (int)threadIdx.x + v * kAccThreads < nvec; }
};

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
__device__ __forceinline__ T warp_sum(T x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

template <typename T>
__device__ __forceinline__ T block_sum(T x) {
    __shared__ T sh[kAccThreads / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    x = warp_sum(x);
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

// Programmatic dependent launch: the kernel may start while the previous one in
// the stream drains; wait here until its results are visible.
__device__ __forceinline__ void grid_dependency_wait() {
#if __CUDA_ARCH__ >= 900
    asm volatile("griddepcontrol.wait;" ::: "memory");
#endif
}

// Last-CTA election on `counter` among `total` arrivals: true in every thread of
// the CTA that arrived last, which also returns the counter to zero.  Only
// thread 0 of a CTA writes that CTA's partial results; its fence before the
// ticket makes them visible to the elected CTA, which reads them from L2.
__device__ __forceinline__ bool elect_last(unsigned int *counter, unsigned int total) {
    __shared__ bool is_last;
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        const unsigned int ticket = atomicAdd(counter, 1u);
        is_last = ticket == total - 1;
        if (is_last) {
            *counter = 0u;
            __threadfence();
        }
    }
    __syncthreads();
    return is_last;
}

// ----------------------------------------------------------------------------
// greedy acceptance
// ----------------------------------------------------------------------------
// 16-byte vector of logits -> floats
template <typename Tin> struct Vec16;
template <> struct Vec16<float> {
    static constexpr int PV = 4;
    __device__ __forceinline__ static void unpack(const uint4 &u, float (&f)[4]) {
        f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y);
        f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
    }
};
template <> struct Vec16<__nv_bfloat16> {
    static constexpr int PV = 8;
    __device__ __forceinline__ static void unpack(const uint4 &u, float (&f)[8]) { unpack_bf16x8(u, f); }
};

// CTA (c, row) streams chunk c of one row: the unaligned head and tail
// element by element, the 16-byte-aligned body in batches of kGreedyBatch
// vectors per thread, the next batch in flight while this one is reduced
template <typename Tin>
__global__ void __launch_bounds__(kAccThreads) greedy_kernel(const GreedyParams p) {
    grid_dependency_wait();
    constexpr int PV = Vec16<Tin>::PV;
    const int c = blockIdx.x, row = blockIdx.y, tid = threadIdx.x;
    const int lo = c * p.chunk, hi = min(p.V, lo + p.chunk);
    const Tin *lg = static_cast<const Tin *>(p.logits) + (long)row * p.V;
    const uintptr_t base = reinterpret_cast<uintptr_t>(lg);
    int a0 = lo;                                   // first 16-byte aligned index >= lo
    while (a0 < hi && ((base + (uintptr_t)a0 * sizeof(Tin)) & 15u)) ++a0;
    const int nvec = (hi - a0) / PV, a1 = a0 + nvec * PV;
    const uint4 *vp = reinterpret_cast<const uint4 *>(lg + a0);
    // kArgChains independent (value, index) chains per thread, so that
    // consecutive compares do not wait on each other; merged at the end by
    // the same rule (larger value, then lower index), so the result does not
    // depend on which chain saw which element
    float cv[kArgChains];
    int ci[kArgChains];
#pragma unroll
    for (int k = 0; k < kArgChains; ++k) { cv[k] = -INFINITY; ci[k] = INT_MAX; }
    for (int i = lo + tid; i < a0; i += kAccThreads) {
        const float x = Elem<Tin>::load(lg + i);
        if (argmax_better(x, i, cv[0], ci[0])) { cv[0] = x; ci[0] = i; }
    }
    uint4 cur[kGreedyBatch], nxt[kGreedyBatch];
    auto load = [&](uint4 (&d)[kGreedyBatch], int v0) {
#pragma unroll
        for (int u = 0; u < kGreedyBatch; ++u) {
            const int vi = v0 + u * kAccThreads;
            d[u] = vi < nvec ? ld_stream_u4(vp + vi) : make_uint4(0u, 0u, 0u, 0u);
        }
    };
    load(cur, tid);
    for (int v0 = tid; v0 < nvec; v0 += kAccThreads * kGreedyBatch) {
        if (v0 + kAccThreads * kGreedyBatch < nvec) load(nxt, v0 + kAccThreads * kGreedyBatch);
#pragma unroll
        for (int u = 0; u < kGreedyBatch; ++u) {
            const int vi = v0 + u * kAccThreads;
            if (vi < nvec) {
                float f[PV];
                Vec16<Tin>::unpack(cur[u], f);
#pragma unroll
                for (int e = 0; e < PV; ++e) {
                    const int i = a0 + vi * PV + e, k = e % kArgChains;
                    if (argmax_better(f[e], i, cv[k], ci[k])) { cv[k] = f[e]; ci[k] = i; }
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kGreedyBatch; ++u) cur[u] = nxt[u];
    }
    for (int i = a1 + tid; i < hi; i += kAccThreads) {
        const float x = Elem<Tin>::load(lg + i);
        if (argmax_better(x, i, cv[0], ci[0])) { cv[0] = x; ci[0] = i; }
    }
    float bv = cv[0];
    int bi = ci[0];
#pragma unroll
    for (int k = 1; k < kArgChains; ++k)
        if (argmax_better(cv[k], ci[k], bv, bi)) { bv = cv[k]; bi = ci[k]; }
    block_argmax(bv, bi);
    if (tid == 0) {
        p.pval[(long)row * p.n_chunks + c] = bv;
        p.pidx[(long)row * p.n_chunks + c] = bi;
    }
    if (!elect_last(p.counter, gridDim.x * gridDim.y)) return;

    // last CTA: every row's argmax from its chunk partials (a warp per row,
    // lanes over chunks), then the first-mismatch scan of every sequence, over
    // windows of W rows that hold whole sequences
    __shared__ int am[kAccThreads];
    const int R = p.B * p.T;
    const int W = (kAccThreads / p.T) * p.T;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    constexpr int kWarps = kAccThreads / 32;
    __shared__ float fin_v[kFinStaged];
    __shared__ int fin_i[kFinStaged];
    for (int r0 = 0; r0 < R; r0 += W) {
        const int nr = min(R - r0, W);
        const int np = nr * p.n_chunks;   // the window's partials, contiguous in pval / pidx
        if (np <= kFinStaged) {
            // all of them in flight at once (the grids are sized so that this
            // is the usual case), then a thread per row over its chunks
            for (int u = threadIdx.x; u < np; u += kAccThreads) {
                fin_v[u] = __ldcg(p.pval + (long)r0 * p.n_chunks + u);
                fin_i[u] = __ldcg(p.pidx + (long)r0 * p.n_chunks + u);
            }
            __syncthreads();
            for (int r = threadIdx.x; r < nr; r += kAccThreads) {
                float v = -INFINITY;
                int ix = INT_MAX;
                for (int k = 0; k < p.n_chunks; ++k) {
                    const float pv = fin_v[r * p.n_chunks + k];
                    const int pi = fin_i[r * p.n_chunks + k];
                    if (argmax_better(pv, pi, v, ix)) { v = pv; ix = pi; }
                }
                if (ix == INT_MAX) { set_fault(p.fault, FAULT_NAN_ROW); ix = 0; }
                am[r] = ix;
            }
        }
        // otherwise warp w takes rows w, w + 8, ... of the window, kFinRows at a
        // time with all their partial loads in flight together; lanes over the chunks
        for (int rb = 0; np > kFinStaged && rb < nr; rb += kWarps * kFinRows) {
            float v[kFinRows];
            int ix[kFinRows];
#pragma unroll
            for (int k = 0; k < kFinRows; ++k) { v[k] = -INFINITY; ix[k] = INT_MAX; }
            for (int k0 = lane; k0 < p.n_chunks; k0 += 32) {
#pragma unroll
                for (int k = 0; k < kFinRows; ++k) {
                    const int r = rb + warp + kWarps * k;
                    if (r < nr) {
                        const long o = (long)(r0 + r) * p.n_chunks + k0;
                        const float pv = __ldcg(p.pval + o);
                        const int pi = __ldcg(p.pidx + o);
                        if (argmax_better(pv, pi, v[k], ix[k])) { v[k] = pv; ix[k] = pi; }
                    }
                }
            }
#pragma unroll
            for (int k = 0; k < kFinRows; ++k) {
                warp_argmax(v[k], ix[k]);
                const int r = rb + warp + kWarps * k;
                if (lane == 0 && r < nr) {
                    if (ix[k] == INT_MAX) { set_fault(p.fault, FAULT_NAN_ROW); ix[k] = 0; }
                    am[r] = ix[k];
                }
            }
        }
        __syncthreads();
        const int b0 = r0 / p.T, nbw = min(p.B - b0, W / p.T);
        for (int bl = threadIdx.x; bl < nbw; bl += kAccThreads) {
            const int b = b0 + bl, rb = bl * p.T;
            if (p.parents) {
                // draft tree: node j is accepted when its parent is and its token
                // equals the target's pick after the parent; the deepest accepted
                // node (lowest index among equals) ends the committed path
                const int32_t *par = p.parents + (long)b * p.T, *tok = p.draft + (long)b * p.T;
                uint64_t acc = 1ull;  // bit j: node j accepted (the anchor always)
                int depth[kMaxTreeT];
                depth[0] = 0;
                int best = 0;
                for (int j = 1; j < p.T; ++j) {
                    const int pj = par[j];
                    if (pj < 0 || pj >= j) { set_fault(p.fault, FAULT_BAD_TREE); depth[j] = 0; continue; }
                    depth[j] = depth[pj] + 1;
                    if (((acc >> pj) & 1ull) && tok[j] == am[rb + pj]) {
                        acc |= 1ull << j;
                        if (depth[j] > depth[best]) best = j;
                    }
                }
                p.n_acc[b] = depth[best];
                p.corr[b] = am[rb + best];
                int32_t *path = p.path + (long)b * p.T;
                for (int k = depth[best]; k < p.T; ++k) path[k] = -1;
                for (int v = best; v != 0; v = par[v]) path[depth[v] - 1] = v;
            } else {
                int n = p.T - 1;
                for (int j = 0; j < p.T - 1; ++j) {
                    if (p.draft[(long)b * (p.T - 1) + j] != am[rb + j]) { n = j; break; }
                }
                p.n_acc[b] = n;
                p.corr[b] = am[rb + n];
            }
        }
        __syncthreads();
    }
}

// ----------------------------------------------------------------------------
// sampled acceptance, pass 1: per-row max and normaliser of softmax(l / tau);
// the last CTA of a row also tests that row's proposal, the last row finds
// the first rejection of every sequence
// ----------------------------------------------------------------------------
template <typename Tin, int NV>
__global__ void __launch_bounds__(kAccThreads) sample_stats_kernel(const SampleParams p) {
    grid_dependency_wait();
    const int c = blockIdx.x, row = blockIdx.y;
    const int lo = c * p.chunk, hi = min(p.V, lo + p.chunk);
    const Tin *lg = static_cast<const Tin *>(p.logits) + (long)row * p.V;
    const float it = p.inv_tau;
    ChunkRegs<Tin, NV> cr;
    cr.load(lg, lo, hi, -INFINITY);
    float m = -INFINITY;
#pragma unroll
    for (int v = 0; v < NV; ++v)
#pragma unroll
        for (int e = 0; e < ChunkRegs<Tin, NV>::PV; ++e) m = fmaxf(m, cr.x[v][e] * it);
    for (int i = lo + (int)threadIdx.x; i < cr.a0; i += kAccThreads) m = fmaxf(m, Elem<Tin>::load(lg + i) * it);
    for (int i = cr.a1 + (int)threadIdx.x; i < hi; i += kAccThreads) m = fmaxf(m, Elem<Tin>::load(lg + i) * it);
    m = block_max(m);
    double z = 0.0;
    if (m != -INFINITY) {
        float zf = 0.f;
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            float zv = 0.f;
#pragma unroll
            for (int e = 0; e < ChunkRegs<Tin, NV>::PV; ++e) zv += expf(cr.x[v][e] * it - m);  // fill -inf -> 0
            zf += zv;
        }
        z = zf;
        for (int i = lo + (int)threadIdx.x; i < cr.a0; i += kAccThreads) z += expf(Elem<Tin>::load(lg + i) * it - m);
        for (int i = cr.a1 + (int)threadIdx.x; i < hi; i += kAccThreads) z += expf(Elem<Tin>::load(lg + i) * it - m);
    }
    z = block_sum<double>(z);
    if (threadIdx.x == 0) {
        p.pm[(long)row * p.n_chunks + c] = m;
        p.pz[(long)row * p.n_chunks + c] = (float)z;
        // the CTA whose chunk holds this row's proposal records its logit and q
        const int b = row / p.T, j = row % p.T;
        if (j < p.T - 1) {
            const int d = p.draft[(long)b * (p.T - 1) + j];
            if (d >= lo && d < hi)
                p.row_stats[row] = make_float2(Elem<Tin>::load(lg + d), __ldg(p.q + (long)row * p.V + d));
        }
    }
    if (!elect_last(p.counters, gridDim.x * gridDim.y)) return;

    // last CTA: every row's max M and normaliser Z (a warp per row, lanes over
    // chunks) and the test of its proposal (rows 0..T-2): accept iff
    // u * q(d) < p(d); then the first rejection of every sequence, over windows
    // of W rows that hold whole sequences
    __shared__ int acc_s[kAccThreads];
    __shared__ float2 mz_s[kAccThreads];
    const int R = p.B * p.T;
    const int W = (kAccThreads / p.T) * p.T;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    constexpr int kWarps = kAccThreads / 32;
    // the accept test of row gr with its max M and normaliser Z
    auto test_row = [&](int gr, float Mr, double Zr) {
        const int b = gr / p.T, j = gr % p.T;
        int accept = 0;
        if (j < p.T - 1) {
            const int d = p.draft[(long)b * (p.T - 1) + j];
            if (d >= 0 && d < p.V) {
                const float2 lq = __ldcg(p.row_stats + gr);
                const double pd = (double)expf(lq.x * it - Mr) / Zr;
                const double u = (double)philox_uniform(p.seed, (uint32_t)j, (uint32_t)b, 0u, p.offset);
                accept = u * (double)lq.y < pd ? 1 : 0;
            } else {
                set_fault(p.fault, FAULT_BAD_DRAFT_ID);
            }
        }
        return accept;
    };
    __shared__ float fin_m[kFinStaged], fin_z[kFinStaged];
    for (int r0 = 0; r0 < R; r0 += W) {
        const int nr = min(R - r0, W);
        const int np = nr * p.n_chunks;   // the window's partials, contiguous in pm / pz
        if (np <= kFinStaged) {
            // all of them in flight at once, then a thread per row
            for (int u = threadIdx.x; u < np; u += kAccThreads) {
                fin_m[u] = __ldcg(p.pm + (long)r0 * p.n_chunks + u);
                fin_z[u] = __ldcg(p.pz + (long)r0 * p.n_chunks + u);
            }
            __syncthreads();
            for (int r = threadIdx.x; r < nr; r += kAccThreads) {
                float Mr = -INFINITY;
                for (int k = 0; k < p.n_chunks; ++k) Mr = fmaxf(Mr, fin_m[r * p.n_chunks + k]);
                double Zr = 0.0;
                for (int k = 0; k < p.n_chunks; ++k) {
                    const float mk = fin_m[r * p.n_chunks + k];
                    if (mk != -INFINITY) Zr += (double)fin_z[r * p.n_chunks + k] * (double)expf(mk - Mr);
                }
                acc_s[r] = test_row(r0 + r, Mr, Zr);
                mz_s[r] = make_float2(Mr, (float)Zr);
            }
        }
        // otherwise warp w takes rows w, w + 8, ... of the window, kFinRows at a
        // time with the loads of all of them in flight together; lanes over the chunks
        for (int rb = 0; np > kFinStaged && rb < nr; rb += kWarps * kFinRows) {
            float M[kFinRows];
            double Z[kFinRows];
#pragma unroll
            for (int k = 0; k < kFinRows; ++k) { M[k] = -INFINITY; Z[k] = 0.0; }
            for (int k0 = lane; k0 < p.n_chunks; k0 += 32) {
#pragma unroll
                for (int k = 0; k < kFinRows; ++k) {
                    const int r = rb + warp + kWarps * k;
                    if (r < nr) M[k] = fmaxf(M[k], __ldcg(p.pm + (long)(r0 + r) * p.n_chunks + k0));
                }
            }
#pragma unroll
            for (int k = 0; k < kFinRows; ++k)
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) M[k] = fmaxf(M[k], __shfl_xor_sync(0xffffffffu, M[k], o));
            for (int k0 = lane; k0 < p.n_chunks; k0 += 32) {
#pragma unroll
                for (int k = 0; k < kFinRows; ++k) {
                    const int r = rb + warp + kWarps * k;
                    if (r < nr) {
                        const long o = (long)(r0 + r) * p.n_chunks + k0;
                        const float mk = __ldcg(p.pm + o);
                        const float zk = __ldcg(p.pz + o);
                        if (mk != -INFINITY) Z[k] += (double)zk * (double)expf(mk - M[k]);
                    }
                }
            }
#pragma unroll
            for (int k = 0; k < kFinRows; ++k) Z[k] = warp_sum(Z[k]);
            if (lane == 0) {
#pragma unroll
                for (int k = 0; k < kFinRows; ++k) {
                    const int r = rb + warp + kWarps * k;
                    if (r >= nr) continue;
                    acc_s[r] = test_row(r0 + r, M[k], Z[k]);
                    mz_s[r] = make_float2(M[k], (float)Z[k]);
                }
            }
        }
        __syncthreads();
        const int b0 = r0 / p.T, nbw = min(p.B - b0, W / p.T);
        for (int bl = threadIdx.x; bl < nbw; bl += kAccThreads) {
            const int b = b0 + bl;
            int n = p.T - 1;
            for (int j = 0; j < p.T - 1; ++j)
                if (!acc_s[bl * p.T + j]) { n = j; break; }
            const float2 st = mz_s[bl * p.T + n];
            p.n_acc[b] = n;
            p.state[b] = make_float4(__int_as_float(n), st.x, st.y, 0.f);
        }
        __syncthreads();
    }
}

// ----------------------------------------------------------------------------
// sampled acceptance, pass 2: on the row that decides the next token, chunk
// sums of the residual r = max(p - q, 0) and of p; the last CTA of the
// sequence picks the chunk where u' * S falls and searches inside it
// ----------------------------------------------------------------------------
// the weight of element i (the same fp32 arithmetic wherever it is used)
__device__ __forceinline__ float residual_or_p(float x, float it, float M, float Z, float qi, bool residual) {
    const float pi = expf(x * it - M) / Z;
    if (!residual) return pi;
    const float r = pi - qi;
    return r > 0.f ? r : 0.f;
}

template <typename Tin, int NV>
__global__ void __launch_bounds__(kAccThreads) sample_draw_kernel(const SampleParams p) {
    grid_dependency_wait();
    const int c = blockIdx.x, b = blockIdx.y;
    const float4 st = p.state[b];
    const int n = __float_as_int(st.x);
    const float M = st.y, Z = st.z;
    const bool rejected = n < p.T - 1;
    const long row = (long)b * p.T + n;
    const Tin *lg = static_cast<const Tin *>(p.logits) + row * p.V;
    const float *qn = p.q + row * p.V;
    const float it = p.inv_tau;
    const int lo = c * p.draw_chunk, hi = min(p.V, lo + p.draw_chunk);
    ChunkRegs<Tin, NV> cr;
    cr.load(lg, lo, hi, -INFINITY);
    // per-thread sums in fp32 (at most a few dozen terms), the CTA total in fp64
    float srf = 0.f, spf = 0.f;
    constexpr int PV = ChunkRegs<Tin, NV>::PV;
    float qv[NV][PV];
#pragma unroll
    for (int v = 0; v < NV; ++v)
#pragma unroll
        for (int e = 0; e < PV; ++e) qv[v][e] = (rejected && cr.valid(v)) ? __ldg(qn + cr.index(v, e)) : 0.f;
#pragma unroll
    for (int v = 0; v < NV; ++v) {
        if (!cr.valid(v)) break;
        float sv = 0.f, rv = 0.f;
#pragma unroll
        for (int e = 0; e < PV; ++e) {
            const float pi = expf(cr.x[v][e] * it - M) / Z;
            sv += pi;
            const float r = pi - qv[v][e];
            rv += r > 0.f ? r : 0.f;
        }
        spf += sv;
        srf += rv;
    }
    auto scalar = [&](int i) {
        const float pi = expf(Elem<Tin>::load(lg + i) * it - M) / Z;
        spf += pi;
        if (rejected) { const float r = pi - __ldg(qn + i); srf += r > 0.f ? r : 0.f; }
    };
    for (int i = lo + (int)threadIdx.x; i < cr.a0; i += kAccThreads) scalar(i);
    for (int i = cr.a1 + (int)threadIdx.x; i < hi; i += kAccThreads) scalar(i);
    const double sr = block_sum<double>(rejected ? (double)srf : 0.0);
    const double sp = block_sum<double>((double)spf);
    if (threadIdx.x == 0) {
        p.rs[(long)b * p.n_draw_chunks + c] = sr;
        p.ps[(long)b * p.n_draw_chunks + c] = sp;
    }
    if (!elect_last(p.row_counter + b, gridDim.x)) return;

    // last CTA of sequence b: which chunk holds u' * S.  The chunk sums are
    // first staged in shared memory by the whole CTA (one round trip).
    __shared__ int sel_chunk, sel_res;
    __shared__ double sel_base, sel_x;
    __shared__ double s_rs[kDrawChunksStaged], s_ps[kDrawChunksStaged];
    const bool staged = p.n_draw_chunks <= kDrawChunksStaged;
    if (staged)
        for (int k = threadIdx.x; k < p.n_draw_chunks; k += kAccThreads) {
            s_rs[k] = __ldcg(p.rs + (long)b * p.n_draw_chunks + k);
            s_ps[k] = __ldcg(p.ps + (long)b * p.n_draw_chunks + k);
        }
    __syncthreads();
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        double Sr = 0.0, Sp = 0.0;
        for (int k = lane; k < p.n_draw_chunks; k += 32) {
            Sr += staged ? s_rs[k] : __ldcg(p.rs + (long)b * p.n_draw_chunks + k);
            Sp += staged ? s_ps[k] : __ldcg(p.ps + (long)b * p.n_draw_chunks + k);
        }
        Sr = warp_sum(Sr);
        Sp = warp_sum(Sp);
        const bool use_r = rejected && Sr > 0.0;
        const double *gcs = (use_r ? p.rs : p.ps) + (long)b * p.n_draw_chunks;
        auto cs_at = [&](int k) { return staged ? (use_r ? s_rs[k] : s_ps[k]) : __ldcg(gcs + k); };
        const double S = use_r ? Sr : Sp;
        const double x = (double)philox_uniform(p.seed, (uint32_t)n, (uint32_t)b, 1u, p.offset) * S;
        // inclusive prefix over the chunk sums, 32 chunks at a time
        double carry = 0.0;
        int found = -1, last_pos = -1;
        double found_base = 0.0;
        for (int k0 = 0; k0 < p.n_draw_chunks && found < 0; k0 += 32) {
            const int k = k0 + lane;
            const double v = k < p.n_draw_chunks ? cs_at(k) : 0.0;
            double incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const double y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            const unsigned pos = __ballot_sync(0xffffffffu, k < p.n_draw_chunks && v > 0.0);
            if (pos) last_pos = k0 + 31 - __clz((int)pos);
            const unsigned hit = __ballot_sync(0xffffffffu, k < p.n_draw_chunks && carry + incl > x);
            if (hit) {
                const int l = __ffs((int)hit) - 1;
                found = k0 + l;
                found_base = carry + __shfl_sync(0xffffffffu, incl - v, l);
            }
            carry += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (found < 0) {  // x reached the total through rounding: the last non-empty chunk
            found = last_pos < 0 ? 0 : last_pos;
            double base = 0.0;
            for (int k = lane; k < found; k += 32) base += cs_at(k);
            found_base = warp_sum(base);
        }
        if (lane == 0) { sel_chunk = found; sel_base = found_base; sel_x = x; sel_res = use_r ? 1 : 0; }
    }
    __syncthreads();

    // inside the chunk: thread t owns a contiguous run of elements; runs are
    // combined by an exclusive scan over the threads, the owner of the
    // crossing then walks its run
    constexpr int kRun = 16;
    static_assert(kRun * kAccThreads >= kDrawChunkMax, "the search covers a whole draw chunk");
    const int clo = sel_chunk * p.draw_chunk, chi = min(p.V, clo + p.draw_chunk);
    const int per = (chi - clo + kAccThreads - 1) / kAccThreads;  // <= kRun (draw chunk <= kDrawChunkMax)
    const int tlo = min(chi, clo + (int)threadIdx.x * per), thi = min(chi, tlo + per);
    const bool res = sel_res != 0;
    float w[kRun], xin[kRun], qin[kRun];
#pragma unroll
    for (int e = 0; e < kRun; ++e) {
        const int i = tlo + e;
        xin[e] = i < thi ? Elem<Tin>::load(lg + i) : 0.f;
        qin[e] = (i < thi && res) ? __ldg(qn + i) : 0.f;
    }
    float runf = 0.f;
#pragma unroll
    for (int e = 0; e < kRun; ++e) {
        w[e] = tlo + e < thi ? residual_or_p(xin[e], it, M, Z, qin[e], res) : 0.f;
        runf += w[e];
    }
    // exclusive prefix of the runs over the threads: warp scans, then warp totals
    const double run = (double)runf;
    __shared__ double wtot[kAccThreads / 32];
    __shared__ int s_id, s_lastpos;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    double incl = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const double y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) wtot[wid] = incl;
    if (threadIdx.x == 0) { s_id = INT_MAX; s_lastpos = -1; }
    __syncthreads();
    double before = 0.0;
    for (int k = 0; k < wid; ++k) before += wtot[k];
    double acc = sel_base + before + (incl - run);
    int last_here = -1;
#pragma unroll
    for (int e = 0; e < kRun; ++e) {
        if (tlo + e >= thi) break;
        if (w[e] > 0.f) last_here = tlo + e;
        const double nxt = acc + (double)w[e];
        if (nxt > sel_x && acc <= sel_x) { atomicMin(&s_id, tlo + e); break; }
        acc = nxt;
    }
    if (last_here >= 0) atomicMax(&s_lastpos, last_here);
    __syncthreads();
    if (threadIdx.x == 0) {
        int id = s_id;
        if (id == INT_MAX) id = s_lastpos >= 0 ? s_lastpos : clo;  // rounding: last positive weight
        p.next_id[b] = id;
    }
}

}  // namespace

// vectors per thread needed to hold one chunk in registers
template <typename Tin> int vec_per_thread(int chunk) {
    const int v = (chunk + Elem<Tin>::kPerVec * kAccThreads - 1) / (Elem<Tin>::kPerVec * kAccThreads);
    return v <= 1 ? 1 : v <= 2 ? 2 : v <= 4 ? 4 : 8;
}

// launch with programmatic stream serialization (overlaps the previous kernel's tail)
template <typename P>
cudaError_t launch_pdl(void (*kern)(const P), dim3 grid, cudaStream_t st, const P &p) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kAccThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

#define SDV_DISPATCH_NV(KERNEL, TIN, NVV, GRID, ST, P, ERR)                     \
    do {                                                                       \
        switch (NVV) {                                                         \
            case 1: ERR = launch_pdl(KERNEL<TIN, 1>, GRID, ST, P); break;      \
            case 2: ERR = launch_pdl(KERNEL<TIN, 2>, GRID, ST, P); break;      \
            case 4: ERR = launch_pdl(KERNEL<TIN, 4>, GRID, ST, P); break;      \
            default: ERR = launch_pdl(KERNEL<TIN, 8>, GRID, ST, P); break;     \
        }                                                                      \
    } while (0)

cudaError_t launch_accept_greedy(const GreedyParams &p, cudaStream_t st) {
    dim3 grid(p.n_chunks, p.B * p.T);
    cudaError_t e;
    if (p.dt == SD_BF16) e = launch_pdl(greedy_kernel<__nv_bfloat16>, grid, st, p);
    else e = launch_pdl(greedy_kernel<float>, grid, st, p);
    return e;
}

cudaError_t launch_accept_sample(const SampleParams &p, cudaStream_t st) {
    dim3 g1(p.n_chunks, p.B * p.T), g2(p.n_draw_chunks, p.B);
    cudaError_t e;
    if (p.dt == SD_BF16) {
        SDV_DISPATCH_NV(sample_stats_kernel, __nv_bfloat16, vec_per_thread<__nv_bfloat16>(p.chunk), g1, st, p, e);
        if (e != cudaSuccess) return e;
        SDV_DISPATCH_NV(sample_draw_kernel, __nv_bfloat16, vec_per_thread<__nv_bfloat16>(p.draw_chunk), g2, st, p, e);
    } else {
        SDV_DISPATCH_NV(sample_stats_kernel, float, vec_per_thread<float>(p.chunk), g1, st, p, e);
        if (e != cudaSuccess) return e;
        SDV_DISPATCH_NV(sample_draw_kernel, float, vec_per_thread<float>(p.draw_chunk), g2, st, p, e);
    }
    return e;
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
