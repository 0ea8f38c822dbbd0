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
// reduces across warps (shuffles, then shared memory) into one partial.  One
// grid-wide ticket counter elects the CTA that finishes last; that CTA
// combines every row's partials (the greedy finisher stages them in shared
// memory, the sampled one takes a warp per row) and runs the per-sequence
// scan.  The sampled rule's second kernel works on the row that decides each
// sequence's next token; a ticket counter per sequence elects the CTA that
// picks the chunk and then the element.  The CTA that takes a counter's last
// ticket returns it to zero, so a zero-filled workspace stays reusable.  No
// CTA ever waits for another.  Sums over a whole vocabulary are carried as
// float-float values (two fp32 words), not in the slow fp64 pipe.
#include "tcgen05.cuh"

#include <atomic>
#include <float.h>
#include <limits.h>
#include <math.h>

namespace sdv {

namespace {

constexpr int kAccThreads = 256;
constexpr int kGreedyBatch = 4;   // 16-byte vectors per thread per batch of the pass-1 streams
constexpr int kFinRows = 4;       // rows per warp whose chunk partials a finisher loads together
constexpr int kFinStaged = 1024;  // chunk partials the greedy finisher stages in shared memory at once

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


// Programmatic dependent launch: the kernel may start while the previous one in
// the stream drains; wait here until its results are visible.
__device__ __forceinline__ void grid_dependency_wait() {
#if __CUDA_ARCH__ >= 900
    asm volatile("griddepcontrol.wait;" ::: "memory");
#endif
}
// lets the next kernel in the stream launch (it still waits for this one's
// results in its own grid_dependency_wait)
__device__ __forceinline__ void grid_launch_dependents() {
#if __CUDA_ARCH__ >= 900
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
#endif
}

// Last-CTA election on `counter` among `total` arrivals: true in every thread of
// the CTA that arrived last, which also returns the counter to zero (seen by
// the next launch once this grid has ended).  Only thread 0 of a CTA writes
// that CTA's partial results; its ticket is an acquire-release atomic at GPU
// scope, so the partials are released with it, and the last CTA's acquire
// (then the barrier) orders its threads' reads of everyone's partials after it.
__device__ __forceinline__ bool elect_last(unsigned int *counter, unsigned int total) {
    __shared__ bool is_last;
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned int ticket;
        asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(ticket) : "l"(counter) : "memory");
        is_last = ticket == total - 1;
        if (is_last) *counter = 0u;
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
    // the largest ordered value of the vector (NaN loses; -inf if all are NaN)
    __device__ __forceinline__ static float max(const uint4 &u) {
        return fmaxf(fmaxf(__uint_as_float(u.x), __uint_as_float(u.y)),
                     fmaxf(__uint_as_float(u.z), __uint_as_float(u.w)));
    }
};
template <> struct Vec16<__nv_bfloat16> {
    static constexpr int PV = 8;
    __device__ __forceinline__ static void unpack(const uint4 &u, float (&f)[8]) { unpack_bf16x8(u, f); }
    // the largest ordered value of the vector, from packed bf16x2 maxima (exact:
    // a maximum picks one of its inputs; NaN loses to a number)
    __device__ __forceinline__ static float max(const uint4 &u) {
        const __nv_bfloat162 a = __hmax2(*reinterpret_cast<const __nv_bfloat162 *>(&u.x),
                                         *reinterpret_cast<const __nv_bfloat162 *>(&u.y));
        const __nv_bfloat162 b = __hmax2(*reinterpret_cast<const __nv_bfloat162 *>(&u.z),
                                         *reinterpret_cast<const __nv_bfloat162 *>(&u.w));
        const __nv_bfloat162 c = __hmax2(a, b);
        return fmaxf(__low2float(c), __high2float(c));
    }
};

// CTA (c, row) streams chunk c of one row: the unaligned head and tail
// element by element, the 16-byte-aligned body in batches of kGreedyBatch
// vectors per thread, the next batch in flight while this one is reduced
// at most 3 CTAs per SM are resident by design (the grid is one such wave)
template <typename Tin>
__global__ void __launch_bounds__(kAccThreads, 3) greedy_kernel(const GreedyParams p) {
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
    // the first finisher window's proposals, loaded by every CTA while its
    // stream runs (only the last CTA uses them: at most 1 KB, from L2)
    const int per_seq = p.parents ? p.T : p.T - 1;
    const int R = p.B * p.T;
    const int W = (kAccThreads / p.T) * p.T;
    const int n_pre = min(R, W) / p.T * per_seq;
    int pre_tok = 0, pre_par = 0;
    if (tid < n_pre) {
        pre_tok = p.draft[tid];
        if (p.parents) pre_par = p.parents[tid];
    }
    // the thread's (value, index) argmax so far
    float cv = -INFINITY;
    int ci = INT_MAX;
    for (int i = lo + tid; i < a0; i += kAccThreads) {
        const float x = Elem<Tin>::load(lg + i);
        if (argmax_better(x, i, cv, ci)) { cv = x; ci = i; }
    }
    // a ring of three batches of kGreedyBatch vectors: while one is reduced
    // the next two are in flight (12 vectors, 192 bytes per thread)
    uint4 r0[kGreedyBatch], r1[kGreedyBatch], r2[kGreedyBatch];
    constexpr int kStep = kAccThreads * kGreedyBatch;   // vectors per batch of the CTA
    auto load = [&](uint4 (&d)[kGreedyBatch], int v0) {
#pragma unroll
        for (int u = 0; u < kGreedyBatch; ++u) {
            const int vi = v0 + u * kAccThreads;
            d[u] = vi < nvec ? ld_stream_u4(vp + vi) : make_uint4(0u, 0u, 0u, 0u);
        }
    };
    // each vector: its largest value first (packed maxima), compared with the
    // running best; only a vector that beats it (rare past the start) is
    // searched for the lowest index holding that value.  A thread meets its
    // indices in increasing order, so an equal value met later never wins;
    // the first ordered value (even -inf) is taken, and NaN never is.
    auto reduce = [&](const uint4 (&d)[kGreedyBatch], int v0) {
#pragma unroll
        for (int u = 0; u < kGreedyBatch; ++u) {
            const int vi = v0 + u * kAccThreads;
            if (vi < nvec) {
                const float vmax = Vec16<Tin>::max(d[u]);
                if (vmax > cv || (vmax == cv && ci == INT_MAX)) {
                    float f[PV];
                    Vec16<Tin>::unpack(d[u], f);
                    int e0 = PV - 1;
#pragma unroll
                    for (int e = PV - 1; e >= 0; --e)
                        if (f[e] == vmax) e0 = e;
                    cv = vmax;
                    ci = a0 + vi * PV + e0;
                }
            }
        }
    };
    load(r0, tid);
    load(r1, tid + kStep);
    for (int v0 = tid; v0 < nvec; v0 += 3 * kStep) {
        load(r2, v0 + 2 * kStep);
        reduce(r0, v0);
        if (v0 + kStep >= nvec) break;
        load(r0, v0 + 3 * kStep);
        reduce(r1, v0 + kStep);
        if (v0 + 2 * kStep >= nvec) break;
        load(r1, v0 + 4 * kStep);
        reduce(r2, v0 + 2 * kStep);
    }
    for (int i = a1 + tid; i < hi; i += kAccThreads) {
        const float x = Elem<Tin>::load(lg + i);
        if (argmax_better(x, i, cv, ci)) { cv = x; ci = i; }
    }
    float bv = cv;
    int bi = ci;
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
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    constexpr int kWarps = kAccThreads / 32;
    __shared__ float fin_v[kFinStaged];
    __shared__ int fin_i[kFinStaged];
    // the window's proposals (chain: T-1 drafts per sequence; tree: T node
    // tokens and T parents), loaded together with the partials
    __shared__ int s_tok[kAccThreads], s_par[kAccThreads];
    for (int r0 = 0; r0 < R; r0 += W) {
        const int nr = min(R - r0, W);
        const int np = nr * p.n_chunks;   // the window's partials, contiguous in pval / pidx
        if (r0 == 0) {
            if (tid < n_pre) { s_tok[tid] = pre_tok; s_par[tid] = pre_par; }
        } else {
            const int b0w = r0 / p.T, nseq = nr / p.T;
            for (int u = threadIdx.x; u < nseq * per_seq; u += kAccThreads) {
                s_tok[u] = p.draft[(long)b0w * per_seq + u];
                if (p.parents) s_par[u] = p.parents[(long)b0w * p.T + u];
            }
        }
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
        // a warp per sequence
        const int b0 = r0 / p.T, nbw = min(p.B - b0, W / p.T);
        for (int bl = warp; bl < nbw; bl += kWarps) {
            const int b = b0 + bl, rb = bl * p.T;
            if (p.parents) {
                // draft tree: node j is accepted when its parent is and its token
                // equals the target's pick after the parent; the deepest accepted
                // node (lowest index among equals) ends the committed path.  Lane
                // l holds nodes l and l + 32.  Pointer jumping over the parent
                // links: each node carries the segment of its root path from
                // itself up to (not including) node A -- all matched, its length,
                // its node set -- and joins A's segment to its own until A is the
                // root (six rounds cover 63 links)
                const int *par = s_par + bl * p.T, *tok = s_tok + bl * p.T;
                int A[2], okd[2];        // okd: bit 16 all matched, low bits the length
                uint64_t M[2];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int j = lane + 32 * h;
                    A[h] = 0; okd[h] = 1 << 16; M[h] = 0ull;   // the root (and nodes past T)
                    if (j >= 1 && j < p.T) {
                        const int pj = par[j];
                        M[h] = 1ull << j;
                        if (pj < 0 || pj >= j) { set_fault(p.fault, FAULT_BAD_TREE); okd[h] = 0; }
                        else { A[h] = pj; okd[h] = ((tok[j] == am[rb + pj]) ? 1 << 16 : 0) | 1; }
                    }
                }
#pragma unroll 1
                for (int round = 0; round < 6; ++round) {
                    int nA[2], nokd[2];
                    uint64_t nM[2];
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int src = A[h] & 31;
                        const bool hi = A[h] >= 32;
                        const int a0 = __shfl_sync(0xffffffffu, A[0], src), a1 = __shfl_sync(0xffffffffu, A[1], src);
                        const int o0 = __shfl_sync(0xffffffffu, okd[0], src), o1 = __shfl_sync(0xffffffffu, okd[1], src);
                        const uint64_t m0 = __shfl_sync(0xffffffffu, M[0], src), m1 = __shfl_sync(0xffffffffu, M[1], src);
                        const int oa = hi ? o1 : o0;
                        nA[h] = hi ? a1 : a0;
                        nokd[h] = (okd[h] & oa & (1 << 16)) | ((okd[h] & 0xffff) + (oa & 0xffff));
                        nM[h] = M[h] | (hi ? m1 : m0);
                    }
#pragma unroll
                    for (int h = 0; h < 2; ++h) { A[h] = nA[h]; okd[h] = nokd[h]; M[h] = nM[h]; }
                }
                // deepest accepted node, lowest index among equals
                int key = -1;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int j = lane + 32 * h;
                    if (j < p.T && (okd[h] >> 16)) key = max(key, ((okd[h] & 0xffff) << 7) | (127 - j));
                }
                key = __reduce_max_sync(0xffffffffu, key);
                const int best = 127 - (key & 127), dbest = key >> 7;
                const uint64_t mb0 = __shfl_sync(0xffffffffu, M[0], best & 31);
                const uint64_t mb1 = __shfl_sync(0xffffffffu, M[1], best & 31);
                const uint64_t mbest = best >= 32 ? mb1 : mb0;   // the nodes of the committed path
                if (lane == 0) {
                    p.n_acc[b] = dbest;
                    p.corr[b] = am[rb + best];
                }
                int32_t *path = p.path + (long)b * p.T;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int j = lane + 32 * h;
                    if (j < p.T && j >= dbest) path[j] = -1;
                    if (j >= 1 && j < p.T && ((mbest >> j) & 1ull)) path[(okd[h] & 0xffff) - 1] = j;
                }
            } else {
                // chain: lane j tests proposal j (T - 1 <= 15); the first
                // mismatch is the lowest set bit of the warp's ballot
                const bool miss = lane < p.T - 1 && s_tok[bl * (p.T - 1) + lane] != am[rb + lane];
                const unsigned int m = __ballot_sync(0xffffffffu, miss);
                if (lane == 0) {
                    const int n = m ? __ffs(m) - 1 : p.T - 1;
                    p.n_acc[b] = n;
                    p.corr[b] = am[rb + n];
                }
            }
        }
        __syncthreads();
    }
}

// ----------------------------------------------------------------------------
// float-float sums: a value held as hi + lo, two fp32 words with hi the fp32
// rounding of the pair, added with Knuth's error-free two-sum; about 48
// significant bits, enough for sums over a whole vocabulary, without the slow
// fp64 pipe
// ----------------------------------------------------------------------------
struct FF {
    float hi, lo;
};
__device__ __forceinline__ FF ff_norm(float s, float e) {   // s + e with |e| small next to |s|
    const float h = s + e;
    return FF{h, e - (h - s)};
}
__device__ __forceinline__ FF ff_add(FF a, FF b) {
    const float s = a.hi + b.hi;
    const float bv = s - a.hi;
    const float e = ((a.hi - (s - bv)) + (b.hi - bv)) + (a.lo + b.lo);
    return ff_norm(s, e);
}
__device__ __forceinline__ FF ff_add(FF a, float b) { return ff_add(a, FF{b, 0.f}); }
// a * f, f a plain fp32 factor
__device__ __forceinline__ FF ff_scale(FF a, float f) {
    const float p = a.hi * f;
    return ff_norm(p, fmaf(a.hi, f, -p) + a.lo * f);
}
// a * b
__device__ __forceinline__ FF ff_mul(FF a, FF b) {
    const float p = a.hi * b.hi;
    return ff_norm(p, fmaf(a.hi, b.hi, -p) + (a.hi * b.lo + a.lo * b.hi));
}
// the exact product of two fp32 numbers
__device__ __forceinline__ FF ff_prod(float a, float b) {
    const float p = a * b;
    return FF{p, fmaf(a, b, -p)};
}
__device__ __forceinline__ bool ff_lt(FF a, FF b) { return a.hi < b.hi || (a.hi == b.hi && a.lo < b.lo); }
__device__ __forceinline__ bool ff_gt0(FF a) { return a.hi > 0.f || (a.hi == 0.f && a.lo > 0.f); }
__device__ __forceinline__ FF ff_shfl_xor(FF a, int o) {
    return FF{__shfl_xor_sync(0xffffffffu, a.hi, o), __shfl_xor_sync(0xffffffffu, a.lo, o)};
}
__device__ __forceinline__ FF ff_shfl_up(FF a, int o) {
    return FF{__shfl_up_sync(0xffffffffu, a.hi, o), __shfl_up_sync(0xffffffffu, a.lo, o)};
}
__device__ __forceinline__ FF ff_warp_sum(FF x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = ff_add(x, ff_shfl_xor(x, o));
    return x;
}
// block-wide sum; result valid in every thread
__device__ __forceinline__ FF ff_block_sum(FF x) {
    __shared__ FF sh[kAccThreads / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    x = ff_warp_sum(x);
    __syncthreads();
    if (lane == 0) sh[warp] = x;
    __syncthreads();
    FF t = sh[0];
    for (int w = 1; w < kAccThreads / 32; ++w) t = ff_add(t, sh[w]);
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

// ----------------------------------------------------------------------------
// sampled acceptance, pass 1: per-row max and normaliser of softmax(l / tau);
// the last CTA tests every row's proposal and finds the first rejection of
// every sequence
// ----------------------------------------------------------------------------
template <typename Tin, int NV>
__global__ void __launch_bounds__(kAccThreads) sample_stats_kernel(const SampleParams p) {
    grid_dependency_wait();
    // the draw kernel may take its place on the SMs now and wait there
    grid_launch_dependents();
    const int c = blockIdx.x, row = blockIdx.y;
    const int lo = c * p.chunk, hi = min(p.V, lo + p.chunk);
    const Tin *lg = static_cast<const Tin *>(p.logits) + (long)row * p.V;
    const float it = p.inv_tau;
    ChunkRegs<Tin, NV> cr;
    cr.load(lg, lo, hi, -INFINITY);
    // the chunk's max, then its sum of exp against it (float-float)
    float m = -INFINITY;
#pragma unroll
    for (int v = 0; v < NV; ++v)
#pragma unroll
        for (int e = 0; e < ChunkRegs<Tin, NV>::PV; ++e) m = fmaxf(m, cr.x[v][e] * it);
    for (int i = lo + (int)threadIdx.x; i < cr.a0; i += kAccThreads) m = fmaxf(m, Elem<Tin>::load(lg + i) * it);
    for (int i = cr.a1 + (int)threadIdx.x; i < hi; i += kAccThreads) m = fmaxf(m, Elem<Tin>::load(lg + i) * it);
    m = block_max(m);
    FF z = FF{0.f, 0.f};
    if (m != -INFINITY) {
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            float zv = 0.f;
#pragma unroll
            for (int e = 0; e < ChunkRegs<Tin, NV>::PV; ++e) zv += expf(cr.x[v][e] * it - m);  // fill -inf -> 0
            z = ff_add(z, zv);
        }
        for (int i = lo + (int)threadIdx.x; i < cr.a0; i += kAccThreads) z = ff_add(z, expf(Elem<Tin>::load(lg + i) * it - m));
        for (int i = cr.a1 + (int)threadIdx.x; i < hi; i += kAccThreads) z = ff_add(z, expf(Elem<Tin>::load(lg + i) * it - m));
    }
    z = ff_block_sum(z);
    if (threadIdx.x == 0) {
        p.pm[(long)row * p.n_chunks + c] = m;
        p.pz[(long)row * p.n_chunks + c] = make_float2(z.hi, z.lo);
        // the CTA whose chunk holds this row's proposal records its logit and q
        const int b = row / p.T, j = row % p.T;
        if (j < p.T - 1) {
            const int d = p.draft[(long)b * (p.T - 1) + j];
            if (d >= lo && d < hi)
                p.row_stats[row] = make_float2(Elem<Tin>::load(lg + d), __ldg(p.q + (long)row * p.V + d));
        }
    }
    if (!elect_last(p.counters, gridDim.x * gridDim.y)) return;

    // last CTA: every row's max M and normaliser Z (from the chunk partials,
    // below) and the test of its proposal (rows 0..T-2): accept iff
    // u * q(d) < p(d) = exp(l(d) / tau - M) / Z, taken as u * q(d) * Z < exp(..)
    // with the product exact; then the first rejection of every sequence, over
    // windows of W rows that hold whole sequences
    __shared__ int acc_s[kAccThreads];
    __shared__ float2 mz_s[kAccThreads];
    const int R = p.B * p.T;
    const int W = (kAccThreads / p.T) * p.T;
    auto test_row = [&](int gr, float Mr, FF Zr, float u) {
        const int b = gr / p.T, j = gr % p.T;
        int accept = 0;
        if (j < p.T - 1) {
            const int d = p.draft[(long)b * (p.T - 1) + j];
            if (d >= 0 && d < p.V) {
                const float2 lq = __ldcg(p.row_stats + gr);
                const float ed = expf(lq.x * it - Mr);
                accept = ff_lt(ff_mul(ff_prod(u, lq.y), Zr), FF{ed, 0.f}) ? 1 : 0;
            } else {
                set_fault(p.fault, FAULT_BAD_DRAFT_ID);
            }
        }
        return accept;
    };
    // the window's partials (contiguous in pm / pz) are staged kFinStaged at a
    // time with all their loads in flight: the row maxima by a thread per row,
    // then every partial rescaled to its row's maximum by a thread per
    // partial, then the rows' float-float sums by a thread per row
    __shared__ float fin_m[kFinStaged];
    __shared__ FF fin_z[kFinStaged];
    __shared__ float row_m[kAccThreads];
    __shared__ FF row_z[kAccThreads];
    for (int r0 = 0; r0 < R; r0 += W) {
        const int nr = min(R - r0, W);
        const int np = nr * p.n_chunks;
        for (int r = threadIdx.x; r < nr; r += kAccThreads) { row_m[r] = -INFINITY; row_z[r] = FF{0.f, 0.f}; }
        // this thread's row's uniform (row r0 + threadIdx.x), drawn while the loads below are in flight
        float u_own = 0.f;
        if ((int)threadIdx.x < nr) {
            const int gr = r0 + (int)threadIdx.x;
            u_own = philox_uniform(p.seed, (uint32_t)(gr % p.T), (uint32_t)(gr / p.T), 0u, p.offset);
        }
        for (int k0 = 0; k0 < np; k0 += kFinStaged) {
            const int nk = min(kFinStaged, np - k0);
            for (int u = threadIdx.x; u < nk; u += kAccThreads) {
                const long o = (long)r0 * p.n_chunks + k0 + u;
                fin_m[u] = __ldcg(p.pm + o);
                const float2 zk = __ldcg(p.pz + o);
                fin_z[u] = FF{zk.x, zk.y};
            }
            __syncthreads();
            // the rows' maxima over this part
            for (int r = threadIdx.x; r < nr; r += kAccThreads) {
                const int u0 = max(0, r * p.n_chunks - k0), u1 = min(nk, (r + 1) * p.n_chunks - k0);
                float mr = row_m[r];
                for (int u = u0; u < u1; ++u) mr = fmaxf(mr, fin_m[u]);
                row_m[r] = mr;
            }
            __syncthreads();
            if (k0 + nk >= np || np <= kFinStaged) {
                // every part's maxima are in: rescale each partial to its row's max
                for (int u = threadIdx.x; u < nk; u += kAccThreads) {
                    const int r = (k0 + u) / p.n_chunks;
                    const float mk = fin_m[u];
                    fin_z[u] = mk == -INFINITY ? FF{0.f, 0.f} : ff_scale(fin_z[u], expf(mk - row_m[r]));
                }
                __syncthreads();
                for (int r = threadIdx.x; r < nr; r += kAccThreads) {
                    const int u0 = max(0, r * p.n_chunks - k0), u1 = min(nk, (r + 1) * p.n_chunks - k0);
                    FF zr = row_z[r];
                    for (int u = u0; u < u1; ++u) zr = ff_add(zr, fin_z[u]);
                    row_z[r] = zr;
                }
                __syncthreads();
            }
        }
        if (np > kFinStaged) {
            // more partials than one stage: the maxima are final only now, so the
            // sums are taken in a second sweep straight from L2
            for (int r = threadIdx.x; r < nr; r += kAccThreads) {
                const long o = (long)(r0 + r) * p.n_chunks;
                const float mr = row_m[r];
                FF zr = FF{0.f, 0.f};
                for (int k = 0; k < p.n_chunks; ++k) {
                    const float mk = __ldcg(p.pm + o + k);
                    const float2 zk = __ldcg(p.pz + o + k);
                    if (mk != -INFINITY) zr = ff_add(zr, ff_scale(FF{zk.x, zk.y}, expf(mk - mr)));
                }
                row_z[r] = zr;
            }
            __syncthreads();
        }
        for (int r = threadIdx.x; r < nr; r += kAccThreads) {   // nr <= W <= kAccThreads: r is threadIdx.x
            acc_s[r] = test_row(r0 + r, row_m[r], row_z[r], u_own);
            mz_s[r] = make_float2(row_m[r], row_z[r].hi + row_z[r].lo);
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
// sums of the residual r = max(p - q, 0) (after a rejection) or of p (every
// proposal accepted); the last CTA of the sequence picks the chunk where
// u' * S falls and searches inside it
// ----------------------------------------------------------------------------
// the weight of element i (the same fp32 arithmetic wherever it is used)
__device__ __forceinline__ float residual_or_p(float x, float it, float M, float Z, float qi, bool residual) {
    const float pi = expf(x * it - M) / Z;
    if (!residual) return pi;
    const float r = pi - qi;
    return r > 0.f ? r : 0.f;
}

// q at the elements a chunk's registers hold (the vectors of ChunkRegs), with
// 16-byte loads where the row allows them; zeros when not needed
template <typename Tin, int NV, int PV>
__device__ __forceinline__ void load_q(const float *qn, const ChunkRegs<Tin, NV> &cr, bool need, float (&qv)[NV][PV]) {
    const bool vec4 = (reinterpret_cast<uintptr_t>(qn + cr.a0) & 15u) == 0;
#pragma unroll
    for (int v = 0; v < NV; ++v) {
        const bool ok = need && cr.valid(v);
        if (ok && vec4) {
#pragma unroll
            for (int e4 = 0; e4 < PV / 4; ++e4) {
                const float4 t = __ldg(reinterpret_cast<const float4 *>(qn + cr.index(v, 4 * e4)));
                qv[v][4 * e4] = t.x; qv[v][4 * e4 + 1] = t.y; qv[v][4 * e4 + 2] = t.z; qv[v][4 * e4 + 3] = t.w;
            }
        } else {
#pragma unroll
            for (int e = 0; e < PV; ++e) qv[v][e] = ok ? __ldg(qn + cr.index(v, e)) : 0.f;
        }
    }
}

// The draw inside chunk [clo, chi) of the deciding row, whose elements (and q
// where the residual needs it) the CTA holds in registers as ChunkRegs: vector
// v of thread t holds 8 (bf16) or 4 (fp32) consecutive elements, vector slots
// in element order v-major.  The weights are recomputed with the same
// arithmetic as the chunk sums, and for each vector slot an exclusive fp32 scan
// of the threads' vector sums from the chunk's start (the chunk is a small part
// of S, so fp32 holds these offsets to far better than 1e-6 S) lets the thread
// whose vector holds the crossing walk it.  The draw is the smallest index
// whose computed inclusive prefix exceeds xl (x minus the chunks before this
// one: the inverse CDF), reduced with a warp minimum before the shared atomic;
// if rounding leaves no such index, the last positive weight.  Every thread of
// the CTA calls it; the id is returned in every thread.
template <typename Tin, int NV>
__device__ int search_chunk(const ChunkRegs<Tin, NV> &sr, const float (&qs)[NV][Elem<Tin>::kPerVec],
                            const Tin *lg, const float *qn, int clo, int chi, float it, float M, float Z,
                            bool res, float xl) {
    constexpr int PV = Elem<Tin>::kPerVec;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    __shared__ float wtot[kAccThreads / 32];
    __shared__ int s_id, s_last;
    if (threadIdx.x == 0) { s_id = INT_MAX; s_last = -1; }
    // the unaligned head [clo, a0) (fewer than 8 elements) comes first in element order
    float head = 0.f;
    for (int i = clo; i < sr.a0; ++i) {
        const float wi = residual_or_p(Elem<Tin>::load(lg + i), it, M, Z, res ? __ldg(qn + i) : 0.f, res);
        if (wi > 0.f) { if (threadIdx.x == 0) atomicMax(&s_last, i); }
        if (threadIdx.x == 0 && head + wi > xl) atomicMin(&s_id, i);
        head += wi;
    }
    float carry = head;
#pragma unroll
    for (int v = 0; v < NV; ++v) {
        float wv[PV];
        float sv = 0.f;
#pragma unroll
        for (int e = 0; e < PV; ++e) {
            wv[e] = sr.valid(v) ? residual_or_p(sr.x[v][e], it, M, Z, qs[v][e], res) : 0.f;
            sv += wv[e];
        }
        float incl = sv;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        __syncthreads();   // wtot of the previous slot is read
        if (lane == 31) wtot[wid] = incl;
        __syncthreads();
        float acc = carry + (incl - sv);
        float slot_tot = 0.f;
        for (int k = 0; k < kAccThreads / 32; ++k) {
            if (k < wid) acc += wtot[k];
            slot_tot += wtot[k];
        }
        int cand = INT_MAX, last_here = -1;
        if (sr.valid(v)) {
#pragma unroll
            for (int e = 0; e < PV; ++e) {
                if (wv[e] > 0.f) last_here = sr.index(v, e);
                acc += wv[e];
                if (acc > xl && cand == INT_MAX) cand = sr.index(v, e);
            }
        }
        cand = __reduce_min_sync(0xffffffffu, cand);
        last_here = __reduce_max_sync(0xffffffffu, last_here);
        if (lane == 0) {
            if (cand != INT_MAX) atomicMin(&s_id, cand);
            if (last_here >= 0) atomicMax(&s_last, last_here);
        }
        carry += slot_tot;
    }
    // the unaligned tail [a1, chi) last
    if (threadIdx.x == 0) {
        float acc = carry;
        for (int i = sr.a1; i < chi; ++i) {
            const float wi = residual_or_p(Elem<Tin>::load(lg + i), it, M, Z, res ? __ldg(qn + i) : 0.f, res);
            if (wi > 0.f) atomicMax(&s_last, i);
            acc += wi;
            if (acc > xl) atomicMin(&s_id, i);
        }
    }
    __syncthreads();
    int id = s_id;
    if (id == INT_MAX) id = s_last >= 0 ? s_last : clo;  // rounding: last positive weight
    return id;
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
    constexpr int PV = ChunkRegs<Tin, NV>::PV;
    float qv[NV][PV];
    load_q(qn, cr, rejected, qv);
    // per-vector fp32 sums of PV terms, accumulated as float-float; only the
    // weights the draw uses (the residual after a rejection, else p)
    FF sw = FF{0.f, 0.f};
#pragma unroll
    for (int v = 0; v < NV; ++v) {
        if (!cr.valid(v)) break;
        float wv = 0.f;
#pragma unroll
        for (int e = 0; e < PV; ++e) wv += residual_or_p(cr.x[v][e], it, M, Z, qv[v][e], rejected);
        sw = ff_add(sw, wv);
    }
    for (int i = lo + (int)threadIdx.x; i < cr.a0; i += kAccThreads)
        sw = ff_add(sw, residual_or_p(Elem<Tin>::load(lg + i), it, M, Z, rejected ? __ldg(qn + i) : 0.f, rejected));
    for (int i = cr.a1 + (int)threadIdx.x; i < hi; i += kAccThreads)
        sw = ff_add(sw, residual_or_p(Elem<Tin>::load(lg + i), it, M, Z, rejected ? __ldg(qn + i) : 0.f, rejected));
    sw = ff_block_sum(sw);
    if (threadIdx.x == 0) p.rs[(long)b * p.n_draw_chunks + c] = make_float2(sw.hi, sw.lo);
    if (!elect_last(p.row_counter + b, gridDim.x)) return;

    // last CTA of sequence b: an inclusive float-float scan of the chunk sums
    // by the whole CTA (thread k holds chunk k, in passes of kAccThreads),
    // the first chunk whose prefix exceeds x = u' * S, then the element inside
    // it, found in fp32 against x minus the chunks before it
    __shared__ FF wsum[kAccThreads / 32];
    __shared__ FF s_carry, s_base, s_x;
    __shared__ int s_found, s_lastpos, s_res;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const float2 *gcs = p.rs + (long)b * p.n_draw_chunks;
    // the deciding row's u' (every thread draws it; no barrier waits on it)
    const float u2 = philox_uniform(p.seed, (uint32_t)n, (uint32_t)b, 1u, p.offset);
    auto scan_select = [&](bool residual) {
        // one inclusive scan over the chunk sums (thread k holds chunk k, in
        // passes of kAccThreads): its last value is S; then the chunk whose
        // interval [prefix - sum, prefix) holds x = u' * S
        constexpr int kPass = 4;   // chunk sums a thread keeps from the scan (nd <= 4 * kAccThreads here)
        FF incl_k[kPass], v_k[kPass];
        if (threadIdx.x == 0) { s_carry = FF{0.f, 0.f}; s_found = INT_MAX; s_lastpos = -1; }
        __syncthreads();
        const int passes = (p.n_draw_chunks + kAccThreads - 1) / kAccThreads;
        const bool keep = passes <= kPass;
#pragma unroll
        for (int q = 0; q < kPass; ++q) { incl_k[q] = FF{0.f, 0.f}; v_k[q] = FF{0.f, 0.f}; }
        for (int q = 0; q < passes; ++q) {
            const int k = q * kAccThreads + (int)threadIdx.x;
            FF v = FF{0.f, 0.f};
            if (k < p.n_draw_chunks) { const float2 t = __ldcg(gcs + k); v = FF{t.x, t.y}; }
            FF incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const FF y = ff_shfl_up(incl, o);
                if (lane >= o) incl = ff_add(incl, y);
            }
            if (lane == 31) wsum[wid] = incl;
            __syncthreads();
            FF pre = s_carry;
            for (int w = 0; w < wid; ++w) pre = ff_add(pre, wsum[w]);
            incl = ff_add(pre, incl);
            if (k < p.n_draw_chunks && ff_gt0(v)) atomicMax(&s_lastpos, k);
#pragma unroll
            for (int qq = 0; qq < kPass; ++qq)
                if (qq == q) { incl_k[qq] = incl; v_k[qq] = v; }
            __syncthreads();
            if (threadIdx.x == kAccThreads - 1) s_carry = incl;   // the total so far
            __syncthreads();
        }
        const FF S = s_carry;
        if (residual && !ff_gt0(S)) {   // residual zero everywhere: draw from p instead
            if (threadIdx.x == 0) s_res = 2;
            __syncthreads();
            return;
        }
        const FF x = ff_mul(FF{u2, 0.f}, S);
        if (keep) {
#pragma unroll
            for (int q = 0; q < kPass; ++q) {
                const int k = q * kAccThreads + (int)threadIdx.x;
                if (q < passes && k < p.n_draw_chunks) {
                    const FF excl = ff_add(incl_k[q], FF{-v_k[q].hi, -v_k[q].lo});
                    if (ff_lt(x, incl_k[q]) && !ff_lt(x, excl)) { s_found = k; s_base = excl; }   // one k at most
                }
            }
        }
        if (threadIdx.x == 0) { s_x = x; s_res = residual ? 1 : 0; }
        __syncthreads();
        if (s_found == INT_MAX) {
            // more chunks than a thread keeps, or x reached the total through
            // rounding: walk the chunk sums once more with one thread
            if (threadIdx.x == 0) {
                FF acc = FF{0.f, 0.f};
                int found = -1;
                for (int k = 0; k < p.n_draw_chunks; ++k) {
                    const float2 t = __ldcg(gcs + k);
                    const FF nxt = ff_add(acc, FF{t.x, t.y});
                    if (ff_lt(x, nxt)) { found = k; break; }
                    acc = nxt;
                }
                if (found < 0) {   // the last non-empty chunk, and the sum before it
                    found = s_lastpos < 0 ? 0 : s_lastpos;
                    acc = FF{0.f, 0.f};
                    for (int k = 0; k < found; ++k) { const float2 t = __ldcg(gcs + k); acc = ff_add(acc, FF{t.x, t.y}); }
                }
                s_found = found;
                s_base = acc;
            }
            __syncthreads();
        }
    };
    scan_select(rejected);
    if (s_res == 2) {
        // a rejection whose residual is zero everywhere (p = q up to rounding):
        // the draw is from p; rare enough to take the p chunk sums here
        for (int k = 0; k < p.n_draw_chunks; ++k) {
            const int klo = k * p.draw_chunk, khi = min(p.V, klo + p.draw_chunk);
            FF part = FF{0.f, 0.f};
            for (int i = klo + (int)threadIdx.x; i < khi; i += kAccThreads)
                part = ff_add(part, residual_or_p(Elem<Tin>::load(lg + i), it, M, Z, 0.f, false));
            part = ff_block_sum(part);
            if (threadIdx.x == 0) p.rs[(long)b * p.n_draw_chunks + k] = make_float2(part.hi, part.lo);
        }
        __syncthreads();
        scan_select(false);
    }

    const int sel_chunk = s_found;
    const bool res = s_res != 0;
    const float xl = ff_add(s_x, FF{-s_base.hi, -s_base.lo}).hi;   // x - base, to fp32
    const int clo = sel_chunk * p.draw_chunk, chi = min(p.V, clo + p.draw_chunk);
    ChunkRegs<Tin, NV> sr;
    sr.load(lg, clo, chi, -INFINITY);
    float qs[NV][PV];
    load_q(qn, sr, res, qs);
    const int id = search_chunk<Tin, NV>(sr, qs, lg, qn, clo, chi, it, M, Z, res, xl);
    if (threadIdx.x == 0) p.next_id[b] = id;
}

// ----------------------------------------------------------------------------
// sampled acceptance in one cooperative launch (every CTA resident at once):
//   1. the B*T*V logits as equal segments, one per CTA, each reduced to the
//      (max, sum of exp) of its pieces of at most two rows, online: a vector
//      whose maximum is new rescales the running sum first; the records of
//      the pieces (and of the proposals that fall in the segment) published;
//      then a grid barrier;
//   2. the CTAs of sequence b (n_fchunks of them) each read the partials
//      of its T rows and combine them into (M, Z) -- all of them the same
//      way, so with the same result -- test the proposals and find the
//      deciding row n;
//   3. each takes one chunk of row n into registers and publishes the chunk's
//      sums of the residual max(p - q, 0) and of p;
//   4. after a barrier of the sequence's CTAs, each scans the chunk sums; the
//      CTA whose chunk holds x = u' * S draws from its registers.
// The two waits are barriers (below), bounded in time; a CTA only ever waits
// for CTAs that are resident and arrive before they wait themselves.
// ----------------------------------------------------------------------------

// A barrier of `n` CTAs on two counters: thread 0 arrives (a release
// reduction, after the CTA's writes) and waits, bounded in time, for the count
// to reach n (acquire loads).  Once its wait is over, whether or not it
// succeeded, thread 0 takes a departure ticket on `dep`; the CTA holding ticket
// n - 1 (every CTA has passed the wait by then, so none reads the counters any
// more) returns both counters to zero when it ends (barrier_reset).  The
// ticket goes out right after the wait and is read only at the end, so its
// round trip overlaps the CTA's work.  The whole CTA calls the wait; false
// (and the fault bit) if it gave up.
__device__ bool barrier_arrive_wait(unsigned int *ctr, unsigned int *dep, unsigned int n, const WaitTest &wt,
                                    unsigned int *fault, unsigned int &ticket) {
    __shared__ int s_ok;
    __syncthreads();
    if (threadIdx.x == 0) {
        asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(ctr) : "memory");
        const unsigned long long t0 = global_timer();
        int ok = 1;
        for (uint32_t i = 0;; ++i) {
            unsigned int v;
            asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
            if (v >= n + wt.extra) break;
            if ((i & 15u) == 15u && global_timer() - t0 > wt.limit_ns) { ok = 0; break; }
            __nanosleep(20);
        }
        if (!ok) set_fault(fault, FAULT_WAIT_TIMEOUT);
        s_ok = ok;
        ticket = atomicAdd(dep, 1u);
    }
    __syncthreads();
    return s_ok != 0;
}
__device__ __forceinline__ void barrier_reset(unsigned int *arrive, unsigned int *dep, unsigned int n,
                                              unsigned int ticket) {
    if (threadIdx.x == 0 && ticket == n - 1) { *arrive = 0u; *dep = 0u; }
}

// two block-wide maxima at once; results valid in every thread
__device__ __forceinline__ void block_max2(float &a, float &b) {
    __shared__ float sh[2][kAccThreads / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
        b = fmaxf(b, __shfl_xor_sync(0xffffffffu, b, o));
    }
    __syncthreads();
    if (lane == 0) { sh[0][warp] = a; sh[1][warp] = b; }
    __syncthreads();
    a = sh[0][0]; b = sh[1][0];
    for (int w = 1; w < kAccThreads / 32; ++w) { a = fmaxf(a, sh[0][w]); b = fmaxf(b, sh[1][w]); }
}
// two block-wide float-float sums at once; results valid in every thread
__device__ __forceinline__ void ff_block_sum2(FF &a, FF &b) {
    __shared__ FF sh[2][kAccThreads / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    a = ff_warp_sum(a);
    b = ff_warp_sum(b);
    __syncthreads();
    if (lane == 0) { sh[0][warp] = a; sh[1][warp] = b; }
    __syncthreads();
    a = sh[0][0]; b = sh[1][0];
    for (int w = 1; w < kAccThreads / 32; ++w) { a = ff_add(a, sh[0][w]); b = ff_add(b, sh[1][w]); }
}
// block-wide inclusive float-float scan of one value per thread (thread order);
// the total is returned in every thread
__device__ __forceinline__ FF ff_block_scan(FF v, FF &total) {
    __shared__ FF wsum[kAccThreads / 32];
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    FF incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const FF y = ff_shfl_up(incl, o);
        if (lane >= o) incl = ff_add(incl, y);
    }
    __syncthreads();
    if (lane == 31) wsum[wid] = incl;
    __syncthreads();
    FF pre = FF{0.f, 0.f}, tot = FF{0.f, 0.f};
    for (int w = 0; w < kAccThreads / 32; ++w) {
        if (w < wid) pre = ff_add(pre, wsum[w]);
        tot = ff_add(tot, wsum[w]);
    }
    total = tot;
    return ff_add(pre, incl);
}

// e^(y - m) for y <= m in the one-launch stream: 2^((y - m) log2 e) from the
// ex2.approx unit (relative error about 2^-22), y - m rounded once
constexpr float kLog2e = 1.4426950408889634f;
__device__ __forceinline__ float exp_rel(float y, float m) { return ex2((y - m) * kLog2e); }
// e^(x / tau - m), x / tau - m taken with one rounding (FMA)
__device__ __forceinline__ float exp_scaled(float x, float it, float m) { return ex2(fmaf(x, it, -m) * kLog2e); }

// online (max, sum of exp) of one row's piece: y = l / tau of a new element
__device__ __forceinline__ void online_add(float &m, FF &z, float y) {
    if (y > m) {
        if (m != -INFINITY) z = ff_scale(z, exp_rel(m, y));
        m = y;
    }
    if (m != -INFINITY) z = ff_add(z, exp_rel(y, m));
}

template <typename Tin, int NV>
__global__ void __launch_bounds__(kAccThreads, kSampleFusedPerSm) sample_fused_kernel(const SampleParams p) {
    grid_dependency_wait();
    constexpr int PV = Elem<Tin>::kPerVec;
    constexpr int kWarps = kAccThreads / 32;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const float it = p.inv_tau;
    const unsigned int C = gridDim.x;
    const int R = p.B * p.T;
    // the proposals of this CTA's sequence and the uniforms of its rows (the
    // tests' u, the draw's u'), ready for steps 2 and 4
    __shared__ int s_draft[kMaxT];
    __shared__ float s_u[2][kMaxT];
    {
        const int bq = blockIdx.x / p.n_fchunks;
        if (bq < p.B) {
            if (tid < p.T - 1) s_draft[tid] = p.draft[(long)bq * (p.T - 1) + tid];
            if (tid >= 32 && tid < 32 + 2 * p.T) {
                const int j = (tid - 32) % p.T, st = (tid - 32) / p.T;
                s_u[st][j] = philox_uniform(p.seed, (uint32_t)j, (uint32_t)bq, (uint32_t)st, p.offset);
            }
        }
    }
    __syncthreads();

    // ---- 1. segment blockIdx.x: [f0, f0 + len) of the flattened logits
    if ((int)blockIdx.x < p.n_segs) {
        const long N = (long)R * p.V;
        const long f0 = (long)blockIdx.x * p.seg;
        const int len = (int)min((long)p.seg, N - f0);
        const int rA = (int)(f0 / p.V);
        const int offA = (int)(f0 - (long)rA * p.V);   // row index of the first element
        const int jb = p.V - offA;                     // where row rA + 1 starts (>= len: not here)
        // threads 0 and 1: the proposal of row rA / rA + 1, if it falls in this
        // segment -- its logit and q, loaded now, written with the partials
        float2 prop = make_float2(0.f, 0.f);
        int prop_row = -1;
        if (tid < 2) {
            const int r = rA + tid;
            const int plo = tid == 0 ? offA : 0, phi = tid == 0 ? offA + min(len, jb) : len - jb;
            if (r < R && plo < phi && (r % p.T) < p.T - 1) {
                const int d = p.draft[(long)(r / p.T) * (p.T - 1) + r % p.T];
                if (d >= plo && d < phi) {
                    prop_row = r;
                    prop = make_float2(Elem<Tin>::load(static_cast<const Tin *>(p.logits) + (long)r * p.V + d),
                                       __ldg(p.q + (long)r * p.V + d));
                }
            }
        }
        float m0 = -INFINITY, m1 = -INFINITY;          // per thread, rows rA and rA + 1
        FF z0 = FF{0.f, 0.f}, z1 = FF{0.f, 0.f};
        // a vector: its maximum first (exact: it is one of its elements), the
        // running sum rescaled when that is new, then the vector's sum of exp
        auto vec = [&](const uint4 &d, float &m, FF &z) {
            const float vm = Vec16<Tin>::max(d) * it;
            if (vm > m) {
                if (m != -INFINITY) z = ff_scale(z, exp_rel(m, vm));
                m = vm;
            }
            if (m != -INFINITY) {
                float f[PV];
                Vec16<Tin>::unpack(d, f);
                float w[PV];
#pragma unroll
                for (int e = 0; e < PV; ++e) w[e] = exp_scaled(f[e], it, m);
#pragma unroll
                for (int h = PV / 2; h > 0; h >>= 1)
#pragma unroll
                    for (int e = 0; e < h; ++e) w[e] += w[e + h];
                z = ff_add(z, w[0]);
            }
        };
        // two vectors of one row: one maximum, one rescale, 2 PV independent exps
        auto vec2 = [&](const uint4 &d0, const uint4 &d1, float &m, FF &z) {
            const float vm = fmaxf(Vec16<Tin>::max(d0), Vec16<Tin>::max(d1)) * it;
            if (vm > m) {
                if (m != -INFINITY) z = ff_scale(z, exp_rel(m, vm));
                m = vm;
            }
            if (m != -INFINITY) {
                float f0[PV], f1[PV];
                Vec16<Tin>::unpack(d0, f0);
                Vec16<Tin>::unpack(d1, f1);
                float w[PV];
#pragma unroll
                for (int e = 0; e < PV; ++e) w[e] = exp_scaled(f0[e], it, m) + exp_scaled(f1[e], it, m);
#pragma unroll
                for (int h = PV / 2; h > 0; h >>= 1)
#pragma unroll
                    for (int e = 0; e < h; ++e) w[e] += w[e + h];
                z = ff_add(z, w[0]);
            }
        };
        // any one vector: its row's pair, or element by element across the row end
        auto one = [&](const uint4 &d, int j) {
            if (j + PV <= jb || j >= jb) {
                const bool inB = j >= jb;
                float m = inB ? m1 : m0;
                FF z = inB ? z1 : z0;
                vec(d, m, z);
                if (inB) { m1 = m; z1 = z; } else { m0 = m; z0 = z; }
            } else {
                float f[PV];
                Vec16<Tin>::unpack(d, f);
#pragma unroll 1
                for (int e = 0; e < PV; ++e) {
                    const bool inB = j + e >= jb;
                    float m = inB ? m1 : m0;
                    FF z = inB ? z1 : z0;
                    online_add(m, z, f[e] * it);
                    if (inB) { m1 = m; z1 = z; } else { m0 = m; z0 = z; }
                }
            }
        };
        // the segment (16-byte aligned: the logits are, and seg is a multiple
        // of 8) as vectors, thread t taking vectors t, t + 256, t + 512, ... in
        // pairs, the next pair's loads in flight while a pair is reduced; the
        // last segment's ragged end (under one vector) read element by element
        const Tin *lg = static_cast<const Tin *>(p.logits) + f0;
        const uint4 *vp = reinterpret_cast<const uint4 *>(lg);
        const int nvec = len / PV;
        auto ld = [&](int i) { return i < nvec ? ld_stream_u4(vp + i) : make_uint4(0u, 0u, 0u, 0u); };
        auto pair = [&](const uint4 &d0, const uint4 &d1, int i) {
            const int i2 = i + kAccThreads;
            const int j = i * PV, j2 = i2 * PV;
            if (i2 < nvec && (j2 + PV <= jb || j >= jb)) {   // both in one row
                const bool inB = j >= jb;
                float m = inB ? m1 : m0;
                FF z = inB ? z1 : z0;
                vec2(d0, d1, m, z);
                if (inB) { m1 = m; z1 = z; } else { m0 = m; z0 = z; }
            } else {
                one(d0, j);
                if (i2 < nvec) one(d1, j2);
            }
        };
        uint4 a0 = ld(tid), a1 = ld(tid + kAccThreads);
        for (int i = tid; i < nvec; i += 2 * kAccThreads) {
            const uint4 b0 = ld(i + 2 * kAccThreads), b1 = ld(i + 3 * kAccThreads);
            pair(a0, a1, i);
            a0 = b0;
            a1 = b1;
        }
        for (int j = nvec * PV + tid; j < len; j += kAccThreads) {
            const float y = Elem<Tin>::load(lg + j) * it;
            if (j < jb) online_add(m0, z0, y); else online_add(m1, z1, y);
        }
        float M0 = m0, M1 = m1;
        block_max2(M0, M1);
        FF t0 = m0 == -INFINITY ? FF{0.f, 0.f} : ff_scale(z0, expf(m0 - M0));
        FF t1 = m1 == -INFINITY ? FF{0.f, 0.f} : ff_scale(z1, expf(m1 - M1));
        ff_block_sum2(t0, t1);
        const float2 prop1 = make_float2(__shfl_sync(0xffffffffu, prop.x, 1), __shfl_sync(0xffffffffu, prop.y, 1));
        const int prop_row1 = __shfl_sync(0xffffffffu, prop_row, 1);
        if (tid == 0) {
            p.pp[2L * blockIdx.x] = make_float4(M0, t0.hi, t0.lo, 0.f);
            p.pp[2L * blockIdx.x + 1] = make_float4(M1, t1.hi, t1.lo, 0.f);
            if (prop_row >= 0) p.row_stats[prop_row] = prop;
            if (prop_row1 >= 0) p.row_stats[prop_row1] = prop1;
        }
    }

    // every segment's partials are in (a grid barrier)
    unsigned int grid_ticket = 0u, seq_ticket = 0u;
    barrier_arrive_wait(p.counters + 1, p.counters + 2, C, p.wt, p.fault, grid_ticket);
    auto depart = [&]() { barrier_reset(p.counters + 1, p.counters + 2, C, grid_ticket); };
    const int b = blockIdx.x / p.n_fchunks, k = blockIdx.x % p.n_fchunks;
    if (b >= p.B) {
        depart();
        return;
    }

    // ---- sequence b: every row's (M, Z), a warp per row (rows w and w + 8)
    // and lanes over the segments that cover it; the proposal tests; the
    // deciding row n
    __shared__ float s_M[kMaxT];
    __shared__ FF s_Z[kMaxT];
    __shared__ int s_acc[kMaxT];
    auto seg_lo = [&](int r) { return (int)((long)r * p.V / p.seg); };
    auto seg_hi = [&](int r) { return (int)(((long)(r + 1) * p.V - 1) / p.seg); };
    // row r is the first row of every segment that covers it but the first,
    // when that one starts inside row r - 1
    auto slot_of = [&](int r, int i) { return 2 * i + (((long)i * p.seg < (long)r * p.V) ? 1 : 0); };
    static_assert(kMaxT <= 2 * kWarps, "two rows per warp");
    // ---- 2. the partials of rows wid and wid + 8 (lanes over the segments
    // that cover a row, the first 32 kept in registers) and lane 0 the
    // proposal's (logit, q), all loads in flight together
    float pm[2], pzh[2], pzl[2], mloc[2];
    float2 lq[2];
    int ni[2], i0[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int j = wid + kWarps * h, r = b * p.T + j;
        pm[h] = -INFINITY; pzh[h] = 0.f; pzl[h] = 0.f; mloc[h] = -INFINITY;
        lq[h] = make_float2(0.f, 0.f);
        ni[h] = 0;
        i0[h] = 0;
        if (j < p.T) {
            i0[h] = seg_lo(r);
            ni[h] = seg_hi(r) - i0[h] + 1;
            float mx = -INFINITY;
            for (int t = lane; t < ni[h]; t += 32) {
                const float4 q4 = __ldcg(p.pp + slot_of(r, i0[h] + t));
                mx = fmaxf(mx, q4.x);
                if (t == lane) { pm[h] = q4.x; pzh[h] = q4.y; pzl[h] = q4.z; }
            }
            mloc[h] = mx;
            if (lane == 0 && j < p.T - 1) lq[h] = __ldcg(p.row_stats + r);
        }
    }
    // ---- 3. (M, Z) of each row, the proposal test
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int j = wid + kWarps * h, r = b * p.T + j;
        if (j >= p.T) continue;                            // warp-uniform
        float mr = mloc[h];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mr = fmaxf(mr, __shfl_xor_sync(0xffffffffu, mr, o));
        FF zr = pm[h] == -INFINITY ? FF{0.f, 0.f} : ff_scale(FF{pzh[h], pzl[h]}, expf(pm[h] - mr));
        for (int t = lane + 32; t < ni[h]; t += 32) {   // rows over more than 32 segments
            const float4 q4 = __ldcg(p.pp + slot_of(r, i0[h] + t));
            if (q4.x != -INFINITY) zr = ff_add(zr, ff_scale(FF{q4.y, q4.z}, expf(q4.x - mr)));
        }
        zr = ff_warp_sum(zr);
        if (lane == 0) {
            int accept = 0;
            if (j < p.T - 1) {
                const int d = s_draft[j];
                if (d >= 0 && d < p.V) {
                    // accept iff u * q(d) < p(d) = exp(l(d) / tau - M) / Z, as
                    // u * q(d) * Z < exp(...) with the product exact
                    const float ed = expf(lq[h].x * it - mr);
                    accept = ff_lt(ff_mul(ff_prod(s_u[0][j], lq[h].y), zr), FF{ed, 0.f}) ? 1 : 0;
                } else {
                    set_fault(p.fault, FAULT_BAD_DRAFT_ID);
                }
            }
            s_M[j] = mr;
            s_Z[j] = zr;
            s_acc[j] = accept;
        }
    }
    __syncthreads();
    const unsigned int rej = __ballot_sync(0xffffffffu, lane < p.T - 1 && !s_acc[lane]);
    const int n = rej ? __ffs(rej) - 1 : p.T - 1;      // the first rejection, else T - 1
    const float M = s_M[n], Z = s_Z[n].hi + s_Z[n].lo;
    const bool rejected = n < p.T - 1;
    if (k == 0 && tid == 0) p.n_acc[b] = n;

    // ---- 3. chunk k of row n in registers; its sums of the residual and of p
    const long row = (long)b * p.T + n;
    const Tin *lg = static_cast<const Tin *>(p.logits) + row * p.V;
    const float *qn = p.q + row * p.V;
    const int clo = k * p.fchunk, chi = min(p.V, clo + p.fchunk);
    ChunkRegs<Tin, NV> sr;
    sr.load(lg, clo, chi, -INFINITY);
    float qs[NV][PV];
    load_q(qn, sr, rejected, qs);
    const float u2 = s_u[1][n];   // the deciding row's u'
    FF sres = FF{0.f, 0.f}, sp = FF{0.f, 0.f};
#pragma unroll
    for (int v = 0; v < NV; ++v) {
        if (!sr.valid(v)) break;
        float wr = 0.f, wp = 0.f;
#pragma unroll
        for (int e = 0; e < PV; ++e) {
            wr += residual_or_p(sr.x[v][e], it, M, Z, qs[v][e], true);
            wp += residual_or_p(sr.x[v][e], it, M, Z, 0.f, false);
        }
        sres = ff_add(sres, wr);
        sp = ff_add(sp, wp);
    }
    // the unaligned head [clo, a0) and tail [a1, chi)
    auto edge = [&](int i) {
        const float x = Elem<Tin>::load(lg + i);
        sres = ff_add(sres, residual_or_p(x, it, M, Z, rejected ? __ldg(qn + i) : 0.f, true));
        sp = ff_add(sp, residual_or_p(x, it, M, Z, 0.f, false));
    };
    for (int i = clo + tid; i < sr.a0; i += kAccThreads) edge(i);
    for (int i = sr.a1 + tid; i < chi; i += kAccThreads) edge(i);
    ff_block_sum2(sres, sp);
    if (tid == 0) p.fs[(long)b * p.n_fchunks + k] = make_float4(sres.hi, sres.lo, sp.hi, sp.lo);

    // then the chunk where x = u' * S falls (residual after a rejection,
    // unless it is zero everywhere, else p), then the element inside it
    __shared__ int s_found, s_lastpos;
    __shared__ FF s_excl[kAccThreads];
    if (tid == 0) { s_found = INT_MAX; s_lastpos = -1; }
    // ---- 4. every chunk sum of the sequence is in (a barrier of its CTAs)
    barrier_arrive_wait(p.row_counter + b, p.row_counter + p.B + b, (unsigned int)p.n_fchunks, p.wt, p.fault,
                        seq_ticket);
    FF vres = FF{0.f, 0.f}, vp = FF{0.f, 0.f};
    if (tid < p.n_fchunks) {
        const float4 t = __ldcg(p.fs + (long)b * p.n_fchunks + tid);
        vres = FF{t.x, t.y};
        vp = FF{t.z, t.w};
    }
    bool res = rejected;
    FF v = res ? vres : vp, S;
    FF incl = ff_block_scan(v, S);
    if (res && !ff_gt0(S)) {   // p = q up to rounding: the draw is from p
        res = false;
        v = vp;
        incl = ff_block_scan(v, S);
    }
    const FF x = ff_mul(FF{u2, 0.f}, S);
    const FF excl = ff_add(incl, FF{-v.hi, -v.lo});
    s_excl[tid] = excl;
    if (tid < p.n_fchunks) {
        if (ff_lt(x, incl) && !ff_lt(x, excl)) s_found = tid;   // one chunk at most
        if (ff_gt0(v)) atomicMax(&s_lastpos, tid);
    }
    __syncthreads();
    int found = s_found;
    if (found == INT_MAX) found = s_lastpos < 0 ? 0 : s_lastpos;   // rounding: the last non-empty chunk
    if (found == k) {
        const float xl = ff_add(x, FF{-s_excl[found].hi, -s_excl[found].lo}).hi;
        const int id = search_chunk<Tin, NV>(sr, qs, lg, qn, clo, chi, it, M, Z, res, xl);
        if (tid == 0) p.next_id[b] = id;
    }
    barrier_reset(p.row_counter + b, p.row_counter + p.B + b, (unsigned int)p.n_fchunks, seq_ticket);
    depart();
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

int sample_vec_per_thread(sd_dtype dt, int chunk) {
    return dt == SD_BF16 ? vec_per_thread<__nv_bfloat16>(chunk) : vec_per_thread<float>(chunk);
}

int sample_fused_per_sm(sd_dtype dt, int nv) {
    // CTAs of the fused kernel that fit on one SM (cached per instantiation)
    static std::atomic<int> cache[2][3][kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    const int di = dt == SD_BF16 ? 0 : 1, ni = nv <= 1 ? 0 : nv <= 2 ? 1 : 2;
    int v = cache[di][ni][dev].load(std::memory_order_relaxed);
    if (!v) {
        int occ = 0;
        auto query = [&](auto kern) {
            return cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kAccThreads, 0);
        };
        cudaError_t e;
        if (dt == SD_BF16) {
            e = ni == 0 ? query(sample_fused_kernel<__nv_bfloat16, 1>)
              : ni == 1 ? query(sample_fused_kernel<__nv_bfloat16, 2>)
                        : query(sample_fused_kernel<__nv_bfloat16, 4>);
        } else {
            e = ni == 0 ? query(sample_fused_kernel<float, 1>)
              : ni == 1 ? query(sample_fused_kernel<float, 2>)
                        : query(sample_fused_kernel<float, 4>);
        }
        if (e != cudaSuccess) { (void)cudaGetLastError(); occ = 0; }
        v = occ > 0 ? occ : -1;
        cache[di][ni][dev].store(v, std::memory_order_relaxed);
    }
    return v < 0 ? 0 : std::min(v, kSampleFusedPerSm);
}

cudaError_t launch_accept_sample_fused(const SampleParams &p, int grid, cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kAccThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeCooperative;
    attr[1].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cudaError_t e;
    const int NVv = p.dt == SD_BF16 ? vec_per_thread<__nv_bfloat16>(p.fchunk) : vec_per_thread<float>(p.fchunk);
    if (p.dt == SD_BF16) {
        switch (NVv) {
            case 1: e = cudaLaunchKernelEx(&cfg, sample_fused_kernel<__nv_bfloat16, 1>, p); break;
            case 2: e = cudaLaunchKernelEx(&cfg, sample_fused_kernel<__nv_bfloat16, 2>, p); break;
            case 4: e = cudaLaunchKernelEx(&cfg, sample_fused_kernel<__nv_bfloat16, 4>, p); break;
            default: return cudaErrorInvalidValue;
        }
    } else {
        switch (NVv) {
            case 1: e = cudaLaunchKernelEx(&cfg, sample_fused_kernel<float, 1>, p); break;
            case 2: e = cudaLaunchKernelEx(&cfg, sample_fused_kernel<float, 2>, p); break;
            case 4: e = cudaLaunchKernelEx(&cfg, sample_fused_kernel<float, 4>, p); break;
            default: return cudaErrorInvalidValue;
        }
    }
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
