// Drafter K/V projector: K = H . W_k^T and V = H . W_v^T, bf16 in, fp32
// accumulation, bf16 out, written row by row into the drafter's context cache.
//
// Source: "VFlash-FM" project page, "How VFlash-FM works": the drafter never
// reads the video; its keys and values are a linear map of the hidden states
// the target has already cached for every context position.  It runs once over
// the whole context (prefill) and then, every cycle, over the few positions
// just committed (the incremental append).
//
// Prefill (many rows): a persistent tcgen05 GEMM, one CTA per SM walking the
// (128-row tile, 256-column tile of [K | V]) tiles; the hidden-state and
// weight tiles (64 features deep, 128-byte swizzle) stream through a 4-stage
// TMA ring that runs on across tiles; one thread issues M128 N256 K16 MMAs
// into one of two 256-column fp32 accumulators in tensor memory while four
// warps convert the other to bf16 and store it.
// Append (a few rows): bound by reading the weights once, so CUDA cores: four
// warps per output column, lanes over the features, up to kProjSmallRows rows
// per CTA.
#include "common.cuh"
#include "tcgen05.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>
#include <algorithm>
#include <atomic>

namespace sdv {

namespace {

constexpr int kPjThreads = 256;   // warp 0 TMA, warp 1 MMA + tensor memory, warps 4-7 epilogue
constexpr int kPjM = 128, kPjN = 256, kPjK = 64;
constexpr int kPjStages = 4;
constexpr int kPjABytes = kPjM * 128;   // [128 rows x 64 features] bf16
constexpr int kPjBBytes = kPjN * 128;   // [256 out-columns x 64 features] bf16
constexpr int kPjStageBytes = kPjABytes + kPjBBytes;
constexpr int kPjOffBar = kPjStages * kPjStageBytes;
constexpr int kPjNumBars = 2 * kPjStages + 5;   // ring full/empty, accumulator full/empty x 2, done
constexpr int kPjOffMisc = kPjOffBar + 8 * kPjNumBars;
constexpr int kPjSmem = kPjOffMisc + 16 + 1024;
static_assert(kPjSmem <= 227 * 1024, "shared memory per CTA");

constexpr int kSmallCols = 4;            // output columns per CTA of the CUDA-core kernel
constexpr int kSmallSplitK = 4;          // warps sharing one column
constexpr int kSmallThreads = kSmallCols * kSmallSplitK * 32;
constexpr int kSmallInFlight = 4;        // weight vectors per lane per batch

__global__ void __launch_bounds__(kPjThreads, 1)
project_tc_kernel(const __grid_constant__ CUtensorMap tm_h, const __grid_constant__ CUtensorMap tm_wk,
                  const __grid_constant__ CUtensorMap tm_wv, const ProjParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    const uint32_t base = (raw_u32 + 1023u) & ~1023u;
    uint8_t *sbase = smem_raw + (base - raw_u32);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // persistent: CTA b takes tiles b, b + grid, ...; tile t is (row tile
    // t / (2 n_per), column tile t % (2 n_per)), so the CTAs working at the
    // same time share row tiles and the hidden states come from L2 after the
    // first read
    const int n_per = (p.Dout + kPjN - 1) / kPjN;   // column tiles per matrix
    const int n_tiles = ((p.N + kPjM - 1) / kPjM) * 2 * n_per;
    const int nk = (p.Hd + kPjK - 1) / kPjK;

    const uint32_t bar0 = base + kPjOffBar;
    auto full_bar = [&](int i) { return bar0 + 8u * i; };
    auto empty_bar = [&](int i) { return bar0 + 8u * (kPjStages + i); };
    auto acc_full = [&](int i) { return bar0 + 8u * (2 * kPjStages + i); };
    auto acc_empty = [&](int i) { return bar0 + 8u * (2 * kPjStages + 2 + i); };
    const uint32_t done_bar = bar0 + 8u * (2 * kPjStages + 4);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(sbase + kPjOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sbase + kPjOffMisc + 8);

    if (tid == 0) {
        for (int i = 0; i < kPjStages; ++i) { mbar_init(full_bar(i), 1); mbar_init(empty_bar(i), 1); }
        for (int i = 0; i < 2; ++i) { mbar_init(acc_full(i), 1); mbar_init(acc_empty(i), 128); }
        mbar_init(done_bar, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_h)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_wk)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_wv)) : "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_holder)), "r"(2 * kPjN) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
#if __CUDA_ARCH__ >= 900
    // the dependents may start once this kernel's inputs are complete, so that
    // a dependent overlaps this kernel alone
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
#endif
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp == 0) {
        // ---------------------------------------------------------------- TMA producer
        if (lane == 0) {
            int g = 0;                               // (tile, k step) pairs issued
            bool ok = true;
            for (int t = blockIdx.x; ok && t < n_tiles; t += gridDim.x) {
                const int mt = t / (2 * n_per), nt = t % (2 * n_per);
                const bool is_v = nt >= n_per;
                const CUtensorMap *tw = is_v ? &tm_wv : &tm_wk;
                const int col0 = (is_v ? nt - n_per : nt) * kPjN;
                for (int kt = 0; kt < nk; ++kt, ++g) {
                    const int st = g % kPjStages;
                    if (g >= kPjStages &&
                        !mbar_wait(empty_bar(st), ((g / kPjStages) - 1) & 1, abort_flag, p.fault)) {
                        ok = false;
                        break;
                    }
                    const uint32_t a = base + st * kPjStageBytes;
                    mbar_arrive_expect_tx(full_bar(st), (uint32_t)kPjStageBytes);
                    tma_load_2d(a, &tm_h, full_bar(st), kt * kPjK, mt * kPjM);
                    tma_load_2d(a + kPjABytes, tw, full_bar(st), kt * kPjK, col0);
                }
            }
            if (*abort_flag)  // let the copies already issued land before the CTA exits
                for (int u = max(0, g - kPjStages); u < g; ++u)
                    mbar_wait(full_bar(u % kPjStages), (u / kPjStages) & 1, nullptr, p.fault);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16(kPjM, kPjN, false);
            int g = 0;
            bool ok = true;
            for (int t = blockIdx.x, i = 0; ok && t < n_tiles; t += gridDim.x, ++i) {
                const int acc = i & 1;
                // the epilogue has drained this accumulator's previous tile
                if (i >= 2 && !mbar_wait(acc_empty(acc), ((i >> 1) - 1) & 1, abort_flag, p.fault)) break;
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(acc * kPjN);
                for (int kt = 0; kt < nk; ++kt, ++g) {
                    const int st = g % kPjStages;
                    if (!mbar_wait(full_bar(st), (g / kPjStages) & 1, abort_flag, p.fault)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a = base + st * kPjStageBytes, bm = a + kPjABytes;
#pragma unroll
                    for (int kk = 0; kk < kPjK / 16; ++kk)
                        umma_ss(d, sw128_desc(a + kk * 32, 16, 1024), sw128_desc(bm + kk * 32, 16, 1024), idesc,
                                (kt > 0 || kk > 0) ? 1u : 0u);
                    umma_commit(empty_bar(st));
                }
                if (ok) umma_commit(acc_full(acc));
            }
            umma_commit(done_bar);  // every MMA issued, complete or not, before teardown
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ---------------------------------------------------------------- epilogue
        const int r = (warp - 4) * 32 + lane;   // tensor-memory lane = tile row
        for (int t = blockIdx.x, i = 0; t < n_tiles; t += gridDim.x, ++i) {
            const int acc = i & 1;
            const bool ok = __all_sync(0xffffffffu, mbar_wait(acc_full(acc), (i >> 1) & 1, abort_flag, p.fault));
            if (!ok) break;
            tc_fence_after();
            const int mt = t / (2 * n_per), nt = t % (2 * n_per);
            const bool is_v = nt >= n_per;
            const int col0 = (is_v ? nt - n_per : nt) * kPjN;
            const long grow = (long)mt * kPjM + r;
            const uint32_t taddr = tmem + (uint32_t)(acc * kPjN) + ((uint32_t)((warp & 3) * 32) << 16);
            __nv_bfloat16 *out = (is_v ? p.v_out : p.k_out) + grow * p.ld_out + col0;
#pragma unroll 1
            for (int c0 = 0; c0 < kPjN; c0 += 32) {
                uint32_t v[32];
                tmem_ld32_async(taddr + (uint32_t)c0, v);   // warp-wide: before any divergence
                tmem_ld_wait();
                tmem_ld_bind(v);
                if (!*abort_flag && grow < p.N && col0 + c0 < p.Dout) {
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const __nv_bfloat162 h2 =
                            __floats2bfloat162_rn(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1]));
                        pk[e] = *reinterpret_cast<const uint32_t *>(&h2);
                    }
                    uint4 *dst = reinterpret_cast<uint4 *>(out + c0);
#pragma unroll
                    for (int q = 0; q < 4; ++q) dst[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
                }
            }
            tc_fence_before();
            mbar_arrive(acc_empty(acc));            // this thread's lane of the accumulator is read
        }
    }
    __syncthreads();
    if (warp == 1) {
        // every MMA has completed before the tensor memory is freed
        if (lane == 0) mbar_wait(done_bar, 0, nullptr, p.fault);
        __syncwarp();
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(2 * kPjN) : "memory");
    }
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\n cp.async.wait_group 0;" ::: "memory");
}

// Few rows: out[n][c] = sum_k h[n][k] w[c][k].  CTA (x, y) takes output
// columns [4x, 4x + 4) of [K | V] and rows [NR y, NR y + NR); each column is
// shared by 4 warps, warp ks taking the 8-feature vectors ks, ks + 4, ...
// interleaved over the lanes, and the 4 partial sums meet in shared memory
// in a fixed order.  The CTA's hidden rows are copied once into shared
// memory (cp.async, all in flight together) while each lane's weight vectors
// are already on their way; the weights stream from memory once per row
// group.  16 warps per CTA and two or more CTAs per SM keep enough
// independent FMA chains in flight to cover their latency.
// kGather (the commit-time append): CTA row y is row group gi of sequence b
// (y = b * groups + gi, groups = ceil(T / NR)); the sequence's rows are
// 0..n_acc[b] of its block (row r >= 1 is tree node path[b][r-1] when a path
// is given), the group takes rows [NR gi, NR gi + NR) of them, and row r lands
// at output row dst_row0[b] + r; all three come from device memory.
template <int NR, bool kGather>
__global__ void __launch_bounds__(kSmallThreads)
project_small_kernel(const ProjParams p) {
    extern __shared__ uint4 hs[];                 // [nr][Hd / 8]: the hidden rows, bf16
    __shared__ long s_off[NR];                    // element offset of row r in p.h
    __shared__ float red[kSmallSplitK][kSmallCols][NR];
#if __CUDA_ARCH__ >= 900
    asm volatile("griddepcontrol.wait;" ::: "memory");
#endif
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int nr;
    long out_row0;                                // element offset of output row 0
    if (kGather) {
        const int groups = (p.T + NR - 1) / NR;
        const int b = blockIdx.y / groups, r0 = (blockIdx.y % groups) * NR;
        const int n = p.n_acc[b];
        const int d0 = p.dst_row0[b];
        bool ok = n >= 0 && n < p.T && d0 >= 0 && (long)d0 + n + 1 <= p.max_rows;
        for (int r = 1; ok && r <= n; ++r) {
            const int src = p.path ? p.path[(long)b * p.T + r - 1] : r;
            ok = src >= 1 && src < p.T;
        }
        if (!ok) {                                // uniform over the CTA
            if (blockIdx.x == 0 && r0 == 0 && tid == 0) set_fault(p.fault, FAULT_BAD_COMMIT);
            return;
        }
        nr = min(NR, n + 1 - r0);
        if (nr <= 0) return;                      // uniform: this group holds none of the rows
        if (tid < nr) {
            const int r = r0 + tid;
            const int src = r == 0 ? 0 : p.path ? p.path[(long)b * p.T + r - 1] : r;
            s_off[tid] = (long)b * p.h_bstride + (long)src * p.ld_h;
        }
        out_row0 = (long)b * p.out_bstride + (long)(d0 + r0) * p.ld_out;
    } else {
        const int n0 = blockIdx.y * NR;
        nr = min(NR, p.N - n0);
        if (tid < nr) s_off[tid] = (long)(n0 + tid) * p.ld_h;
        out_row0 = (long)n0 * p.ld_out;
    }
    __syncthreads();
    const int hv = p.Hd / 8;                      // 16-byte vectors per hidden row
    for (int i = tid; i < nr * hv; i += kSmallThreads) {
        const int r = i / hv, x = i - r * hv;
        cp_async16(smem_u32(hs + i), p.h + s_off[r] + 8 * x);
    }

    const int col_in = warp % kSmallCols, ks = warp / kSmallCols;
    const int c = min(blockIdx.x * kSmallCols + col_in, 2 * p.Dout - 1);
    const bool is_v = c >= p.Dout;
    const int cc = is_v ? c - p.Dout : c;
    const __nv_bfloat16 *w = (is_v ? p.wv : p.wk) + (long)cc * p.Hd;
    constexpr int kU = kSmallInFlight;
    constexpr int kStep = 32 * kSmallSplitK;      // vectors between a lane's consecutive ones
    uint4 cur[kU], nxt[kU];
    auto load = [&](uint4 (&dst)[kU], int v0) {
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int v = v0 + u * kStep;
            dst[u] = v < hv ? ld_stream_u4(w + 8 * v) : make_uint4(0u, 0u, 0u, 0u);
        }
    };
    const int v_first = lane + 32 * ks;
    load(cur, v_first);
    cp_async_wait_all();
    __syncthreads();

    float acc[NR];
#pragma unroll
    for (int n = 0; n < NR; ++n) acc[n] = 0.f;
    for (int v0 = v_first; v0 < hv; v0 += kStep * kU) {
        if (v0 + kStep * kU < hv) load(nxt, v0 + kStep * kU);
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int v = v0 + u * kStep;
            if (v < hv) {
                float wf[8];
                unpack_bf16x8(cur[u], wf);
#pragma unroll
                for (int n = 0; n < NR; ++n) {
                    if (n < nr) {
                        float hf[8];
                        unpack_bf16x8(hs[n * hv + v], hf);
#pragma unroll
                        for (int e = 0; e < 8; ++e) acc[n] = fmaf(hf[e], wf[e], acc[n]);
                    }
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) cur[u] = nxt[u];
    }
#pragma unroll
    for (int n = 0; n < NR; ++n) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc[n] += __shfl_xor_sync(0xffffffffu, acc[n], o);
    }
    if (lane < nr) {
        float v = acc[0];
#pragma unroll
        for (int n = 1; n < NR; ++n) v = lane == n ? acc[n] : v;
        red[ks][col_in][lane] = v;
    }
    __syncthreads();
    if (tid < kSmallCols * NR) {
        const int ci = tid / NR, n = tid % NR;
        const int col = blockIdx.x * kSmallCols + ci;
        if (n < nr && col < 2 * p.Dout) {
            float v = red[0][ci][n];
#pragma unroll
            for (int q = 1; q < kSmallSplitK; ++q) v += red[q][ci][n];
            const bool ov = col >= p.Dout;
            (ov ? p.v_out : p.k_out)[out_row0 + (long)n * p.ld_out + (ov ? col - p.Dout : col)] =
                __float2bfloat16_rn(v);
        }
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn_pj() {
    // looked up once; the initialisation of a function-local static is thread-safe
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
        return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
    }();
    return fn;
}

// 2-D map over a row-major bf16 matrix [rows, cols] with row stride ld (elements);
// box: 64 columns x box_rows rows, 128-byte swizzle
bool make_map_2d(CUtensorMap *m, const void *ptr, long rows, long cols, long ld, int box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn_pj();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)box_rows}, estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename K, typename P>
cudaError_t launch_pdl_pj(K kern, dim3 grid, dim3 block, size_t smem, cudaStream_t st, const P &args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args);
}

// dynamic shared memory of the CUDA-core kernel: NR hidden rows
size_t small_smem(int NR, int Hd) { return (size_t)NR * Hd * 2; }

template <int NR, bool kGather>
cudaError_t launch_small(const ProjParams &p, dim3 grid, cudaStream_t st) {
    static std::atomic<bool> opted_in[64];  // per device: shared-memory limit raised
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !opted_in[dev].load(std::memory_order_acquire)) {
        e = cudaFuncSetAttribute(project_small_kernel<NR, kGather>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kProjSmallSmemMax);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) opted_in[dev].store(true, std::memory_order_release);
    }
    return launch_pdl_pj(project_small_kernel<NR, kGather>, grid, dim3(kSmallThreads), small_smem(NR, p.Hd), st, p);
}

}  // namespace

bool project_tc_supported() {
    if (!encode_fn_pj()) return false;
    int dev = 0, optin = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return false;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    return optin >= kPjSmem && major == 10 && minor == 3;
}

bool project_small_supported(int rows_per_cta, int Hd) {
    return small_smem(rows_per_cta, Hd) <= kProjSmallSmemMax;
}

cudaError_t launch_project_commit(const ProjParams &p, cudaStream_t st) {
    const int groups = (p.T + kMaxT - 1) / kMaxT;   // row groups of kMaxT rows per sequence
    const dim3 grid((unsigned)((2 * p.Dout + kSmallCols - 1) / kSmallCols), (unsigned)(p.B * groups));
    return launch_small<kMaxT, true>(p, grid, st);
}

cudaError_t launch_project(const ProjParams &p, int path, cudaStream_t st) {
    if (p.N <= 0) return cudaSuccess;
    if (path == 1) {
        const int nr = (p.N <= 8 || small_smem(kProjSmallRows, p.Hd) > kProjSmallSmemMax) ? 8 : kProjSmallRows;
        const dim3 grid((unsigned)((2 * p.Dout + kSmallCols - 1) / kSmallCols), (unsigned)((p.N + nr - 1) / nr));
        if (nr == 8) return launch_small<8, false>(p, grid, st);
        return launch_small<kProjSmallRows, false>(p, grid, st);
    }
    alignas(64) CUtensorMap mh, mk, mv;
    if (!make_map_2d(&mh, p.h, p.N, p.Hd, p.ld_h, kPjM)) return cudaErrorInvalidValue;
    if (!make_map_2d(&mk, p.wk, p.Dout, p.Hd, p.Hd, kPjN)) return cudaErrorInvalidValue;
    if (!make_map_2d(&mv, p.wv, p.Dout, p.Hd, p.Hd, kPjN)) return cudaErrorInvalidValue;
    static std::atomic<bool> opted_in[64];  // per device: shared-memory limit raised
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !opted_in[dev].load(std::memory_order_acquire)) {
        e = cudaFuncSetAttribute(project_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPjSmem);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) opted_in[dev].store(true, std::memory_order_release);
    }
    const long n_tiles = (long)((p.N + kPjM - 1) / kPjM) * 2 * ((p.Dout + kPjN - 1) / kPjN);
    const dim3 grid((unsigned)std::min<long>(n_tiles, device_sm_count()));   // persistent: one CTA per SM
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kPjThreads);
    cfg.dynamicSmemBytes = kPjSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, project_tc_kernel, mh, mk, mv, p);
}

}  // namespace sdv
