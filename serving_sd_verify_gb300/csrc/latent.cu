// SpecFLASH latent visual compressor: out = softmax(Q . F^T) . F per frame,
// Q the Cq (<= 64) learned queries [Cq, d], F a frame's N visual features
// [N, d], no scale on the scores.
//
// Source: "SpecFLASH" README, the first of the draft model's two
// components: a learned set of query vectors attends over the visual
// features of the target's second-to-top layer and replaces them with a few
// latent features (LLaVA-1.5: 576 -> 64; Qwen2.5-VL: 324 -> 36).
//
// Two tensor-core kernels, F read twice (the second time mostly from L2):
//  scores (CTA per (frame, 128-feature tile)): S^T = F_tile . Q^T, M 128
//    features x N 64 queries x K d, with TMA tiles of F and Q through a
//    6-stage ring; the epilogue writes S^T (fp32) and the tile's softmax
//    statistics per query (max, sum of exp) to the workspace.
//  output (CTA per (frame, 256-wide slice of d)): combines the statistics,
//    builds P = softmax rows as bf16 tiles [128 query rows x 64 features] in
//    a 3-slot ring (rows >= Cq stay zero) while TMA brings the matching F
//    tiles [64 features x 256 d] (MN-major B operand), and accumulates
//    O = P . F in tensor memory (M 128 x N 256 x K 16 MMAs); frames in
//    reverse order, so the last frames the scores kernel read come first.
#include "common.cuh"
#include "tcgen05.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>

namespace sdv {

namespace {

constexpr int kLcThreads = 256;          // warp 0 TMA, warp 1 MMA + tensor memory, warps 4-7 the rest
constexpr int kLcQ = kLatentMaxQueries;  // query columns (zero beyond Cq)
constexpr float kLog2e = 1.4426950408889634f;

// ---- scores kernel ----
constexpr int kScStages = 6;
constexpr int kScABytes = 128 * 128;     // [128 features x 64 d] bf16
constexpr int kScBBytes = kLcQ * 128;    // [64 queries x 64 d] bf16
constexpr int kScStageBytes = kScABytes + kScBBytes;
constexpr int kScOffBar = kScStages * kScStageBytes;
constexpr int kScNumBars = 2 * kScStages + 1;
constexpr int kScOffMisc = kScOffBar + 8 * kScNumBars;
constexpr int kScSmem = kScOffMisc + 16 + 1024;
constexpr int kScRowStride = kLcQ + 1;   // floats per staged score row (bank-conflict free)
static_assert(128 * kScRowStride * 4 + 2 * 2 * kLcQ * 4 <= kScOffBar, "staging fits the ring");
static_assert(kScSmem <= 227 * 1024, "shared memory per CTA");

// ---- output kernel ----
constexpr int kOutStages = 3;
constexpr int kOutN = 256;               // d columns per CTA
constexpr int kOutKeys = 64;             // features per stage
constexpr int kOutFBytes = kOutKeys * kOutN * 2;   // 32 KB
constexpr int kOutPBytes = 128 * kOutKeys * 2;     // 16 KB
constexpr int kOutOffP = kOutStages * kOutFBytes;
constexpr int kOutOffBar = kOutOffP + kOutStages * kOutPBytes;
constexpr int kOutNumBars = 3 * kOutStages + 1;
constexpr int kOutOffMisc = kOutOffBar + 8 * kOutNumBars;
constexpr int kOutSmem = kOutOffMisc + 16 + 1024;
static_assert(kOutSmem <= 227 * 1024, "shared memory per CTA");

__global__ void __launch_bounds__(kLcThreads, 1)
latent_scores_kernel(const __grid_constant__ CUtensorMap tm_f, const __grid_constant__ CUtensorMap tm_q,
                     const LatentParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    const uint32_t base = (raw_u32 + 1023u) & ~1023u;
    uint8_t *sbase = smem_raw + (base - raw_u32);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tile = blockIdx.x, frame = blockIdx.y;
    const int nk = p.d / 64;

    const uint32_t bar0 = base + kScOffBar;
    auto full_bar = [&](int i) { return bar0 + 8u * i; };
    auto empty_bar = [&](int i) { return bar0 + 8u * (kScStages + i); };
    const uint32_t done_bar = bar0 + 8u * (2 * kScStages);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(sbase + kScOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sbase + kScOffMisc + 8);

    if (tid == 0) {
        for (int i = 0; i < kScStages; ++i) { mbar_init(full_bar(i), 1); mbar_init(empty_bar(i), 1); }
        mbar_init(done_bar, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_f)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_q)) : "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_holder)), "r"(64) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
#if __CUDA_ARCH__ >= 900
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
#endif
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp == 0) {
        if (lane == 0) {
            int issued = 0;
            for (int kt = 0; kt < nk; ++kt) {
                const int st = kt % kScStages;
                if (kt >= kScStages &&
                    !mbar_wait(empty_bar(st), ((kt / kScStages) - 1) & 1, abort_flag, p.fault))
                    break;
                const uint32_t a = base + st * kScStageBytes;
                mbar_arrive_expect_tx(full_bar(st), (uint32_t)kScStageBytes);
                tma_load_3d(a, &tm_f, full_bar(st), kt * 64, tile * 128, frame);
                tma_load_2d(a + kScABytes, &tm_q, full_bar(st), kt * 64, 0);
                issued = kt + 1;
            }
            if (*abort_flag)
                for (int u = max(0, issued - kScStages); u < issued; ++u)
                    mbar_wait(full_bar(u % kScStages), (u / kScStages) & 1, nullptr, p.fault);
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16(128, kLcQ, false);
            for (int kt = 0; kt < nk; ++kt) {
                const int st = kt % kScStages;
                if (!mbar_wait(full_bar(st), (kt / kScStages) & 1, abort_flag, p.fault)) break;
                tc_fence_after();
                const uint32_t a = base + st * kScStageBytes, b = a + kScABytes;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    umma_ss(tmem, sw128_desc(a + kk * 32, 16, 1024), sw128_desc(b + kk * 32, 16, 1024), idesc,
                            (kt > 0 || kk > 0) ? 1u : 0u);
                umma_commit(empty_bar(st));
            }
            umma_commit(done_bar);
        }
        __syncwarp();
    }
    // warps 4-7: thread = feature row of the tile = tensor-memory lane
    const bool epi = warp >= 4;
    const int r = (warp & 3) * 32 + lane;
    const int key = tile * 128 + r;
    float *stage = reinterpret_cast<float *>(sbase);   // [128][kScRowStride], over the ring once all MMAs are done
    bool ok = true;
    if (epi) {
        ok = __all_sync(0xffffffffu, mbar_wait(done_bar, 0, abort_flag, p.fault));
        tc_fence_after();
        const uint32_t taddr = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        uint32_t v[32];
        float *srow = p.scores + (((long)frame * p.n_tiles + tile) * 128 + r) * kLcQ;
#pragma unroll
        for (int h = 0; h < kLcQ / 32; ++h) {
            tmem_ld32_async(taddr + (uint32_t)(32 * h), v);
            tmem_ld_wait();
            tmem_ld_bind(v);
#pragma unroll
            for (int c = 0; c < 32; ++c) stage[r * kScRowStride + 32 * h + c] = __uint_as_float(v[c]);
            if (ok && key < p.N) {
                float4 *dst = reinterpret_cast<float4 *>(srow + 32 * h);
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    dst[c] = make_float4(__uint_as_float(v[4 * c]), __uint_as_float(v[4 * c + 1]),
                                         __uint_as_float(v[4 * c + 2]), __uint_as_float(v[4 * c + 3]));
            }
        }
        tc_fence_before();
    }
    __syncthreads();
    // the tile's statistics per query: thread t takes query t % 64 over half the rows
    if (epi) {
        const int t = tid - 128;
        const int q = t % kLcQ, half = t / kLcQ;
        const int r0 = half * 64, r1 = min(r0 + 64, p.N - tile * 128);
        float m = -INFINITY;
        for (int rr = r0; rr < r1; ++rr) m = fmaxf(m, stage[rr * kScRowStride + q]);
        float l = 0.f;
        if (m != -INFINITY)
            for (int rr = r0; rr < r1; ++rr) l += ex2((stage[rr * kScRowStride + q] - m) * kLog2e);
        float *xs = stage + 128 * kScRowStride;   // [2 halves][2][kLcQ]
        xs[(half * 2 + 0) * kLcQ + q] = m;
        xs[(half * 2 + 1) * kLcQ + q] = l;
        named_sync(1, 128);
        if (half == 0 && ok && !*abort_flag) {
            const float m1 = xs[(2 + 0) * kLcQ + q], l1 = xs[(2 + 1) * kLcQ + q];
            const float mm = fmaxf(m, m1);
            const float ll = (m == -INFINITY ? 0.f : l * ex2((m - mm) * kLog2e)) +
                             (m1 == -INFINITY ? 0.f : l1 * ex2((m1 - mm) * kLog2e));
            const long si = ((long)frame * p.n_tiles + tile) * kLcQ + q;
            p.stat_m[si] = mm;
            p.stat_l[si] = ll;
        }
    }
    __syncthreads();
    if (warp == 1) {
        if (*abort_flag && lane == 0) mbar_wait(done_bar, 0, nullptr, p.fault);
        __syncwarp();
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(64) : "memory");
    }
}

__global__ void __launch_bounds__(kLcThreads, 1)
latent_output_kernel(const __grid_constant__ CUtensorMap tm_f4, const LatentParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    const uint32_t base = (raw_u32 + 1023u) & ~1023u;
    uint8_t *sbase = smem_raw + (base - raw_u32);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int dt = blockIdx.x, frame = p.frames - 1 - (int)blockIdx.y;
    const int nkt = (p.N + kOutKeys - 1) / kOutKeys;

    const uint32_t bar0 = base + kOutOffBar;
    auto f_full = [&](int i) { return bar0 + 8u * i; };
    auto p_full = [&](int i) { return bar0 + 8u * (kOutStages + i); };
    auto empty_bar = [&](int i) { return bar0 + 8u * (2 * kOutStages + i); };
    const uint32_t done_bar = bar0 + 8u * (3 * kOutStages);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(sbase + kOutOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sbase + kOutOffMisc + 8);

    // P slots start as zeros: rows >= Cq are never written again
    for (int i = tid; i < kOutStages * kOutPBytes / 16; i += kLcThreads)
        reinterpret_cast<uint4 *>(sbase + kOutOffP)[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
    if (tid == 0) {
        for (int i = 0; i < kOutStages; ++i) {
            mbar_init(f_full(i), 1);
            mbar_init(p_full(i), 128);
            mbar_init(empty_bar(i), 1);
        }
        mbar_init(done_bar, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_f4)) : "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_holder)), "r"(kOutN) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
#if __CUDA_ARCH__ >= 900
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
#endif
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp == 0) {
        if (lane == 0) {
            int issued = 0;
            for (int kt = 0; kt < nkt; ++kt) {
                const int st = kt % kOutStages;
                if (kt >= kOutStages &&
                    !mbar_wait(empty_bar(st), ((kt / kOutStages) - 1) & 1, abort_flag, p.fault))
                    break;
                mbar_arrive_expect_tx(f_full(st), (uint32_t)kOutFBytes);
                tma_load_4d(base + st * kOutFBytes, &tm_f4, f_full(st), 0, kt * kOutKeys, dt * (kOutN / 64), frame);
                issued = kt + 1;
            }
            if (*abort_flag)
                for (int u = max(0, issued - kOutStages); u < issued; ++u)
                    mbar_wait(f_full(u % kOutStages), (u / kOutStages) & 1, nullptr, p.fault);
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16(128, kOutN, true);
            for (int kt = 0; kt < nkt; ++kt) {
                const int st = kt % kOutStages;
                const uint32_t par = (kt / kOutStages) & 1;
                if (!mbar_wait(f_full(st), par, abort_flag, p.fault)) break;
                if (!mbar_wait(p_full(st), par, abort_flag, p.fault)) break;
                tc_fence_after();
                const uint32_t fb = base + st * kOutFBytes, pa = base + kOutOffP + st * kOutPBytes;
#pragma unroll
                for (int kk = 0; kk < kOutKeys / 16; ++kk)
                    umma_ss(tmem, sw128_desc(pa + kk * 32, 16, 1024),
                            sw128_desc(fb + kk * 2048, kOutKeys * 128, 1024), idesc, (kt > 0 || kk > 0) ? 1u : 0u);
                umma_commit(empty_bar(st));
            }
            umma_commit(done_bar);
        }
        __syncwarp();
    } else if (warp >= 4) {
        // P builders: thread t takes query q = t % 64 and features [32 h, 32 h + 32) of each tile
        const int t = tid - 128;
        const int q = t % kLcQ, h = t / kLcQ;
        const bool live = q < p.Cq;
        float M = -INFINITY, invL = 0.f;
        if (live) {
            for (int i = 0; i < p.n_tiles; ++i)
                M = fmaxf(M, p.stat_m[((long)frame * p.n_tiles + i) * kLcQ + q]);
            float L = 0.f;
            for (int i = 0; i < p.n_tiles; ++i) {
                const long si = ((long)frame * p.n_tiles + i) * kLcQ + q;
                const float mi = p.stat_m[si];
                if (mi != -INFINITY) L += p.stat_l[si] * ex2((mi - M) * kLog2e);
            }
            invL = 1.f / L;
        }
        const float Ml = M * kLog2e;
        const float *sc = p.scores + (long)frame * p.n_tiles * 128 * kLcQ + q;
        bool ok = true;
        for (int kt = 0; kt < nkt; ++kt) {
            const int st = kt % kOutStages;
            if (kt >= kOutStages)
                ok = ok && mbar_wait(empty_bar(st), ((kt / kOutStages) - 1) & 1, abort_flag, p.fault);
            if (ok && live) {
                uint8_t *slot = sbase + kOutOffP + st * kOutPBytes;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int k0 = kt * kOutKeys + 32 * h + 8 * c;
                    uint32_t pk[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int ka = k0 + 2 * e, kb = ka + 1;
                        const float pa = ka < p.N ? ex2(fmaf(sc[(long)ka * kLcQ], kLog2e, -Ml)) * invL : 0.f;
                        const float pb = kb < p.N ? ex2(fmaf(sc[(long)kb * kLcQ], kLog2e, -Ml)) * invL : 0.f;
                        const __nv_bfloat162 v2 = __floats2bfloat162_rn(pa, pb);
                        pk[e] = *reinterpret_cast<const uint32_t *>(&v2);
                    }
                    *reinterpret_cast<uint4 *>(slot + sw128_off(q, 4 * h + c)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                }
                fence_proxy_async_smem();
            }
            mbar_arrive(p_full(st));
        }
        // epilogue: thread = query row = tensor-memory lane (warps 4-7 own lanes 0-127)
        const bool done = __all_sync(0xffffffffu, mbar_wait(done_bar, 0, abort_flag, p.fault));
        tc_fence_after();
        const int row = (warp & 3) * 32 + lane;
        const uint32_t taddr = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        __nv_bfloat16 *orow = p.out + (long)frame * p.out_fstride + (long)row * p.ld_out + dt * kOutN;
#pragma unroll 1
        for (int c0 = 0; c0 < kOutN; c0 += 32) {
            uint32_t v[32];
            tmem_ld32_async(taddr + (uint32_t)c0, v);
            tmem_ld_wait();
            tmem_ld_bind(v);
            if (done && ok && !*abort_flag && row < p.Cq && dt * kOutN + c0 < p.d) {
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const __nv_bfloat162 h2 = __floats2bfloat162_rn(__uint_as_float(v[2 * e]),
                                                                     __uint_as_float(v[2 * e + 1]));
                    pk[e] = *reinterpret_cast<const uint32_t *>(&h2);
                }
                uint4 *dst = reinterpret_cast<uint4 *>(orow + c0);
#pragma unroll
                for (int e = 0; e < 4; ++e) dst[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
            }
        }
        tc_fence_before();
    }
    __syncthreads();
    if (warp == 1) {
        if (*abort_flag && lane == 0) mbar_wait(done_bar, 0, nullptr, p.fault);
        __syncwarp();
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kOutN) : "memory");
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn_lc() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

bool encode(CUtensorMap *m, const void *ptr, int rank, const cuuint64_t *dims, const cuuint64_t *strides,
            const cuuint32_t *box) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn_lc();
    if (!fn) return false;
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void *>(ptr), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename K, typename... A>
cudaError_t launch_lc(K kern, dim3 grid, int smem, cudaStream_t st, A... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kLcThreads);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

}  // namespace

bool latent_supported() {
    if (!encode_fn_lc()) return false;
    int dev = 0, optin = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return false;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    return optin >= kScSmem && optin >= kOutSmem && major == 10 && minor == 3;
}

cudaError_t launch_latent(const LatentParams &p, cudaStream_t st) {
    alignas(64) CUtensorMap mf, mq, mf4;
    {   // F as (d, N, frames): box 64 d x 128 features
        const cuuint64_t dims[3] = {(cuuint64_t)p.d, (cuuint64_t)p.N, (cuuint64_t)p.frames};
        const cuuint64_t strides[2] = {(cuuint64_t)p.ld_f * 2, (cuuint64_t)p.f_fstride * 2};
        const cuuint32_t box[3] = {64, 128, 1};
        if (!encode(&mf, p.f, 3, dims, strides, box)) return cudaErrorInvalidValue;
    }
    {   // Q as (d, Cq): box 64 d x 64 queries (rows >= Cq read as zeros)
        const cuuint64_t dims[2] = {(cuuint64_t)p.d, (cuuint64_t)p.Cq};
        const cuuint64_t strides[1] = {(cuuint64_t)p.d * 2};
        const cuuint32_t box[2] = {64, (cuuint32_t)kLcQ};
        if (!encode(&mq, p.q, 2, dims, strides, box)) return cudaErrorInvalidValue;
    }
    {   // F as (d % 64, N, d / 64, frames): box 64 x 64 features x 4 chunks = [64 features x 256 d]
        const cuuint64_t dims[4] = {64, (cuuint64_t)p.N, (cuuint64_t)(p.d / 64), (cuuint64_t)p.frames};
        const cuuint64_t strides[3] = {(cuuint64_t)p.ld_f * 2, 128, (cuuint64_t)p.f_fstride * 2};
        const cuuint32_t box[4] = {64, (cuuint32_t)kOutKeys, (cuuint32_t)(kOutN / 64), 1};
        if (!encode(&mf4, p.f, 4, dims, strides, box)) return cudaErrorInvalidValue;
    }
    static bool opted_in[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !opted_in[dev]) {
        e = cudaFuncSetAttribute(latent_scores_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kScSmem);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(latent_output_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kOutSmem);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) opted_in[dev] = true;
    }
    e = launch_lc(latent_scores_kernel, dim3((unsigned)p.n_tiles, (unsigned)p.frames), kScSmem, st, mf, mq, p);
    if (e != cudaSuccess) return e;
    return launch_lc(latent_output_kernel, dim3((unsigned)((p.d + kOutN - 1) / kOutN), (unsigned)p.frames), kOutSmem,
                     st, mf4, p);
}

}  // namespace sdv
