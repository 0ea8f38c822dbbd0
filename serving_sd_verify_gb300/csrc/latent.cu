// SpecFLASH latent visual compressor: out = softmax(Q . F^T) . F per frame,
// Q the Cq (<= 64) learned queries [Cq, d], F a frame's N visual features
// [N, d], no scale on the scores.
//
// Source: "SpecFLASH" README, the first of the draft model's two
// components: a learned set of query vectors attends over the visual
// features of the target's second-to-top layer and replaces them with a few
// latent features (LLaVA-1.5: 576 -> 64; Qwen2.5-VL: 324 -> 36).
//
// Three launches, F read twice (the second time mostly from L2):
//  scores (tensor cores, CTA per (128-feature tile, frame, slice of d)):
//    S^T = F_tile . Q^T over the CTA's slice of d, M 128 features x N 64
//    queries x K 16 MMAs over TMA tiles of F and Q, 256 of d per stage (512
//    contiguous bytes of every feature row per copy), through a 2-stage ring;
//    the epilogue writes the partial S as [query][feature] (fp32).  Slicing d
//    gives enough CTAs to fill the GPU when frames x tiles alone do not.
//  softmax (CTA per (query, frame)): sums the slices in a fixed order, takes
//    the row's max and sum of exp, and writes the normalised weights P
//    [query][feature] as bf16.
//  output (tensor cores, CTA per (frame, 256-wide slice of d)): O = P . F,
//    M 128 (query rows, zero beyond Cq) x N 256 x K 16 MMAs over TMA tiles
//    of P [128 x 64 features] and F [64 features x 256 d] (MN-major B
//    operand) through a 4-stage ring; frames in reverse order, so the frames
//    the scores kernel read last are re-read first, from L2.
#include "common.cuh"
#include "tcgen05.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>
#include <atomic>

namespace sdv {

namespace {

constexpr int kLcThreads = 256;          // warp 0 TMA, warp 1 MMA + tensor memory, warps 4-7 the rest
constexpr int kLcQ = kLatentMaxQueries;  // query columns (zero beyond Cq)
constexpr float kLog2e = 1.4426950408889634f;

// ---- scores kernel ----
constexpr int kScStages = 2;
constexpr int kScChunks = kLatentStageD / 64;      // 64-wide chunks of d per stage
constexpr int kScABytes = kScChunks * 128 * 128;   // [128 features x 256 d] bf16, as 4 chunks of 16 KB
constexpr int kScBBytes = kScChunks * kLcQ * 128;  // [64 queries x 256 d] bf16, as 4 chunks of 8 KB
constexpr int kScStageBytes = kScABytes + kScBBytes;
constexpr int kScOffBar = kScStages * kScStageBytes;
constexpr int kScNumBars = 2 * kScStages + 1;
constexpr int kScOffMisc = kScOffBar + 8 * kScNumBars;
constexpr int kScSmem = kScOffMisc + 16 + 1024;
static_assert(kScSmem <= 227 * 1024, "shared memory per CTA");

// ---- softmax kernel ----
constexpr int kSmThreads = 256;

// ---- output kernel ----
constexpr int kOutStages = 4;
constexpr int kOutN = 256;               // d columns per CTA
constexpr int kOutKeys = 64;             // features per stage
constexpr int kOutPBytes = 128 * kOutKeys * 2;     // [128 query rows x 64 features] bf16, 16 KB
constexpr int kOutFBytes = kOutKeys * kOutN * 2;   // [64 features x 256 d] bf16, 32 KB
constexpr int kOutStageBytes = kOutPBytes + kOutFBytes;
constexpr int kOutOffBar = kOutStages * kOutStageBytes;
constexpr int kOutNumBars = 2 * kOutStages + 1;
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
    const int tile = blockIdx.x, frame = blockIdx.y, split = blockIdx.z;
    const int kt0 = split * p.ksteps_per_split;
    const int nk = min((p.d + kLatentStageD - 1) / kLatentStageD - kt0, p.ksteps_per_split);   // stages of d

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
                tma_load_4d(a, &tm_f, full_bar(st), 0, tile * 128, (kt0 + kt) * kScChunks, frame);
                tma_load_3d(a + kScABytes, &tm_q, full_bar(st), 0, 0, (kt0 + kt) * kScChunks);
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
                for (int c = 0; c < kScChunks; ++c)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        umma_ss(tmem, sw128_desc(a + c * (128 * 128) + kk * 32, 16, 1024),
                                sw128_desc(b + c * (kLcQ * 128) + kk * 32, 16, 1024), idesc,
                                (kt > 0 || c > 0 || kk > 0) ? 1u : 0u);
                umma_commit(empty_bar(st));
            }
            umma_commit(done_bar);
        }
        __syncwarp();
    } else if (warp >= 4) {
        // thread = feature row of the tile = tensor-memory lane; S_split[frame][query][feature]:
        // for each query the warp's 32 features are contiguous
        const int r = (warp & 3) * 32 + lane;
        const int key = tile * 128 + r;
        const bool ok = __all_sync(0xffffffffu, mbar_wait(done_bar, 0, abort_flag, p.fault));
        tc_fence_after();
        const uint32_t taddr = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        float *scol = p.scores + ((long)split * p.frames + frame) * kLcQ * p.ld_s + key;
#pragma unroll
        for (int h = 0; h < kLcQ / 32; ++h) {
            uint32_t v[32];
            tmem_ld32_async(taddr + (uint32_t)(32 * h), v);
            tmem_ld_wait();
            tmem_ld_bind(v);
            if (ok && !*abort_flag && key < p.N) {
#pragma unroll
                for (int c = 0; c < 32; ++c) scol[(long)(32 * h + c) * p.ld_s] = __uint_as_float(v[c]);
            }
        }
        tc_fence_before();
    }
    __syncthreads();
    if (warp == 1) {
        if (*abort_flag && lane == 0) mbar_wait(done_bar, 0, nullptr, p.fault);
        __syncwarp();
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(64) : "memory");
    }
}

// CTA per (query row, frame): S[q][n] = sum of the slices' partial scores
// (in slice order), then P[q][n] = exp(S[q][n] - max_n S[q]) / sum_n exp(...)
// as bf16.  Each thread keeps a running (max, sum of exp) over its features;
// the CTA combines them in a fixed tree order.
__global__ void __launch_bounds__(kSmThreads) latent_softmax_kernel(const LatentParams p) {
#if __CUDA_ARCH__ >= 900
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
#endif
    const int q = blockIdx.x, frame = blockIdx.y, tid = threadIdx.x;
    __shared__ float s_m[kSmThreads / 32], s_l[kSmThreads / 32];
    const long slice = (long)p.frames * kLcQ * p.ld_s;
    const float *srow = p.scores + ((long)frame * kLcQ + q) * p.ld_s;
    auto score = [&](int n) {
        float v = srow[n];
        for (int s2 = 1; s2 < p.n_splits; ++s2) v += srow[s2 * slice + n];
        return v * kLog2e;
    };
    float m = -INFINITY, l = 0.f;
    for (int n = tid; n < p.N; n += kSmThreads) {
        const float v = score(n);
        if (v > m) { l = l * ex2(m - v) + 1.f; m = v; }
        else l += ex2(v - m);
    }
    auto combine = [](float &m1, float &l1, float m2, float l2) {
        const float mm = fmaxf(m1, m2);
        l1 = (m1 == -INFINITY ? 0.f : l1 * ex2(m1 - mm)) + (m2 == -INFINITY ? 0.f : l2 * ex2(m2 - mm));
        m1 = mm;
    };
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) combine(m, l, __shfl_xor_sync(0xffffffffu, m, o), __shfl_xor_sync(0xffffffffu, l, o));
    if ((tid & 31) == 0) { s_m[tid >> 5] = m; s_l[tid >> 5] = l; }
    __syncthreads();
    m = s_m[0];
    l = s_l[0];
    for (int w = 1; w < kSmThreads / 32; ++w) combine(m, l, s_m[w], s_l[w]);
    const float invL = 1.f / l;
    __nv_bfloat16 *prow = p.probs + ((long)frame * p.Cq + q) * p.ld_p;
    for (int n = tid; n < p.N; n += kSmThreads) prow[n] = __float2bfloat16_rn(ex2(score(n) - m) * invL);
}

__global__ void __launch_bounds__(kLcThreads, 1)
latent_output_kernel(const __grid_constant__ CUtensorMap tm_p, const __grid_constant__ CUtensorMap tm_f4,
                     const LatentParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    const uint32_t base = (raw_u32 + 1023u) & ~1023u;
    uint8_t *sbase = smem_raw + (base - raw_u32);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int dt = blockIdx.x, frame = p.frames - 1 - (int)blockIdx.y;
    const int nkt = (p.N + kOutKeys - 1) / kOutKeys;

    const uint32_t bar0 = base + kOutOffBar;
    auto full_bar = [&](int i) { return bar0 + 8u * i; };
    auto empty_bar = [&](int i) { return bar0 + 8u * (kOutStages + i); };
    const uint32_t done_bar = bar0 + 8u * (2 * kOutStages);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(sbase + kOutOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sbase + kOutOffMisc + 8);

    if (tid == 0) {
        for (int i = 0; i < kOutStages; ++i) { mbar_init(full_bar(i), 1); mbar_init(empty_bar(i), 1); }
        mbar_init(done_bar, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_p)) : "memory");
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
                const uint32_t a = base + st * kOutStageBytes;
                mbar_arrive_expect_tx(full_bar(st), (uint32_t)kOutStageBytes);
                tma_load_3d(a, &tm_p, full_bar(st), kt * kOutKeys, 0, frame);
                tma_load_4d(a + kOutPBytes, &tm_f4, full_bar(st), 0, kt * kOutKeys, dt * (kOutN / 64), frame);
                issued = kt + 1;
            }
            if (*abort_flag)
                for (int u = max(0, issued - kOutStages); u < issued; ++u)
                    mbar_wait(full_bar(u % kOutStages), (u / kOutStages) & 1, nullptr, p.fault);
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16(128, kOutN, true);
            for (int kt = 0; kt < nkt; ++kt) {
                const int st = kt % kOutStages;
                if (!mbar_wait(full_bar(st), (kt / kOutStages) & 1, abort_flag, p.fault)) break;
                tc_fence_after();
                const uint32_t pa = base + st * kOutStageBytes, fb = pa + kOutPBytes;
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
            if (done && !*abort_flag && row < p.Cq && dt * kOutN + c0 < p.d) {
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
cudaError_t launch_lc(K kern, dim3 grid, int threads, int smem, cudaStream_t st, A... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3((unsigned)threads);
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
    alignas(64) CUtensorMap mf, mq, mp, mf4;
    {   // F as (d % 64, N, d / 64, frames): box 64 x 128 features x 4 chunks (512 contiguous bytes per row)
        const cuuint64_t dims[4] = {64, (cuuint64_t)p.N, (cuuint64_t)(p.d / 64), (cuuint64_t)p.frames};
        const cuuint64_t strides[3] = {(cuuint64_t)p.ld_f * 2, 128, (cuuint64_t)p.f_fstride * 2};
        const cuuint32_t box[4] = {64, 128, (cuuint32_t)kScChunks, 1};
        if (!encode(&mf, p.f, 4, dims, strides, box)) return cudaErrorInvalidValue;
    }
    {   // Q as (d % 64, Cq, d / 64): box 64 x 64 queries x 4 chunks (rows >= Cq read as zeros)
        const cuuint64_t dims[3] = {64, (cuuint64_t)p.Cq, (cuuint64_t)(p.d / 64)};
        const cuuint64_t strides[2] = {(cuuint64_t)p.d * 2, 128};
        const cuuint32_t box[3] = {64, (cuuint32_t)kLcQ, (cuuint32_t)kScChunks};
        if (!encode(&mq, p.q, 3, dims, strides, box)) return cudaErrorInvalidValue;
    }
    {   // P as (N, Cq, frames): box 64 features x 128 query rows (rows >= Cq read as zeros)
        const cuuint64_t dims[3] = {(cuuint64_t)p.N, (cuuint64_t)p.Cq, (cuuint64_t)p.frames};
        const cuuint64_t strides[2] = {(cuuint64_t)p.ld_p * 2, (cuuint64_t)p.ld_p * 2 * p.Cq};
        const cuuint32_t box[3] = {(cuuint32_t)kOutKeys, 128, 1};
        if (!encode(&mp, p.probs, 3, dims, strides, box)) return cudaErrorInvalidValue;
    }
    {   // F as (d % 64, N, d / 64, frames): box 64 x 64 features x 4 chunks = [64 features x 256 d]
        const cuuint64_t dims[4] = {64, (cuuint64_t)p.N, (cuuint64_t)(p.d / 64), (cuuint64_t)p.frames};
        const cuuint64_t strides[3] = {(cuuint64_t)p.ld_f * 2, 128, (cuuint64_t)p.f_fstride * 2};
        const cuuint32_t box[4] = {64, (cuuint32_t)kOutKeys, (cuuint32_t)(kOutN / 64), 1};
        if (!encode(&mf4, p.f, 4, dims, strides, box)) return cudaErrorInvalidValue;
    }
    static std::atomic<bool> opted_in[64];  // per device: shared-memory limit raised
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !opted_in[dev].load(std::memory_order_acquire)) {
        e = cudaFuncSetAttribute(latent_scores_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kScSmem);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(latent_output_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kOutSmem);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) opted_in[dev].store(true, std::memory_order_release);
    }
    e = launch_lc(latent_scores_kernel, dim3((unsigned)p.n_tiles, (unsigned)p.frames, (unsigned)p.n_splits), kLcThreads,
                  kScSmem, st, mf, mq, p);
    if (e != cudaSuccess) return e;
    e = launch_lc(latent_softmax_kernel, dim3((unsigned)p.Cq, (unsigned)p.frames), kSmThreads, 0, st, p);
    if (e != cudaSuccess) return e;
    return launch_lc(latent_output_kernel, dim3((unsigned)((p.d + kOutN - 1) / kOutN), (unsigned)p.frames),
                     kLcThreads, kOutSmem, st, mp, mf4, p);
}

}  // namespace sdv
