// Tensor-core split-KV attention for sm_103a: TMA-fed K/V tiles, tcgen05 MMAs
// with fp32 accumulators in tensor memory, an fp32 online softmax on the CUDA
// cores.  bf16 storage, D = 128, (Hq/Hkv) * T <= 128.
//
// Target verify: "VFlash-FM" project page, "How VFlash-FM works" -- the
// target scores the 16 block slots in one forward with grouped-query
// attention over its KV cache, slot j only seeing keys before slot j+1.
// Drafter: same page -- every block query sees every projected context key
// and every block key.
//
// One CTA owns one (split, kv head, sequence).  All G*T query rows that read
// that kv head form the M = 128 rows of the MMAs (zero-padded), so every K/V
// tile is fetched from HBM once and serves every row:
//   S_t = Q . K_t^T   (M 128, N 64 keys, K 128)   -> tensor memory, 2 buffers
//   P_t = exp2(S_t * scale * log2e - m), split as P_hi + P_lo, both bf16
//   O  += P_hi . V_t + P_lo . V_t   (M 128, N 128, K 64)  -> tensor memory
// (the two-term split keeps the weights to about 2^-17 relative, so the
// product is as accurate as an fp32 P even when a few keys dominate)
// Warp roles (192 threads): warps 0-3 own one query row per thread (tensor
// memory lane = row) and run the softmax, warp 4 issues the TMA loads of a
// 3-stage K/V ring, warp 5 allocates tensor memory and issues the MMAs from one
// elected thread.  The running max is only moved when it grows by more than
// 2^8, so O is rescaled in tensor memory rarely (exact either way: the same
// reference max is used for P and for l).  Every wait is bounded by the
// global timer; a wait that gives up sets the fault word, and the CTA drains
// its copies and MMAs and frees its tensor memory before it returns.
#include "common.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>

#include <math.h>
#include <string.h>

namespace sdv {

namespace {

constexpr int kTcThreads = 192;
constexpr int kStages = 3;
constexpr int kBN = kTileKeys;             // keys per tile (64)
constexpr int kQBytes = 2 * 128 * 128;      // two K-blocks of [128 rows x 128 B]
constexpr int kKBytes = 2 * kBN * 128;      // two K-blocks of [64 keys x 128 B]
constexpr int kVBytes = 2 * kBN * 128;      // two d-chunks of [64 keys x 128 B]
constexpr int kPBytes = 128 * 128;          // [128 rows x 64 keys] bf16 (one of the hi / lo halves)
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kQBytes;
constexpr int kOffV = kOffK + kStages * kKBytes;
constexpr int kOffP = kOffV + kStages * kVBytes;
constexpr int kOffBar = kOffP + 4 * kPBytes;  // 2 buffers x (hi, lo)
constexpr int kNumBars = 2 * kStages + 9;
constexpr int kOffMisc = kOffBar + 8 * kNumBars;
constexpr int kSmemBytes = kOffMisc + 64 + 1024;  // + slack for 1024-byte alignment
constexpr uint32_t kTmemCols = 256;         // O: cols [0,128), S0: [128,192), S1: [192,256)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;   // log2 units
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

struct TcParams {
    AttnParams a;
    int dim_s, dim_h;   // tensor-map dimension index of the slot and kv-head axes (1 or 2)
};

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ unsigned long long global_timer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}

// Bounded wait for the phase of parity `parity` to complete.  Gives up when
// another thread of the CTA gave up (abort flag) or after kWaitLimitNs.
__device__ __noinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                       unsigned int *fault) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_timer();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 0) {
            if (*abort_flag) return false;
            if (global_timer() - t0 > kWaitLimitNs) {
                *abort_flag = 1;
                set_fault(fault, FAULT_WAIT_TIMEOUT);
                return false;
            }
        }
    }
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap *map, uint32_t bar, int c0, int c1,
                                            int c2, int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// shared-memory matrix descriptor, 128-byte swizzle, sm_100 descriptor version 1
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// instruction descriptor, kind::f16: bf16 A and B, fp32 D
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool b_mn_major) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

#define SDV_R8(i) "=r"(r[i]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), "=r"(r[i + 4]), \
                  "=r"(r[i + 5]), "=r"(r[i + 6]), "=r"(r[i + 7])
#define SDV_W8(i) "+r"(r[i]), "+r"(r[i + 1]), "+r"(r[i + 2]), "+r"(r[i + 3]), "+r"(r[i + 4]), \
                  "+r"(r[i + 5]), "+r"(r[i + 6]), "+r"(r[i + 7])
#define SDV_S8(i) "r"(r[i]), "r"(r[i + 1]), "r"(r[i + 2]), "r"(r[i + 3]), "r"(r[i + 4]), \
                  "r"(r[i + 5]), "r"(r[i + 6]), "r"(r[i + 7])

// 32 consecutive fp32 columns of this thread's lane; waits for completion
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13,"
        " %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : SDV_R8(0), SDV_R8(8), SDV_R8(16), SDV_R8(24)
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
    // tie the registers to the wait so no use is scheduled above it
    asm volatile("" : SDV_W8(0), SDV_W8(8), SDV_W8(16), SDV_W8(24));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12,"
        " %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};"
        ::"r"(taddr), SDV_S8(0), SDV_S8(8), SDV_S8(16), SDV_S8(24)
        : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}

// byte offset of 16-byte chunk c (0..7) of row r in a [rows x 128 B] tile with 128-byte swizzle
__device__ __forceinline__ uint32_t sw128_off(int r, int c) { return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4)); }

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kTcThreads, 1)
attn_split_tc_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                     const TcParams tp) {
    const AttnParams &p = tp.a;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    const uint32_t base = (raw_u32 + 1023u) & ~1023u;
    uint8_t *sbase = smem_raw + (base - raw_u32);

    const int s = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int T = p.T, G = p.Hq / p.Hkv, M = G * T;
    const bool drafter = p.mode == 1;

    int nb = p.nctx[b];
    if (nb < 1 || nb > p.max_ctx) {
        if (tid == 0) set_fault(p.fault, FAULT_BAD_CTX);
        nb = max(1, min(nb, p.max_ctx));
    }
    const int k0 = s * p.keys_per_split;
    const int k1 = k0 + p.keys_per_split;
    // end of this split's keys taken from the cache (exclusive)
    const int cend = drafter ? min(k1, nb) : min(k1, nb + T - 1);
    const int n_cache_tiles = cend > k0 ? (cend - k0 + kBN - 1) / kBN : 0;
    const bool has_block_tile = drafter && s == 0;
    const int n_tiles = n_cache_tiles + (has_block_tile ? 1 : 0);
    const long rows_total = (long)p.B * T * p.Hq;

    if (n_tiles == 0) {  // nothing to read: mark the split empty for the merge
        if (tid < M) {
            const int j = tid / G, h = g * G + tid % G;
            p.lse_part[(long)s * rows_total + ((long)b * T + j) * p.Hq + h] = -INFINITY;
        }
        return;
    }

    const uint32_t sQ = base + kOffQ, sK = base + kOffK, sV = base + kOffV, sP = base + kOffP;
    const uint32_t bar0 = base + kOffBar;
    auto full_bar = [&](int i) { return bar0 + 8u * i; };
    auto empty_bar = [&](int i) { return bar0 + 8u * (kStages + i); };
    auto sfull_bar = [&](int i) { return bar0 + 8u * (2 * kStages + i); };
    auto sempty_bar = [&](int i) { return bar0 + 8u * (2 * kStages + 2 + i); };
    auto pfull_bar = [&](int i) { return bar0 + 8u * (2 * kStages + 4 + i); };
    auto pempty_bar = [&](int i) { return bar0 + 8u * (2 * kStages + 6 + i); };
    const uint32_t drain_bar = bar0 + 8u * (2 * kStages + 8);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(sbase + kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sbase + kOffMisc + 8);

    // tile t -> first key index (cache tiles) ; the drafter's block tile is t == 0 of split 0
    auto tile_key0 = [&](int t) { return k0 + (t - (has_block_tile ? 1 : 0)) * kBN; };
    auto is_block_tile = [&](int t) { return has_block_tile && t == 0; };

    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) { mbar_init(full_bar(i), 1); mbar_init(empty_bar(i), 1); }
        for (int i = 0; i < 2; ++i) {
            mbar_init(sfull_bar(i), 1); mbar_init(sempty_bar(i), 128);
            mbar_init(pfull_bar(i), 128); mbar_init(pempty_bar(i), 1);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 5) {  // tensor memory for O and the two S buffers
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_holder)), "r"(kTmemCols) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    // Q rows r = j*G + hl of this kv head, zero-padded to 128 rows, 128-byte swizzled
    if (warp < 4) {
        const int r = tid;
        const __nv_bfloat16 *q = static_cast<const __nv_bfloat16 *>(p.q);
        for (int ch = 0; ch < 16; ++ch) {
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (r < M) {
                const int j = r / G, h = g * G + r % G;
                v = __ldg(reinterpret_cast<const uint4 *>(q + (((long)b * T + j) * p.Hq + h) * 128) + ch);
            }
            *reinterpret_cast<uint4 *>(sbase + kOffQ + (ch >> 3) * (128 * 128) + sw128_off(r, ch & 7)) = v;
        }
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
#if __CUDA_ARCH__ >= 900
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
#endif

    if (warp == 4) {
        // ------------------------------------------------------------------ producer
        const __nv_bfloat16 *kb = static_cast<const __nv_bfloat16 *>(p.kb);
        const __nv_bfloat16 *vb = static_cast<const __nv_bfloat16 *>(p.vb);
        int issued = 0;
        for (int t = 0; t < n_tiles; ++t) {
            const int st = t % kStages;
            if (t >= kStages && !mbar_wait(empty_bar(st), ((t / kStages) - 1) & 1, abort_flag, p.fault)) break;
            const uint32_t dK = sK + st * kKBytes, dV = sV + st * kVBytes;
            if (is_block_tile(t)) {
                // the T block keys / values from [B, T, Hkv, D], rows >= T zero
                for (int idx = lane; idx < kBN * 16; idx += 32) {
                    const int row = idx >> 4, ch = idx & 15;
                    uint4 kv4 = make_uint4(0u, 0u, 0u, 0u), vv4 = make_uint4(0u, 0u, 0u, 0u);
                    if (row < T) {
                        const long off = (((long)b * T + row) * p.Hkv + g) * 128;
                        kv4 = __ldg(reinterpret_cast<const uint4 *>(kb + off) + ch);
                        vv4 = __ldg(reinterpret_cast<const uint4 *>(vb + off) + ch);
                    }
                    const uint32_t o = (ch >> 3) * (kBN * 128) + sw128_off(row, ch & 7);
                    *reinterpret_cast<uint4 *>(sbase + kOffK + st * kKBytes + o) = kv4;
                    *reinterpret_cast<uint4 *>(sbase + kOffV + st * kVBytes + o) = vv4;
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(full_bar(st));
            } else if (lane == 0) {
                const int key0 = tile_key0(t);
                int c[4] = {0, 0, 0, b};
                c[tp.dim_s] = key0;
                c[tp.dim_h] = g;
                mbar_arrive_expect_tx(full_bar(st), (uint32_t)(kKBytes + kVBytes));
                tma_load_4d(dK, &tmap_k, full_bar(st), 0, c[1], c[2], c[3]);
                tma_load_4d(dK + kBN * 128, &tmap_k, full_bar(st), 64, c[1], c[2], c[3]);
                tma_load_4d(dV, &tmap_v, full_bar(st), 0, c[1], c[2], c[3]);
                tma_load_4d(dV + kBN * 128, &tmap_v, full_bar(st), 64, c[1], c[2], c[3]);
            }
            __syncwarp();
            issued = t + 1;
        }
        // on abort: let the copies already issued land before the CTA exits
        if (*abort_flag && lane == 0) {
            for (int t = max(0, issued - kStages); t < issued; ++t) {
                volatile int never = 0;
                mbar_wait(full_bar(t % kStages), (t / kStages) & 1, &never, p.fault);
            }
        }
    } else if (warp == 5) {
        // ------------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idS = idesc_bf16(128, kBN, false);
            const uint32_t idO = idesc_bf16(128, 128, true);
            auto issue_S = [&](int t) {
                const int st = t % kStages;
                const uint32_t dcol = tmem + 128u + 64u * (t & 1);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint64_t a = sw128_desc(sQ + (kk >> 2) * (128 * 128) + (kk & 3) * 32, 16, 1024);
                    const uint64_t bd = sw128_desc(sK + st * kKBytes + (kk >> 2) * (kBN * 128) + (kk & 3) * 32, 16, 1024);
                    umma_bf16(dcol, a, bd, idS, kk > 0 ? 1u : 0u);
                }
                umma_commit(sfull_bar(t & 1));
            };
            bool ok = mbar_wait(full_bar(0), 0, abort_flag, p.fault);
            if (ok) { tc_fence_after(); issue_S(0); }
            for (int t = 0; ok && t < n_tiles; ++t) {
                if (t + 1 < n_tiles) {
                    const int t1 = t + 1;
                    ok = mbar_wait(full_bar(t1 % kStages), (t1 / kStages) & 1, abort_flag, p.fault);
                    if (ok && t1 >= 2) ok = mbar_wait(sempty_bar(t1 & 1), ((t1 - 2) >> 1) & 1, abort_flag, p.fault);
                    if (!ok) break;
                    tc_fence_after();
                    issue_S(t1);
                }
                ok = mbar_wait(pfull_bar(t & 1), (t >> 1) & 1, abort_flag, p.fault);
                if (!ok) break;
                tc_fence_after();
                const int st = t % kStages;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t a = sw128_desc(sP + ((t & 1) * 2 + half) * kPBytes + kk * 32, 16, 1024);
                        const uint64_t bd = sw128_desc(sV + st * kVBytes + kk * 16 * 128, kBN * 128, 1024);
                        umma_bf16(tmem, a, bd, idO, (t > 0 || half > 0 || kk > 0) ? 1u : 0u);
                    }
                }
                umma_commit(pempty_bar(t & 1));
                umma_commit(empty_bar(st));
            }
            // every MMA issued above has completed before tensor memory is freed
            umma_commit(drain_bar);
            volatile int never = 0;
            mbar_wait(drain_bar, 0, &never, p.fault);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------------ softmax (warps 0-3)
        const int r = tid;                      // query row = tensor-memory lane
        const bool row_ok = r < M;
        const int j = row_ok ? r / G : 0;
        const float qk = p.scale * kLog2e;
        const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
        float m_used = -INFINITY, l = 0.f;
        bool ok = true;
        for (int t = 0; t < n_tiles && ok; ++t) {
            ok = __all_sync(0xffffffffu, mbar_wait(sfull_bar(t & 1), (t >> 1) & 1, abort_flag, p.fault));
            if (!ok) break;
            tc_fence_after();
            uint32_t sr[64];
            {
                uint32_t (&lo)[32] = *reinterpret_cast<uint32_t (*)[32]>(&sr[0]);
                uint32_t (&hi)[32] = *reinterpret_cast<uint32_t (*)[32]>(&sr[32]);
                tmem_ld32(lane_base + 128u + 64u * (t & 1), lo);
                tmem_ld32(lane_base + 128u + 64u * (t & 1) + 32u, hi);
            }
            tc_fence_before();
            mbar_arrive(sempty_bar(t & 1));

            // mask: keys this row may see in this tile
            const bool blk = is_block_tile(t);
            int nvalid;  // keys [0, nvalid) of the tile are visible to this row
            if (blk) {
                nvalid = T;
            } else {
                const int key0 = tile_key0(t);
                const int lim = drafter ? cend : min(cend, nb + j);
                nvalid = max(0, min(kBN, lim - key0));
            }
            if (!row_ok) nvalid = 0;
            float x[64];
            float tmax = -INFINITY;
#pragma unroll
            for (int c = 0; c < 64; ++c) {
                x[c] = c < nvalid ? __uint_as_float(sr[c]) * qk : -INFINITY;
                tmax = fmaxf(tmax, x[c]);
            }
            // move the reference max only when it grows by more than 2^8
            const bool need = t > 0 && tmax > m_used + kRescaleThreshold;
            float alpha = 1.f;
            float m_new = m_used;
            if (t == 0) m_new = tmax;
            else if (need) { m_new = tmax; alpha = ex2(m_used - m_new); }
            if (__any_sync(0xffffffffu, need)) {
                // O is read-modify-written in tensor memory once PV_{t-1} is complete
                ok = mbar_wait(pempty_bar((t - 1) & 1), ((t - 1) >> 1) & 1, abort_flag, p.fault);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                tc_fence_after();
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    uint32_t o[32];
                    tmem_ld32(lane_base + 32u * cc, o);
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                    tmem_st32(lane_base + 32u * cc, o);
                }
                tc_fence_before();
            }
            m_used = m_new;
            l *= alpha;
            const bool live = m_used != -INFINITY;
            uint32_t pk[32], pl[32];
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                const float p0 = live ? ex2(x[2 * c] - m_used) : 0.f;
                const float p1 = live ? ex2(x[2 * c + 1] - m_used) : 0.f;
                l += p0 + p1;
                pk[c] = pack_bf16(p0, p1);
                // residual after rounding to bf16 (exact in fp32), itself rounded to bf16
                const float r0 = p0 - __uint_as_float(pk[c] << 16);
                const float r1 = p1 - __uint_as_float(pk[c] & 0xffff0000u);
                pl[c] = pack_bf16(r0, r1);
            }
            // P buffer (t & 1) is free once PV_{t-2} completed
            if (t >= 2) {
                ok = __all_sync(0xffffffffu, mbar_wait(pempty_bar(t & 1), ((t - 2) >> 1) & 1, abort_flag, p.fault));
                if (!ok) break;
            }
            uint8_t *pb = sbase + kOffP + (t & 1) * 2 * kPBytes;
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
                *reinterpret_cast<uint4 *>(pb + sw128_off(r, ch)) =
                    make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
                *reinterpret_cast<uint4 *>(pb + kPBytes + sw128_off(r, ch)) =
                    make_uint4(pl[4 * ch], pl[4 * ch + 1], pl[4 * ch + 2], pl[4 * ch + 3]);
            }
            // value rows past the last cache key of the split may hold anything: zero them
            if (!blk) {
                const int v0 = max(0, min(kBN, cend - tile_key0(t)));
                if (v0 < kBN) {
                    uint8_t *vt = sbase + kOffV + (t % kStages) * kVBytes;
                    for (int idx = tid; idx < (kBN - v0) * 16; idx += 128) {
                        const int row = v0 + (idx >> 4), ch = idx & 15;
                        *reinterpret_cast<uint4 *>(vt + (ch >> 3) * (kBN * 128) + sw128_off(row, ch & 7)) =
                            make_uint4(0u, 0u, 0u, 0u);
                    }
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(pfull_bar(t & 1));
        }
        // epilogue: O / l and the log-sum-exp of this split
        if (ok) ok = mbar_wait(pempty_bar((n_tiles - 1) & 1), ((n_tiles - 1) >> 1) & 1, abort_flag, p.fault);
        ok = __all_sync(0xffffffffu, ok);
        if (ok) {
            tc_fence_after();
            const float inv = l > 0.f ? 1.f / l : 0.f;
            const int h = g * G + (row_ok ? r % G : 0);
            const long frow = ((long)b * T + j) * p.Hq + h;
            float *dst = p.o_part + ((long)s * rows_total + frow) * 128;
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                uint32_t o[32];
                tmem_ld32(lane_base + 32u * cc, o);
                if (row_ok) {
#pragma unroll
                    for (int e = 0; e < 32; e += 4)
                        *reinterpret_cast<float4 *>(dst + 32 * cc + e) =
                            make_float4(__uint_as_float(o[e]) * inv, __uint_as_float(o[e + 1]) * inv,
                                        __uint_as_float(o[e + 2]) * inv, __uint_as_float(o[e + 3]) * inv);
                }
            }
            if (row_ok)
                p.lse_part[(long)s * rows_total + frow] = l > 0.f ? m_used * kLn2 + logf(l) : -INFINITY;
        }
        tc_fence_before();
    }

    // teardown: wait for every MMA of this CTA, then free tensor memory
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                     : "memory");
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

// 4-D map over a [B, S, Hkv, D] bf16 tensor with element strides kv; the slot
// and head axes are ordered by stride.  Box: 64 d x 64 slots x 1 head x 1 seq.
bool make_map(CUtensorMap *m, const void *ptr, const sd_strides &kv, int S, int Hkv, int B, int *dim_s,
              int *dim_h) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn) return false;
    const bool s_inner = kv.s <= kv.h;
    *dim_s = s_inner ? 1 : 2;
    *dim_h = s_inner ? 2 : 1;
    cuuint64_t dims[4], strides[3];
    cuuint32_t box[4], estr[4] = {1, 1, 1, 1};
    dims[0] = 128;
    dims[*dim_s] = (cuuint64_t)S;
    dims[*dim_h] = (cuuint64_t)Hkv;
    dims[3] = (cuuint64_t)B;
    strides[*dim_s - 1] = (cuuint64_t)kv.s * 2;
    strides[*dim_h - 1] = (cuuint64_t)kv.h * 2;
    strides[2] = (cuuint64_t)kv.b * 2;
    box[0] = 64;
    box[*dim_s] = kBN;
    box[*dim_h] = 1;
    box[3] = 1;
    const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(ptr), dims, strides, box,
                          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

int cache_slots(const AttnParams &p) { return p.mode == 0 ? p.max_ctx + p.T - 1 : p.max_ctx; }

}  // namespace

bool attn_tc_supported(const AttnParams &p) {
    if (p.dt != SD_BF16 || p.D != 128 || p.T < 1 || p.T > kMaxT) return false;
    if ((p.Hq / p.Hkv) * p.T > 128) return false;
    if ((long)p.max_ctx + p.T > (1L << 30)) return false;
    if (!encode_fn()) return false;
    int dev = 0, optin = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return false;
    if (optin < kSmemBytes) return false;
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    return major == 10 && minor == 3;
}

size_t attn_tc_smem_bytes(const AttnParams &) { return kSmemBytes; }

cudaError_t launch_attn_tc(const AttnParams &p, cudaStream_t st) {
    alignas(64) CUtensorMap mk, mv;
    TcParams tp;
    tp.a = p;
    int ds2 = 0, dh2 = 0;
    if (!make_map(&mk, p.kc, p.kv, cache_slots(p), p.Hkv, p.B, &tp.dim_s, &tp.dim_h)) return cudaErrorInvalidValue;
    if (!make_map(&mv, p.vc, p.kv, cache_slots(p), p.Hkv, p.B, &ds2, &dh2)) return cudaErrorInvalidValue;
    static bool opted_in[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !opted_in[dev]) {
        e = cudaFuncSetAttribute(attn_split_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) opted_in[dev] = true;
    }
    dim3 grid(p.n_splits, p.Hkv, p.B);
    attn_split_tc_kernel<<<grid, kTcThreads, kSmemBytes, st>>>(mk, mv, tp);
    return cudaGetLastError();
}

}  // namespace sdv
