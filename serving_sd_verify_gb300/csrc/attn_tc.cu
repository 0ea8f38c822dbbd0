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
// tile is fetched from HBM once and serves every row.  For key tile t:
//   S_t = Q . K_t^T                       (M 128, N 64 keys, K 128)
//   P_t = exp2(S_t * scale * log2e - m)   split as P_hi + P_lo, both bf16
//   O_(t mod 2) += P_hi . V_t + P_lo . V_t  (M 128, N 128, K 64)
// The two-term split keeps every weight to within 2^-14 relative, so the
// product is as accurate as an fp32 P even when a few keys dominate.
//
// Warp roles (352 threads):
//   warps 0-3 / 4-7  two softmax warpgroups; warpgroup w takes the tiles with
//                    t mod 2 == w, has two S/P buffers and its own O
//                    accumulator in tensor memory and its own running max /
//                    sum; thread = row (= tensor-memory lane).  The two halves
//                    are merged at the end like two splits.
//   warp 8           TMA producer: Q first, then a K/V ring in shared memory
//   warp 9           allocates tensor memory; one thread issues the S MMAs
//   warp 10          one thread issues the P.V MMAs
// The two issuers each wait only on their own barriers, so a finished softmax
// never waits behind the issue of the next S (or the other way round).
// Tensor memory: O0 [0,128), O1 [128,256), three S/P buffers of 64 columns
// and Q (64 columns, the A operand of every S, so S reads only K from shared
// memory); tile t uses buffer t mod 3, so S of the next tiles is computed
// while P.V of tile t is still pending.  P is written back into the columns that held S
// (variant kPTmem) and read by the MMA as its A operand, which leaves shared
// memory to a 6-stage K/V ring; the other variant stages P through shared
// memory.  The partial output leaves through shared memory so that the global
// stores are coalesced.
// The running max only moves when it grows by more than 2^8, so O is rescaled
// in tensor memory rarely (exact either way: P and l use the same reference).
// Every wait is bounded by the global timer; a wait that gives up sets the
// fault word and the CTA drains its copies and MMAs before freeing tensor
// memory and returning.
#include "common.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>

#include <math.h>
#include <string.h>

namespace sdv {

namespace {

constexpr int kTcThreads = 352;
constexpr int kBN = kTileKeys;              // keys per tile (64)
constexpr int kQBytes = 2 * 128 * 128;      // two K-blocks of [128 rows x 128 B]
constexpr int kKBytes = 2 * kBN * 128;      // two K-blocks of [64 keys x 128 B]
constexpr int kVBytes = 2 * kBN * 128;      // two d-chunks of [64 keys x 128 B]
constexpr int kStageBytes = kKBytes + kVBytes;
constexpr int kPBytes = 128 * 128;          // [128 rows x 64 keys] bf16, one half (hi or lo)
constexpr uint32_t kTmemCols = 512;         // O0 [0,128) O1 [128,256) SP0..SP2 [256 + 64 i, +64) Q [448,512)
constexpr int kSP = 3;                      // S/P buffers in tensor memory
constexpr uint32_t kQCol = 448;             // Q as the A operand of S: bf16 pairs, 64 columns
constexpr int kOStride = 132;               // floats per staged output row (bank-conflict padding)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;   // log2 units
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

template <bool kPTmem> struct Layout {
    static constexpr int kStages = kPTmem ? 6 : 3;
    static constexpr int kOffQ = 0;
    static constexpr int kOffStage = kQBytes;
    static constexpr int kOffP = kOffStage + kStages * kStageBytes;          // smem P (variant 2 only)
    static constexpr int kOffBar = kOffP + (kPTmem ? 0 : 4 * kPBytes);
    // full[S], empty[S], sfull[3], pfull[3], pempty[3], qready, qtmem, drain x2
    static constexpr int kNumBars = 2 * kStages + 3 * kSP + 4;
    static constexpr int kOffMisc = kOffBar + 8 * kNumBars;                  // tmem base, abort flag
    static constexpr int kOffXchg = kOffQ;  // (m, l) exchange, in the Q tile once every MMA is done
    static constexpr int kSmemBytes = kOffMisc + 16 + 1024;                  // + alignment slack
};

struct TcParams {
    AttnParams a;
    int dim_s, dim_h;   // tensor-map dimension index of the slot and kv-head axes (1 or 2)
};
static_assert(128 * kOStride * 4 <= 5 * (2 * 64 * 128 * 2), "output staging fits in the K/V ring");

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
// another thread of the CTA gave up (abort flag, if given) or after kWaitLimitNs.
__device__ __noinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                       unsigned int *fault) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_timer();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 0) {
            if (abort_flag && *abort_flag) return false;
            if (global_timer() - t0 > kWaitLimitNs) {
                if (abort_flag) *abort_flag = 1;
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
__device__ __forceinline__ void named_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

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

// instruction descriptor, kind::f16: bf16 A and B, fp32 D, A K-major
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool b_mn_major) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// D (tensor memory) (+)= A (shared memory, descriptor) . B (shared memory)
__device__ __forceinline__ void umma_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                        uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// D (tensor memory) (+)= A (tensor memory) . B (shared memory)
__device__ __forceinline__ void umma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                        uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
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

// 32 consecutive 32-bit columns of this thread's lane; completes at tmem_ld_wait
__device__ __forceinline__ void tmem_ld32_async(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13,"
        " %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : SDV_R8(0), SDV_R8(8), SDV_R8(16), SDV_R8(24)
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// ties registers filled by tmem_ld32_async to the preceding wait
__device__ __forceinline__ void tmem_ld_bind(uint32_t (&r)[32]) {
    asm volatile("" : SDV_W8(0), SDV_W8(8), SDV_W8(16), SDV_W8(24));
}

// 64 consecutive columns: both loads in flight before the single wait
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t (&r)[64]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13,"
        " %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31,"
        " %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47,"
        " %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];"
        : SDV_R8(0), SDV_R8(8), SDV_R8(16), SDV_R8(24), SDV_R8(32), SDV_R8(40), SDV_R8(48), SDV_R8(56)
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
    asm volatile("" : SDV_W8(0), SDV_W8(8), SDV_W8(16), SDV_W8(24), SDV_W8(32), SDV_W8(40), SDV_W8(48),
                 SDV_W8(56));
}
// store without waiting (callers issue tmem_st_wait once after a batch)
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12,"
        " %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};"
        ::"r"(taddr), SDV_S8(0), SDV_S8(8), SDV_S8(16), SDV_S8(24)
        : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// byte offset of 16-byte chunk c (0..7) of row r in a [rows x 128 B] tile with 128-byte swizzle
__device__ __forceinline__ uint32_t sw128_off(int r, int c) { return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4)); }

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
template <bool kPTmem>
__global__ void __launch_bounds__(kTcThreads, 1)
attn_split_tc_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                     const __grid_constant__ CUtensorMap tmap_v, const TcParams tp) {
    using L = Layout<kPTmem>;
    constexpr int NS = L::kStages;
    const AttnParams &p = tp.a;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    const uint32_t base = (raw_u32 + 1023u) & ~1023u;
    uint8_t *sbase = smem_raw + (base - raw_u32);

    const int s = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    const uint32_t sQ = base + L::kOffQ, sStage = base + L::kOffStage, sP = base + L::kOffP;
    const uint32_t bar0 = base + L::kOffBar;
    auto full_bar = [&](int i) { return bar0 + 8u * i; };
    auto empty_bar = [&](int i) { return bar0 + 8u * (NS + i); };
    auto sfull_bar = [&](int i) { return bar0 + 8u * (2 * NS + i); };
    auto pfull_bar = [&](int i) { return bar0 + 8u * (2 * NS + kSP + i); };
    auto pempty_bar = [&](int i) { return bar0 + 8u * (2 * NS + 2 * kSP + i); };
    const uint32_t qready_bar = bar0 + 8u * (2 * NS + 3 * kSP);
    const uint32_t qtmem_bar = bar0 + 8u * (2 * NS + 3 * kSP + 1);
    const uint32_t drain_bar = bar0 + 8u * (2 * NS + 3 * kSP + 2);
    const uint32_t drain2_bar = bar0 + 8u * (2 * NS + 3 * kSP + 3);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(sbase + L::kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sbase + L::kOffMisc + 8);
    float2 *xchg = reinterpret_cast<float2 *>(sbase + L::kOffXchg);  // [2][128] (m, l) per warpgroup

    // ---- prologue that reads nothing produced upstream ----
    if (tid == 0) {
        for (int i = 0; i < NS; ++i) { mbar_init(full_bar(i), 1); mbar_init(empty_bar(i), 1); }
        for (int i = 0; i < kSP; ++i) { mbar_init(sfull_bar(i), 1); mbar_init(pfull_bar(i), 4); mbar_init(pempty_bar(i), 1); }
        mbar_init(qready_bar, 1);  // the Q copy, with its bytes
        mbar_init(qtmem_bar, 4);   // the four warps that move Q into tensor memory
        mbar_init(drain_bar, 1);
        mbar_init(drain2_bar, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 9) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_holder)), "r"(kTmemCols) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
#if __CUDA_ARCH__ >= 900
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");  // inputs of an upstream kernel are visible now
#endif

    const int T = p.T, G = p.Hq / p.Hkv, M = G * T;
    const bool drafter = p.mode == 1;
    int nb = p.nctx[b];
    if (nb < 1 || nb > p.max_ctx) {
        if (tid == 0) set_fault(p.fault, FAULT_BAD_CTX);
        nb = max(1, min(nb, p.max_ctx));
    }
    const int k0 = s * p.keys_per_split;
    const int k1 = k0 + p.keys_per_split;
    const int cend = drafter ? min(k1, nb) : min(k1, nb + T - 1);  // end of this split's cache keys
    const int n_cache_tiles = cend > k0 ? (cend - k0 + kBN - 1) / kBN : 0;
    const bool has_block_tile = drafter && s == 0;
    const int n_tiles = n_cache_tiles + (has_block_tile ? 1 : 0);
    const long rows_total = (long)p.B * T * p.Hq;
    auto tile_key0 = [&](int t) { return k0 + (t - (has_block_tile ? 1 : 0)) * kBN; };
    auto is_block_tile = [&](int t) { return has_block_tile && t == 0; };

    if (n_tiles == 0) {
        // nothing to read: an empty split (lse = -inf, zero partial) for the merge
        for (int idx = tid; idx < M * 32; idx += kTcThreads) {
            const int rr = idx >> 5, c4 = idx & 31;
            const long frow = ((long)b * T + rr / G) * p.Hq + g * G + rr % G;
            reinterpret_cast<float4 *>(p.o_part + ((long)s * rows_total + frow) * 128)[c4] =
                make_float4(0.f, 0.f, 0.f, 0.f);
            if (c4 == 0) p.lse_part[(long)s * rows_total + frow] = -INFINITY;
        }
    } else if (warp == 8) {
        // ------------------------------------------------------------------ producer
        if (lane == 0) {
            // Q first: rows r = j*G + hl of this kv head, two 64-column halves
            mbar_arrive_expect_tx(qready_bar, (uint32_t)(256 * M));
            tma_load_4d(sQ, &tmap_q, qready_bar, 0, g * G, 0, b);
            tma_load_4d(sQ + 128 * 128, &tmap_q, qready_bar, 64, g * G, 0, b);
        }
        int t = 0;
        if (has_block_tile) {
            // the T block keys / values from [B, T, Hkv, D] into stage 0; rows >= T zero
            const __nv_bfloat16 *kb = static_cast<const __nv_bfloat16 *>(p.kb);
            const __nv_bfloat16 *vb = static_cast<const __nv_bfloat16 *>(p.vb);
            uint8_t *stg = sbase + L::kOffStage;
            for (int idx = lane; idx < kBN * 16; idx += 32) {
                const int row = idx >> 4, ch = idx & 15;
                uint4 kv4 = make_uint4(0u, 0u, 0u, 0u), vv4 = make_uint4(0u, 0u, 0u, 0u);
                if (row < T) {
                    const long off = (((long)b * T + row) * p.Hkv + g) * 128;
                    kv4 = __ldg(reinterpret_cast<const uint4 *>(kb + off) + ch);
                    vv4 = __ldg(reinterpret_cast<const uint4 *>(vb + off) + ch);
                }
                const uint32_t o = (ch >> 3) * (kBN * 128) + sw128_off(row, ch & 7);
                *reinterpret_cast<uint4 *>(stg + o) = kv4;
                *reinterpret_cast<uint4 *>(stg + kKBytes + o) = vv4;
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(full_bar(0));
            t = 1;
        }
        int issued = t;
        if (lane == 0) {
            for (; t < n_tiles; ++t) {
                const int st = t % NS;
                if (t >= NS && !mbar_wait(empty_bar(st), ((t / NS) - 1) & 1, abort_flag, p.fault)) break;
                const uint32_t dK = sStage + st * kStageBytes, dV = dK + kKBytes;
                int c[4] = {0, 0, 0, b};
                c[tp.dim_s] = tile_key0(t);
                c[tp.dim_h] = g;
                mbar_arrive_expect_tx(full_bar(st), (uint32_t)kStageBytes);
                tma_load_4d(dK, &tmap_k, full_bar(st), 0, c[1], c[2], c[3]);
                tma_load_4d(dK + kBN * 128, &tmap_k, full_bar(st), 64, c[1], c[2], c[3]);
                tma_load_4d(dV, &tmap_v, full_bar(st), 0, c[1], c[2], c[3]);
                tma_load_4d(dV + kBN * 128, &tmap_v, full_bar(st), 64, c[1], c[2], c[3]);
                issued = t + 1;
            }
            // on abort: let the copies already issued land before the CTA exits
            if (*abort_flag) {
                mbar_wait(qready_bar, 0, nullptr, p.fault);
                for (int u = max(0, issued - NS); u < issued; ++u)
                    mbar_wait(full_bar(u % NS), (u / NS) & 1, nullptr, p.fault);
            }
        }
        __syncwarp();
    } else if (warp == 9) {
        // ------------------------------------------------------------------ S issuer
        if (lane == 0) {
            const uint32_t idS = idesc_bf16(128, kBN, false);
            bool ok = mbar_wait(qtmem_bar, 0, abort_flag, p.fault);
            for (int t = 0; ok && t < n_tiles; ++t) {
                // K of tile t loaded, and buffer t % 3 consumed by the P.V of tile t-3
                const int bi = t % kSP;
                ok = mbar_wait(full_bar(t % NS), (t / NS) & 1, abort_flag, p.fault);
                if (ok && t >= kSP) ok = mbar_wait(pempty_bar(bi), ((t / kSP) - 1) & 1, abort_flag, p.fault);
                if (!ok) break;
                tc_fence_after();
                const uint32_t dcol = tmem + 256u + 64u * bi;
                const uint32_t kbase = sStage + (t % NS) * kStageBytes;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint64_t bd = sw128_desc(kbase + (kk >> 2) * (kBN * 128) + (kk & 3) * 32, 16, 1024);
                    umma_ts(dcol, tmem + kQCol + 8u * kk, bd, idS, kk > 0 ? 1u : 0u);
                }
                umma_commit(sfull_bar(bi));
            }
            // every MMA this thread issued has completed before tensor memory is freed
            umma_commit(drain_bar);
            mbar_wait(drain_bar, 0, nullptr, p.fault);
        }
        __syncwarp();
    } else if (warp == 10) {
        // ------------------------------------------------------------------ P.V issuer
        if (lane == 0) {
            const uint32_t idO = idesc_bf16(128, 128, true);
            bool ok = true;
            for (int t = 0; ok && t < n_tiles; ++t) {
                ok = mbar_wait(pfull_bar(t % kSP), (t / kSP) & 1, abort_flag, p.fault);
                if (!ok) break;
                tc_fence_after();
                const int st = t % NS;
                const int wb = t & 1;
                const uint32_t vbase = sStage + st * kStageBytes + kKBytes;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t bd = sw128_desc(vbase + kk * 16 * 128, kBN * 128, 1024);
                        const uint32_t acc = (t >= 2 || half > 0 || kk > 0) ? 1u : 0u;
                        if (kPTmem) {
                            const uint32_t a_t = tmem + 256u + 64u * (t % kSP) + 32u * half + 8u * kk;
                            umma_ts(tmem + 128u * wb, a_t, bd, idO, acc);
                        } else {
                            const uint64_t a = sw128_desc(sP + (wb * 2 + half) * kPBytes + kk * 32, 16, 1024);
                            umma_ss(tmem + 128u * wb, a, bd, idO, acc);
                        }
                    }
                }
                umma_commit(pempty_bar(t % kSP));
                umma_commit(empty_bar(st));
            }
            umma_commit(drain2_bar);
            mbar_wait(drain2_bar, 0, nullptr, p.fault);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------------ softmax (warps 0-7)
        const int wg = warp >> 2;               // warpgroup: tiles t with t % 2 == wg
        const int r = tid & 127;                // query row = tensor-memory lane
        const bool row_ok = r < M;
        const int j = row_ok ? r / G : 0;
        const float qk = p.scale * kLog2e;
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t o_col = tmem + lane_off + 128u * wg;
        if (wg == 0) {
            // Q into tensor memory (the A operand of S): row r = lane r, bf16
            // pairs along K; rows past the M real ones are zero
            const bool qok = __all_sync(0xffffffffu, mbar_wait(qready_bar, 0, abort_flag, p.fault));
            uint32_t qa[32], qb[32];
#pragma unroll
            for (int ch = 0; ch < 16; ++ch) {
                uint4 v = make_uint4(0u, 0u, 0u, 0u);
                if (row_ok && qok)
                    v = *reinterpret_cast<const uint4 *>(sbase + L::kOffQ + (ch >> 3) * (128 * 128) + sw128_off(r, ch & 7));
                uint32_t *dst = ch < 8 ? &qa[4 * ch] : &qb[4 * (ch - 8)];
                dst[0] = v.x; dst[1] = v.y; dst[2] = v.z; dst[3] = v.w;
            }
            tmem_st32(tmem + lane_off + kQCol, qa);
            tmem_st32(tmem + lane_off + kQCol + 32u, qb);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(qtmem_bar);
        }

        float m_used = -INFINITY, l = 0.f;
        bool ok = true;
        int last_t = -1;
        for (int t = wg; t < n_tiles; t += 2) {
            const int bi = t % kSP;  // S/P buffer
            const int u = t / kSP;   // use index of that buffer
            const uint32_t sp_col = tmem + lane_off + 256u + 64u * bi;
            ok = __all_sync(0xffffffffu, mbar_wait(sfull_bar(bi), u & 1, abort_flag, p.fault));
            if (!ok) break;
            tc_fence_after();
            uint32_t sr[64];
            tmem_ld64(sp_col, sr);
            // keys [0, nvalid) of the tile are visible to this row
            const bool blk = is_block_tile(t);
            int nvalid;
            if (blk) {
                nvalid = T;
            } else {
                const int lim = drafter ? cend : min(cend, nb + j);
                nvalid = max(0, min(kBN, lim - tile_key0(t)));
            }
            if (!row_ok) nvalid = 0;
            // tile max of the raw scores (qk > 0 keeps the order)
            float mx[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                float m8 = -INFINITY;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int c = 8 * i + e;
                    m8 = fmaxf(m8, c < nvalid ? __uint_as_float(sr[c]) : -INFINITY);
                }
                mx[i] = m8;
            }
            const float smax = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                     fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
            const float tmax = smax * qk;
            // move the reference max only when it grows by more than 2^8
            const bool first = t == wg;
            const bool need = !first && tmax > m_used + kRescaleThreshold;
            float alpha = 1.f;
            if (first) m_used = tmax;
            else if (need) { alpha = ex2(m_used - tmax); m_used = tmax; }
            // this warpgroup's previous P.V (tile t-2) must be done before O or
            // (shared-memory variant) the P buffer is touched again
            if (!first && (!kPTmem || __any_sync(0xffffffffu, need))) {
                ok = __all_sync(0xffffffffu,
                                mbar_wait(pempty_bar((t - 2) % kSP), ((t - 2) / kSP) & 1, abort_flag, p.fault));
                if (!ok) break;
                tc_fence_after();
            }
            if (__any_sync(0xffffffffu, need)) {
#pragma unroll
                for (int cc = 0; cc < 4; cc += 2) {
                    uint32_t oa[32], ob[32];
                    tmem_ld32_async(o_col + 32u * cc, oa);
                    tmem_ld32_async(o_col + 32u * (cc + 1), ob);
                    tmem_ld_wait();
                    tmem_ld_bind(oa);
                    tmem_ld_bind(ob);
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        oa[e] = __float_as_uint(__uint_as_float(oa[e]) * alpha);
                        ob[e] = __float_as_uint(__uint_as_float(ob[e]) * alpha);
                    }
                    tmem_st32(o_col + 32u * cc, oa);
                    tmem_st32(o_col + 32u * (cc + 1), ob);
                }
            }
            l *= alpha;
            const bool live = m_used != -INFINITY;
            const float neg_m = live ? -m_used : 0.f;
            uint32_t pk[32], pl[32];
            float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                const float e0 = ex2(fmaf(__uint_as_float(sr[2 * c]), qk, neg_m));
                const float e1 = ex2(fmaf(__uint_as_float(sr[2 * c + 1]), qk, neg_m));
                const float p0 = (live && 2 * c < nvalid) ? e0 : 0.f;
                const float p1 = (live && 2 * c + 1 < nvalid) ? e1 : 0.f;
                ls[c & 3] += p0 + p1;
                // hi = p truncated to bf16; lo = the exact fp32 remainder truncated
                // to bf16: |p - hi - lo| < 2^-14 p.  Byte permutes instead of
                // conversion instructions.
                const uint32_t b0 = __float_as_uint(p0), b1 = __float_as_uint(p1);
                pk[c] = __byte_perm(b0, b1, 0x7632);
                const uint32_t q0 = __float_as_uint(p0 - __uint_as_float(b0 & 0xffff0000u));
                const uint32_t q1 = __float_as_uint(p1 - __uint_as_float(b1 & 0xffff0000u));
                pl[c] = __byte_perm(q0, q1, 0x7632);
            }
            l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
            if (kPTmem) {
                // P over the S columns it came from: hi in [0,32), lo in [32,64)
                tmem_st32(sp_col, pk);
                tmem_st32(sp_col + 32u, pl);
            } else {
                uint8_t *pb = sbase + L::kOffP + wg * 2 * kPBytes;
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    *reinterpret_cast<uint4 *>(pb + sw128_off(r, ch)) =
                        make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
                    *reinterpret_cast<uint4 *>(pb + kPBytes + sw128_off(r, ch)) =
                        make_uint4(pl[4 * ch], pl[4 * ch + 1], pl[4 * ch + 2], pl[4 * ch + 3]);
                }
            }
            // value rows past the split's last cache key may hold anything: zero them
            if (!blk) {
                const int v0 = max(0, min(kBN, cend - tile_key0(t)));
                if (v0 < kBN) {
                    uint8_t *vt = sbase + L::kOffStage + (t % NS) * kStageBytes + kKBytes;
                    for (int idx = r; idx < (kBN - v0) * 16; idx += 128) {
                        const int row = v0 + (idx >> 4), ch = idx & 15;
                        *reinterpret_cast<uint4 *>(vt + (ch >> 3) * (kBN * 128) + sw128_off(row, ch & 7)) =
                            make_uint4(0u, 0u, 0u, 0u);
                    }
                }
            }
            tmem_st_wait();
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(pfull_bar(bi));
            last_t = t;
        }
        // ---- epilogue: merge the two warpgroups' (m, l, O), write this split's partial ----
        if (ok && last_t >= 0)
            ok = mbar_wait(pempty_bar(last_t % kSP), (last_t / kSP) & 1, abort_flag, p.fault);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok || last_t < 0) { m_used = -INFINITY; l = 0.f; }
        tc_fence_before();
        // both warpgroups' last P.V, hence every MMA of the CTA, are complete past
        // this point: the Q tile is free for the (m, l) exchange
        named_sync(1, 256);
        xchg[wg * 128 + r] = make_float2(m_used, l);
        named_sync(1, 256);
        const float2 mine = xchg[wg * 128 + r], other = xchg[(wg ^ 1) * 128 + r];
        const float m0 = wg == 0 ? mine.x : other.x, l0 = wg == 0 ? mine.y : other.y;
        const float m1 = wg == 0 ? other.x : mine.x, l1 = wg == 0 ? other.y : mine.y;
        const float Mx = fmaxf(m0, m1);
        const float f0 = l0 > 0.f ? ex2(m0 - Mx) : 0.f;
        const float f1 = l1 > 0.f ? ex2(m1 - Mx) : 0.f;
        const float Lsum = l0 * f0 + l1 * f1;
        const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
        const bool abort_seen = *abort_flag != 0;
        // stage the normalised rows in shared memory (the K/V ring is idle now);
        // warpgroup wg fills output columns [64 wg, 64 wg + 64)
        float *ostage = reinterpret_cast<float *>(sbase + L::kOffStage);
        if (!abort_seen) {
            tc_fence_after();
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                const uint32_t col = 64u * wg + 32u * cc;
                uint32_t oa[32], ob[32];
                tmem_ld32_async(tmem + lane_off + col, oa);
                tmem_ld32_async(tmem + lane_off + 128u + col, ob);
                tmem_ld_wait();
                tmem_ld_bind(oa);
                tmem_ld_bind(ob);
#pragma unroll
                for (int e = 0; e < 32; e += 4) {
                    float v[4];
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        const float a0 = l0 > 0.f ? __uint_as_float(oa[e + q4]) * f0 : 0.f;
                        const float a1 = l1 > 0.f ? __uint_as_float(ob[e + q4]) * f1 : 0.f;
                        v[q4] = (a0 + a1) * inv;
                    }
                    *reinterpret_cast<float4 *>(ostage + r * kOStride + col + e) = make_float4(v[0], v[1], v[2], v[3]);
                }
            }
            if (row_ok && wg == 0) {
                const int h = g * G + r % G;
                p.lse_part[(long)s * rows_total + ((long)b * T + j) * p.Hq + h] =
                    Lsum > 0.f ? Mx * kLn2 + logf(Lsum) : -INFINITY;
            }
        }
        tc_fence_before();
        named_sync(1, 256);
        if (!abort_seen) {
            // rows (j, hl) of one j are G consecutive rows of the partial output:
            // copy them out as contiguous float4 runs
            const int per_j = G * 32;  // float4s
            for (int idx = tid; idx < M * 32; idx += 256) {
                const int jj = idx / per_j, rem = idx % per_j, hl = rem >> 5, c4 = rem & 31;
                const int rr = jj * G + hl;
                const float4 v = *reinterpret_cast<const float4 *>(ostage + rr * kOStride + c4 * 4);
                float *dst = p.o_part + ((long)s * rows_total + ((long)b * T + jj) * p.Hq + g * G + hl) * 128;
                *reinterpret_cast<float4 *>(dst + c4 * 4) = v;
            }
        }
    }

    // teardown: every MMA has completed (drain above); free tensor memory
    __syncthreads();
    if (warp == 9) {
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

// 4-D map over the contiguous queries [B, T, Hq, D]; box: 64 d x G heads x T rows x 1,
// which lands in shared memory as rows j*G + hl of 128 bytes
bool make_q_map(CUtensorMap *m, const AttnParams &p) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn) return false;
    const int G = p.Hq / p.Hkv;
    cuuint64_t dims[4] = {128, (cuuint64_t)p.Hq, (cuuint64_t)p.T, (cuuint64_t)p.B};
    cuuint64_t strides[3] = {256, (cuuint64_t)p.Hq * 256, (cuuint64_t)p.T * p.Hq * 256};
    cuuint32_t box[4] = {64, (cuuint32_t)G, (cuuint32_t)p.T, 1}, estr[4] = {1, 1, 1, 1};
    const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(p.q), dims, strides, box,
                          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <bool kPTmem>
cudaError_t launch_tc_t(const AttnParams &p, cudaStream_t st) {
    alignas(64) CUtensorMap mq, mk, mv;
    TcParams tp;
    tp.a = p;
    int ds2 = 0, dh2 = 0;
    if (!make_q_map(&mq, p)) return cudaErrorInvalidValue;
    if (!make_map(&mk, p.kc, p.kv, cache_slots(p), p.Hkv, p.B, &tp.dim_s, &tp.dim_h)) return cudaErrorInvalidValue;
    if (!make_map(&mv, p.vc, p.kv, cache_slots(p), p.Hkv, p.B, &ds2, &dh2)) return cudaErrorInvalidValue;
    constexpr int smem = Layout<kPTmem>::kSmemBytes;
    static bool opted_in[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !opted_in[dev]) {
        e = cudaFuncSetAttribute(attn_split_tc_kernel<kPTmem>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) opted_in[dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.n_splits, p.Hkv, p.B);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, attn_split_tc_kernel<kPTmem>, mq, mk, mv, tp);
}

}  // namespace

bool attn_tc_supported(const AttnParams &p) {
    if (p.dt != SD_BF16 || p.D != 128 || p.T < 1 || p.T > kMaxT) return false;
    if ((p.Hq / p.Hkv) * p.T > 128) return false;
    if ((long)p.max_ctx + p.T > (1L << 30)) return false;
    if (!encode_fn()) return false;
    int dev = 0, optin = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return false;
    if (optin < Layout<true>::kSmemBytes || optin < Layout<false>::kSmemBytes) return false;
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    return major == 10 && minor == 3;
}

size_t attn_tc_smem_bytes(const AttnParams &) { return Layout<true>::kSmemBytes; }

cudaError_t launch_attn_tc(const AttnParams &p, cudaStream_t st) { return launch_tc_t<true>(p, st); }
cudaError_t launch_attn_tc_smem_p(const AttnParams &p, cudaStream_t st) { return launch_tc_t<false>(p, st); }

}  // namespace sdv
