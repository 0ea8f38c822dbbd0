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
// tile is fetched from HBM once and serves every row.  For key tile t
// (128 keys):
//   S_t = Q . K_t^T                       (M 128, N 128 keys, K 128)
//   P_t = exp2(S_t * scale * log2e - m)   split as P_hi + P_lo, both bf16
//   O  += P_hi . V_t + P_lo . V_t         (M 128, N 128, K 128)
// The two-term split keeps every weight to within 2^-14 relative, so the
// product is as accurate as an fp32 P even when a few keys dominate.
//
// Warp roles (384 threads):
//   warp 0           TMA producer: Q, then K tiles and V tiles into rings of
//                    three 32 KB slots each
//   warp 1           allocates tensor memory; one thread issues every MMA: S
//                    up to three tiles ahead, and P.V as soon as its P is written
//   warps 4-7, 8-11  two softmax warpgroups, both on every tile: warpgroup w
//                    takes keys [64 w, 64 w + 64) of it; thread = row (=
//                    tensor-memory lane).  They exchange the row max through
//                    shared memory, so both hold the same reference max and O
//                    is a single accumulator.
// A K slot is refilled as soon as the S that read it has completed, a V slot
// once its P.V has.  The producer sets up the barriers and issues Q and the
// first K/V tiles before the CTA-wide sync, so the copies overlap the tensor
// memory allocation.
// Tensor memory: O [0,128) and three S/P buffers [128 + 128 i, +128).  P is
// written back over the S columns it came from (hi and lo halves of each
// 64-key half) and read by the P.V MMAs as their A operand.  The partial
// output leaves through shared memory so that the global stores are
// coalesced.  With several splits the kernel also merges them (see
// merge_group); with one it writes the output itself.
// The running max only moves when it grows by more than 2^8, so O is rescaled
// in tensor memory rarely (exact either way: P and l use the same reference).
// Tiles that every row sees in full skip the per-key masks.
// Every wait is bounded by the global timer; a wait that gives up sets the
// fault word and the CTA drains its copies and MMAs before freeing tensor
// memory and returning.
#include "common.cuh"
#include "tcgen05.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>

#include <math.h>
#include <string.h>
#include <atomic>

namespace sdv {

namespace {

constexpr int kTcThreads = 384;
constexpr int kProducerWarp = 0;            // TMA producer
constexpr int kMmaWarp = 1;                 // tensor-memory allocation, MMA issue
constexpr int kSoftmaxWarp0 = 4;            // warps 4-7 and 8-11: the two softmax warpgroups
constexpr int kBN = kTcTileKeys;            // keys per tile (128)
constexpr int kTileBytes = 2 * kBN * 128;   // K or V tile: two 64-column blocks of [128 keys x 128 B]
constexpr int kQBytes = 2 * 128 * 128;      // Q: two 64-column blocks of [128 rows x 128 B]
constexpr int kKSlots = 3, kVSlots = 3;
constexpr int kSP = 3;                      // S/P buffers in tensor memory
constexpr uint32_t kTmemCols = 512;         // O [0,128), S/P buffer i at [128 + 128 i, +128)
constexpr int kOStride = 132;               // floats per staged output row (bank-conflict padding)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;   // log2 units
// A tile whose weights are all at most kLoFrac of the running sum (in every
// row) is multiplied with P rounded to nearest bf16 alone; any other tile
// with the two-term P (hi + lo).
constexpr float kLoFrac = 0.25f;

struct Layout {
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kQBytes;
    static constexpr int kOffV = kOffK + kKSlots * kTileBytes;
    static constexpr int kOffBar = kOffV + kVSlots * kTileBytes;
    // kfull[3] kempty[3] vfull[3] vempty[3] sfull[3] pfull[3] pempty[3] qready drain
    static constexpr int kNumBars = 2 * kKSlots + 2 * kVSlots + 3 * kSP + 2;
    static constexpr int kOffMisc = kOffBar + 8 * kNumBars;                 // tmem base, abort flag, merge flag
    static constexpr int kOffX = kOffMisc + 16;                             // [2][128] per-row exchange
    static constexpr int kOffLo = kOffX + 2 * 128 * 4;                      // [kSP] tile + 1 when its P needs lo
    // epilogue, once every copy and MMA is done: the staged output rows, in the
    // (then idle) K ring
    static constexpr int kOffOStage = kOffK;
    static constexpr int kSmemBytes = kOffLo + 16 + 1024;                   // + alignment slack
    static_assert(128 * kOStride * 4 <= kKSlots * kTileBytes, "staging fits in the K ring");
    static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
};

// ---------------------------------------------------------------------------
// merge of the splits inside the kernel
// ---------------------------------------------------------------------------
// Bounded wait until the counter reaches `target`.
__device__ __noinline__ bool wait_count(const unsigned int *ctr, unsigned int target) {
    const unsigned long long t0 = global_timer();
    for (uint32_t it = 0;; ++it) {
        unsigned int v;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
        if (v >= target) return true;
        if ((it & 15u) == 15u && global_timer() - t0 > kWaitLimitNs) return false;
        __nanosleep(32);
    }
}

// Every split of sequence b, kv head g, row block mb has written its partial
// (rows normalised by their own sum, plus their log-sum-exp); once all of them
// have arrived, split s combines rows s, s + n, s + 2n, ... of the group's M
// rows (n = splits; row rr is block row j0 + rr / G, query head g G + rr % G):
// out = sum_s w_s o_s / sum_s w_s with w_s = exp(lse_s - max).
// The whole grid is resident (at most one CTA per SM), so the wait ends.  The
// counter is returned to zero by the last split to finish merging.  `scratch`
// is idle shared memory (the K/V rings).
constexpr int kMergeBatch = 12;  // loads one merge thread keeps in flight
__device__ void merge_group(const AttnParams &p, int s, int g, int b, int mb, int j0, int M, int G,
                            long rows_total, volatile int *go, uint8_t *scratch) {
    unsigned int *ctr = p.merge_ctr + (((long)b * p.Hkv + g) * p.n_mblk + mb);
    const int n = (int)gridDim.x;
    const int tid = threadIdx.x;
    __threadfence();  // this thread's partial stores are visible device-wide
    __syncthreads();
    if (tid == 0) {
        atomicAdd(ctr, 1u);
        const bool ok = wait_count(ctr, (unsigned int)n);
        if (!ok) set_fault(p.fault, FAULT_WAIT_TIMEOUT);
        *go = ok ? 1 : 0;
    }
    __syncthreads();
    const int R = s < M ? (M - s + n - 1) / n : 0;   // rows of this split
    // the splits of a row are cut into K chunks, so that about one (row, 4
    // columns, chunk) unit falls to each thread; a unit loads its chunk's
    // partials and their log-sum-exps together (one round trip), weighs them
    // against the chunk's own largest log-sum-exp, and the K chunk results are
    // then combined against the largest of those
    const int K = max(1, min(n, kTcThreads / max(1, R * 32)));
    const int chunk = (n + K - 1) / K;
    float4 *pacc = reinterpret_cast<float4 *>(scratch);                    // [K][R][32] weighted sums
    float *pm = reinterpret_cast<float *>(scratch + (size_t)K * R * 32 * 16);  // [K][R][32] chunk reference
    float *pw = pm + K * R * 32;                                           // [K][R][32] sum of weights
    auto frow_of = [&](int ri) {
        const int rr = s + ri * n;
        return ((long)b * p.T + j0 + rr / G) * p.Hq + g * G + rr % G;
    };
    if (*go && R > 0) {
        for (int u = tid; u < K * R * 32; u += kTcThreads) {
            const int k = u / (R * 32), ri = (u / 32) % R, c4 = u & 31;
            const long frow = frow_of(ri);
            const int sp0 = k * chunk, sp1 = min(n, sp0 + chunk);
            float m_run = -INFINITY, w_run = 0.f;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int sb = sp0; sb < sp1; sb += kMergeBatch) {
                // branch-free, so that the batch's loads are all in flight at
                // once: past the chunk's end, re-read its last split and drop it
                float4 v[kMergeBatch];
                float l[kMergeBatch];
#pragma unroll
                for (int e = 0; e < kMergeBatch; ++e) {
                    const int sp = min(sb + e, sp1 - 1);
                    v[e] = __ldcg(reinterpret_cast<const float4 *>(p.o_part + ((long)sp * rows_total + frow) * 128) + c4);
                    l[e] = sb + e < sp1 ? __ldcg(p.lse_part + (long)sp * rows_total + frow) : -INFINITY;
                }
                float bm = l[0];
#pragma unroll
                for (int e = 1; e < kMergeBatch; ++e) bm = fmaxf(bm, l[e]);
                if (bm == -INFINITY) continue;                 // only empty splits so far in this batch
                if (bm > m_run) {                              // a new reference: rescale what is held
                    const float f = m_run == -INFINITY ? 0.f : __expf(m_run - bm);
                    acc.x *= f; acc.y *= f; acc.z *= f; acc.w *= f;
                    w_run *= f;
                    m_run = bm;
                }
#pragma unroll
                for (int e = 0; e < kMergeBatch; ++e) {
                    const float w = __expf(l[e] - m_run);       // 0 for an empty split (l = -inf)
                    w_run += w;
                    acc.x = fmaf(w, v[e].x, acc.x); acc.y = fmaf(w, v[e].y, acc.y);
                    acc.z = fmaf(w, v[e].z, acc.z); acc.w = fmaf(w, v[e].w, acc.w);
                }
            }
            pacc[u] = acc;
            pm[u] = m_run;
            pw[u] = w_run;
        }
        __syncthreads();
        for (int i = tid; i < R * 32; i += kTcThreads) {
            const int ri = i / 32, c4 = i & 31;
            float M = -INFINITY;
            for (int k = 0; k < K; ++k) M = fmaxf(M, pm[k * R * 32 + i]);
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            float wsum = 0.f;
            if (M != -INFINITY) {
                for (int k = 0; k < K; ++k) {
                    const float mk = pm[k * R * 32 + i];
                    const float f = mk == -INFINITY ? 0.f : __expf(mk - M);
                    const float4 a = pacc[k * R * 32 + i];
                    acc.x = fmaf(f, a.x, acc.x); acc.y = fmaf(f, a.y, acc.y);
                    acc.z = fmaf(f, a.z, acc.z); acc.w = fmaf(f, a.w, acc.w);
                    wsum = fmaf(f, pw[k * R * 32 + i], wsum);
                }
            }
            const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
            reinterpret_cast<float4 *>(p.out + frow_of(ri) * 128)[c4] =
                make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
        }
    }
    // every split takes a second ticket, whether or not its wait succeeded, so
    // the counter sees exactly 2n increments per launch and the last of them
    // returns it to zero: a launch whose wait gave up (fault bit set, its rows
    // left unmerged) still leaves the workspace ready for the next call
    __syncthreads();
    if (tid == 0) {
        const unsigned int ticket = atomicAdd(ctr, 1u);
        if (ticket == 2u * (unsigned int)n - 1u) atomicExch(ctr, 0u);
    }
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kTcThreads, 1)
attn_split_tc_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                     const __grid_constant__ CUtensorMap tmap_v, const AttnParams p) {
    using L = Layout;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    const uint32_t base = (raw_u32 + 1023u) & ~1023u;
    uint8_t *sbase = smem_raw + (base - raw_u32);

    // grid: (split, kv head x row block, sequence)
    const int s = blockIdx.x, g = blockIdx.y / p.n_mblk, mb = blockIdx.y % p.n_mblk, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    const uint32_t sQ = base + L::kOffQ, sK = base + L::kOffK, sV = base + L::kOffV;
    const uint32_t bar0 = base + L::kOffBar;
    auto kfull_bar = [&](int i) { return bar0 + 8u * i; };
    auto kempty_bar = [&](int i) { return bar0 + 8u * (kKSlots + i); };
    auto vfull_bar = [&](int i) { return bar0 + 8u * (2 * kKSlots + i); };
    auto vempty_bar = [&](int i) { return bar0 + 8u * (2 * kKSlots + kVSlots + i); };
    const uint32_t bar1 = bar0 + 8u * (2 * kKSlots + 2 * kVSlots);
    auto sfull_bar = [&](int i) { return bar1 + 8u * i; };               // S in buffer i computed
    auto pfull_bar = [&](int i) { return bar1 + 8u * (kSP + i); };       // P in buffer i written (8 warps)
    auto pempty_bar = [&](int i) { return bar1 + 8u * (2 * kSP + i); };  // P.V of buffer i completed
    const uint32_t qready_bar = bar1 + 8u * (3 * kSP);
    const uint32_t drain_bar = bar1 + 8u * (3 * kSP + 1);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(sbase + L::kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sbase + L::kOffMisc + 8);
    float *xrow = reinterpret_cast<float *>(sbase + L::kOffX);  // [2][128]: one value per row and warpgroup
    // lo_flag[i] == t + 1: tile t, in S/P buffer i, is multiplied with the two-term P
    volatile int *lo_flag = reinterpret_cast<volatile int *>(sbase + L::kOffLo);

    const bool producer = warp == kProducerWarp && lane == 0;
    if (producer) {
        for (int i = 0; i < kKSlots; ++i) { mbar_init(kfull_bar(i), 1); mbar_init(kempty_bar(i), 1); }
        for (int i = 0; i < kVSlots; ++i) { mbar_init(vfull_bar(i), 1); mbar_init(vempty_bar(i), 1); }
        for (int i = 0; i < kSP; ++i) { mbar_init(sfull_bar(i), 1); mbar_init(pfull_bar(i), 8); mbar_init(pempty_bar(i), 1); }
        mbar_init(qready_bar, 1);  // the Q copy, with its bytes
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        for (int i = 0; i < kSP; ++i) lo_flag[i] = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_q)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_k)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_v)) : "memory");
    }
    if (warp == kMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_holder)), "r"(kTmemCols) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
#if __CUDA_ARCH__ >= 900
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");  // inputs of an upstream kernel are visible now
#endif

    // this CTA's rows: block rows [j0, j0 + Tb) of the G query heads of kv head g
    const int T = p.T, G = p.Hq / p.Hkv;
    const int j0 = mb * p.mblk_nodes, Tb = min(p.mblk_nodes, T - j0), M = G * Tb;
    const int MQ = G * p.mblk_nodes;  // rows the Q copy writes (those past block row T - 1 as zeros)
    if (producer) {
        // Q first: rows r = (j - j0)*G + hl of this kv head, two 64-column halves;
        // the copy always moves the whole box (out-of-range rows are zero-filled)
        mbar_arrive_expect_tx(qready_bar, (uint32_t)(256 * MQ));
        tma_load_4d(sQ, &tmap_q, qready_bar, 0, g * G, j0, b);
        tma_load_4d(sQ + 128 * 128, &tmap_q, qready_bar, 64, g * G, j0, b);
    }
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
    const int first_tma = has_block_tile ? 1 : 0;  // tile 0 of the drafter's split 0 is the block
    const long rows_total = (long)p.B * T * p.Hq;
    auto tile_key0 = [&](int t) { return k0 + (t - first_tma) * kBN; };
    auto is_block_tile = [&](int t) { return has_block_tile && t == 0; };
    // keys every row of the block sees: the drafter's context, the target's
    // cache before the block (before the anchor for a tree)
    const bool tree = p.mode == 2;
    const int all_see = min(cend, tree ? nb - 1 : nb);

    // one copy per tile: map coordinates (d within a half, key, half, kv head, sequence)
    auto issue_k = [&](int t) {
        const int slot = t % kKSlots;
        mbar_arrive_expect_tx(kfull_bar(slot), (uint32_t)kTileBytes);
        tma_load_5d(sK + slot * kTileBytes, &tmap_k, kfull_bar(slot), 0, tile_key0(t), 0, g, b);
    };
    auto issue_v = [&](int t) {
        const int slot = t % kVSlots;
        mbar_arrive_expect_tx(vfull_bar(slot), (uint32_t)kTileBytes);
        tma_load_5d(sV + slot * kTileBytes, &tmap_v, vfull_bar(slot), 0, tile_key0(t), 0, g, b);
    };
    // first wave, before the CTA-wide sync: every slot of both rings
    int next_k = first_tma, next_v = first_tma;
    if (producer) {
        for (; next_k < min(n_tiles, kKSlots); ++next_k) {
            issue_k(next_k);
            if (next_v < min(n_tiles, kVSlots)) issue_v(next_v++);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (n_tiles == 0) {
        // nothing to read: an empty split (lse = -inf, zero partial) for the merge;
        // the Q copy issued above lands before the CTA exits
        if (producer) mbar_wait(qready_bar, 0, nullptr, p.fault);
        for (int idx = tid; idx < M * 32; idx += kTcThreads) {
            const int rr = idx >> 5, c4 = idx & 31;
            const long frow = ((long)b * T + j0 + rr / G) * p.Hq + g * G + rr % G;
            float *dst = p.merge == 2 ? p.out + frow * 128 : p.o_part + ((long)s * rows_total + frow) * 128;
            reinterpret_cast<float4 *>(dst)[c4] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (c4 == 0 && p.merge != 2) p.lse_part[(long)s * rows_total + frow] = -INFINITY;
        }
    } else if (warp == kProducerWarp) {
        // ------------------------------------------------------------------ producer
        if (has_block_tile) {
            // the T block keys / values from [B, T, Hkv, D] into slot 0 of each ring; rows >= T zero
            const __nv_bfloat16 *kb = static_cast<const __nv_bfloat16 *>(p.kb);
            const __nv_bfloat16 *vb = static_cast<const __nv_bfloat16 *>(p.vb);
            uint8_t *ks = sbase + L::kOffK, *vs = sbase + L::kOffV;
            for (int idx = lane; idx < kBN * 16; idx += 32) {
                const int row = idx >> 4, ch = idx & 15;
                uint4 kv4 = make_uint4(0u, 0u, 0u, 0u), vv4 = make_uint4(0u, 0u, 0u, 0u);
                if (row < T) {
                    const long off = (((long)b * T + row) * p.Hkv + g) * 128;
                    kv4 = __ldg(reinterpret_cast<const uint4 *>(kb + off) + ch);
                    vv4 = __ldg(reinterpret_cast<const uint4 *>(vb + off) + ch);
                }
                const uint32_t o = (ch >> 3) * (kBN * 128) + sw128_off(row, ch & 7);
                *reinterpret_cast<uint4 *>(ks + o) = kv4;
                *reinterpret_cast<uint4 *>(vs + o) = vv4;
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) { mbar_arrive(kfull_bar(0)); mbar_arrive(vfull_bar(0)); }
        }
        if (lane == 0) {
            // whichever ring has a free slot first: a K slot frees when its S has
            // completed, a V slot when its P.V has, so neither waits behind the other
            unsigned long long t_last = global_timer();
            for (uint32_t spin = 0; next_k < n_tiles || next_v < n_tiles;) {
                if (next_k < n_tiles &&
                    (next_k < kKSlots || mbar_test(kempty_bar(next_k % kKSlots), ((next_k / kKSlots) - 1) & 1))) {
                    issue_k(next_k++);
                    t_last = global_timer();
                    continue;
                }
                if (next_v < n_tiles &&
                    (next_v < kVSlots || mbar_test(vempty_bar(next_v % kVSlots), ((next_v / kVSlots) - 1) & 1))) {
                    issue_v(next_v++);
                    t_last = global_timer();
                    continue;
                }
                // nothing free yet: back off, so the poll does not take issue
                // slots and shared-memory bandwidth from the softmax warps
                __nanosleep(64);
                if ((++spin & 15u) == 0) {
                    if (*abort_flag) break;
                    if (global_timer() - t_last > kWaitLimitNs) {
                        *abort_flag = 1;
                        set_fault(p.fault, FAULT_WAIT_TIMEOUT);
                        break;
                    }
                }
            }
            // on abort: let the copies already issued land before the CTA exits
            if (*abort_flag) {
                mbar_wait(qready_bar, 0, nullptr, p.fault);
                for (int u = max(first_tma, next_k - kKSlots); u < next_k; ++u)
                    mbar_wait(kfull_bar(u % kKSlots), (u / kKSlots) & 1, nullptr, p.fault);
                for (int u = max(first_tma, next_v - kVSlots); u < next_v; ++u)
                    mbar_wait(vfull_bar(u % kVSlots), (u / kVSlots) & 1, nullptr, p.fault);
            }
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------------ MMA issuer
        // Q rows past the MQ the copy writes are zero, so the padding rows of S
        // are finite (the copy itself zero-fills rows [M, MQ))
        for (int idx = lane; idx < (128 - MQ) * 16; idx += 32) {
            const int row = MQ + (idx >> 4), ch = idx & 15;
            *reinterpret_cast<uint4 *>(sbase + L::kOffQ + (ch >> 3) * (128 * 128) + sw128_off(row, ch & 7)) =
                make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            const uint32_t idS = idesc_bf16(128, kBN, false);
            const uint32_t idO = idesc_bf16(128, 128, true);
            bool ok = mbar_wait(qready_bar, 0, abort_flag, p.fault);
            // S runs up to kSP tiles ahead of P.V; whichever of the next S and
            // the next P.V can go is issued, P.V first
            int ns = 0, npv = 0;
            unsigned long long t_last = global_timer();
            for (uint32_t spin = 0; ok && npv < n_tiles;) {
                if (npv < ns && mbar_test(pfull_bar(npv % kSP), (npv / kSP) & 1) &&
                    mbar_test(vfull_bar(npv % kVSlots), (npv / kVSlots) & 1)) {
                    // P.V(npv): O += P_hi . V (+ P_lo . V when the softmax warps asked
                    // for the two-term P) over the 128 keys
                    tc_fence_after();
                    const uint32_t vb = sV + (npv % kVSlots) * kTileBytes;
                    const uint32_t pb = tmem + 128u + 128u * (npv % kSP);
                    const bool two_term = lo_flag[npv % kSP] == npv + 1;
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        // 16 keys: V rows 16 kk.., P columns of the 64-key half kk / 4
                        const uint64_t bd = sw128_desc(vb + kk * 16 * 128, kBN * 128, 1024);
                        const uint32_t a = pb + 64u * (kk >> 2) + 8u * (kk & 3);
                        umma_ts(tmem, a, bd, idO, (npv > 0 || kk > 0) ? 1u : 0u);
                        if (two_term) umma_ts(tmem, a + 32u, bd, idO, 1u);
                    }
                    umma_commit(pempty_bar(npv % kSP));
                    umma_commit(vempty_bar(npv % kVSlots));
                    ++npv;
                    t_last = global_timer();
                    continue;
                }
                if (ns < n_tiles && ns < npv + kSP && mbar_test(kfull_bar(ns % kKSlots), (ns / kKSlots) & 1) &&
                    (ns < kSP || mbar_test(pempty_bar(ns % kSP), ((ns / kSP) - 1) & 1))) {
                    // S(ns) into buffer ns % 3, free once P.V(ns - 3) has read it
                    tc_fence_after();
                    const uint32_t kb = sK + (ns % kKSlots) * kTileBytes;
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint32_t off = (kk >> 2) * (128 * 128) + (kk & 3) * 32;
                        umma_ss(tmem + 128u + 128u * (ns % kSP), sw128_desc(sQ + off, 16, 1024),
                                sw128_desc(kb + (kk >> 2) * (kBN * 128) + (kk & 3) * 32, 16, 1024), idS,
                                kk > 0 ? 1u : 0u);
                    }
                    umma_commit(sfull_bar(ns % kSP));
                    umma_commit(kempty_bar(ns % kKSlots));
                    ++ns;
                    t_last = global_timer();
                    continue;
                }
                // nothing ready yet: back off (see the producer), bounded
                __nanosleep(32);
                if ((++spin & 15u) == 0) {
                    if (*abort_flag) ok = false;
                    else if (global_timer() - t_last > kWaitLimitNs) {
                        *abort_flag = 1;
                        set_fault(p.fault, FAULT_WAIT_TIMEOUT);
                        ok = false;
                    }
                }
            }
            // every MMA has completed before tensor memory is freed
            umma_commit(drain_bar);
            mbar_wait(drain_bar, 0, nullptr, p.fault);
        }
        __syncwarp();
    } else if (warp >= kSoftmaxWarp0) {
        // ------------------------------------------------------------------ softmax (warps 4-11)
        // both warpgroups take every tile: warpgroup wg the keys [64 wg, 64 wg + 64);
        // they share the row max through shared memory, so O is one accumulator
        const int sidx = tid - 32 * kSoftmaxWarp0;  // thread index among the softmax warps
        const int wg = sidx >> 7;                   // key half of every tile
        const int r = sidx & 127;                   // query row = tensor-memory lane (warp % 4 picks the lanes)
        const bool row_ok = r < M;
        const int j = row_ok ? j0 + r / G : 0;   // block row (tree node) of this query row
        const float qk = p.scale * kLog2e;
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t o_col = tmem + lane_off + 64u * wg;   // this warpgroup's half of O (rescale, epilogue)

        // Every softmax warp runs every iteration, whatever happens: the two
        // warpgroups meet at named barriers each tile.  After a failed wait the
        // warp keeps going on meaningless values (the fault word is set and
        // every later wait returns at once) so that no barrier is left short.
        float m_used = -INFINITY, l = 0.f;
        bool ok = true;
        for (int t = 0; t < n_tiles; ++t) {
            const int bi = t % kSP;
            const uint32_t sp_col = tmem + lane_off + 128u + 128u * bi + 64u * wg;
            ok = __all_sync(0xffffffffu, mbar_wait(sfull_bar(bi), (t / kSP) & 1, abort_flag, p.fault)) && ok;
            tc_fence_after();
            // keys [0, nvalid) of the tile are visible to this row; a tile below
            // every row's limit needs no mask (the padding rows past M compute
            // finite values that are never stored)
            const bool blk = is_block_tile(t);
            const bool whole = !blk && tile_key0(t) + kBN <= all_see;
            // bit c: key c of this warpgroup's half of the tile is visible to the row
            uint64_t vis = ~0ull;
            if (!whole) {
                auto prefix = [](int n) { return n <= 0 ? 0ull : n >= 64 ? ~0ull : (1ull << n) - 1ull; };
                const int key0h = tile_key0(t) + 64 * wg;
                if (!row_ok) {
                    vis = 0ull;
                } else if (blk) {
                    vis = prefix(T - 64 * wg);
                } else if (tree) {
                    vis = prefix(min(cend, nb - 1) - key0h);
                    const uint64_t tm = p.tree_mask[(long)b * T + j];
                    for (int k = 0; k < T; ++k) {
                        const int pos = nb - 1 + k - key0h;
                        if (pos >= 0 && pos < 64 && key0h + pos < cend && ((tm >> k) & 1ull)) vis |= 1ull << pos;
                    }
                } else {
                    vis = prefix((drafter ? cend : min(cend, nb + j)) - key0h);
                }
            }
            uint32_t sa[32], sb[32];
            tmem_ld32_async(sp_col, sa);
            tmem_ld32_async(sp_col + 32u, sb);
            tmem_ld_wait();
            tmem_ld_bind(sa);
            tmem_ld_bind(sb);
            // row max of the raw scores (qk > 0 keeps the order), shared with the
            // other warpgroup: both then take the same decisions below
            // (separate loops: a select folded into the unmasked one costs ~6x)
            float mx[8];
            if (whole) {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const uint32_t *src = i < 4 ? sa : sb;
                    const int o = 8 * (i & 3);
                    float m8 = __uint_as_float(src[o]);
#pragma unroll
                    for (int e = 1; e < 8; ++e) m8 = fmaxf(m8, __uint_as_float(src[o + e]));
                    mx[i] = m8;
                }
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const uint32_t *src = i < 4 ? sa : sb;
                    const int o = 8 * (i & 3);
                    float m8 = -INFINITY;
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        m8 = fmaxf(m8, ((vis >> (8 * i + e)) & 1ull) ? __uint_as_float(src[o + e]) : -INFINITY);
                    mx[i] = m8;
                }
            }
            const float hmax = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                     fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
            // the two-term P is needed for the split's first tile, and for any tile
            // where a row's largest weight, in the reference of the tiles before,
            // exceeds kLoFrac of that row's running sum; the vote of all rows is
            // one flag, read after the barrier by every softmax warp and, after
            // the P arrival, by the MMA issuer
            const bool vote = t == 0 || (row_ok && !(ex2(hmax * qk - m_used) <= kLoFrac * l));
            if (__any_sync(0xffffffffu, vote) && lane == 0) lo_flag[bi] = t + 1;
            xrow[wg * 128 + r] = hmax;
            named_sync(1, 256);
            const float omax = xrow[(wg ^ 1) * 128 + r];
            const bool two_term = lo_flag[bi] == t + 1;
            named_sync(1, 256);  // both read before the next tile writes
            const float tmax = fmaxf(hmax, omax) * qk;
            // move the reference max only when it grows by more than 2^8
            const bool first = t == 0;
            const bool need = !first && tmax > m_used + kRescaleThreshold;
            float alpha = 1.f;
            if (first) m_used = tmax;
            else if (need) { alpha = ex2(m_used - tmax); m_used = tmax; }
            if (__any_sync(0xffffffffu, need)) {
                // the previous P.V must be done before O is rescaled (this
                // warpgroup's 64 columns of it)
                ok = __all_sync(0xffffffffu,
                                mbar_wait(pempty_bar((t - 1) % kSP), ((t - 1) / kSP) & 1, abort_flag, p.fault)) && ok;
                tc_fence_after();
#pragma unroll 1
                for (int cc = 0; cc < 2; ++cc) {
                    uint32_t oa[32];
                    tmem_ld32_async(o_col + 32u * cc, oa);
                    tmem_ld_wait();
                    tmem_ld_bind(oa);
#pragma unroll
                    for (int e = 0; e < 32; ++e) oa[e] = __float_as_uint(__uint_as_float(oa[e]) * alpha);
                    tmem_st32(o_col + 32u * cc, oa);
                }
            }
            l *= alpha;
            const bool live = m_used != -INFINITY;
            const float neg_m = live ? -m_used : 0.f;
            if (!live) vis = 0ull;
            float ls[4] = {0.f, 0.f, 0.f, 0.f};
            // the masked keys of an edge tile are cleared in the scores first
            // (-inf gives a weight of 0), so the exponential loop has no selects
            if (!whole || !live) {
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    if (!((vis >> c) & 1ull)) sa[c] = 0xff800000u;
                    if (!((vis >> (32 + c)) & 1ull)) sb[c] = 0xff800000u;
                }
            }
            if (two_term) {
                // P of this 64-key half over the S columns it came from: hi in
                // [0,32), lo in [32,64).  hi = p truncated to bf16; lo = the exact
                // fp32 remainder truncated to bf16: |p - hi - lo| < 2^-14 p.  Byte
                // permutes instead of conversion instructions.
#pragma unroll
                for (int q = 0; q < 2; ++q) {   // 32 keys at a time
                    const uint32_t *sq = q == 0 ? sa : sb;
                    uint32_t pk[16], pl[16];
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        const float p0 = ex2(fmaf(__uint_as_float(sq[2 * c]), qk, neg_m));
                        const float p1 = ex2(fmaf(__uint_as_float(sq[2 * c + 1]), qk, neg_m));
                        ls[c & 3] += p0 + p1;
                        const uint32_t b0 = __float_as_uint(p0), b1 = __float_as_uint(p1);
                        pk[c] = __byte_perm(b0, b1, 0x7632);
                        const uint32_t q0 = __float_as_uint(p0 - __uint_as_float(b0 & 0xffff0000u));
                        const uint32_t q1 = __float_as_uint(p1 - __uint_as_float(b1 & 0xffff0000u));
                        pl[c] = __byte_perm(q0, q1, 0x7632);
                    }
                    tmem_st16(sp_col + 16u * q, pk);
                    tmem_st16(sp_col + 32u + 16u * q, pl);
                }
            } else {
                // P rounded to nearest bf16 in [0,32), and the running sum taken
                // over the rounded weights themselves, so that the output is the
                // exact average under those weights (rounding common to all of
                // them cancels)
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const uint32_t *sq = q == 0 ? sa : sb;
                    uint32_t pk[16];
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        const float p0 = ex2(fmaf(__uint_as_float(sq[2 * c]), qk, neg_m));
                        const float p1 = ex2(fmaf(__uint_as_float(sq[2 * c + 1]), qk, neg_m));
                        const __nv_bfloat162 h2 = __floats2bfloat162_rn(p0, p1);   // .x = p0 in the low half
                        const uint32_t h = *reinterpret_cast<const uint32_t *>(&h2);
                        pk[c] = h;
                        ls[c & 3] += __uint_as_float(h << 16) + __uint_as_float(h & 0xffff0000u);
                    }
                    tmem_st16(sp_col + 16u * q, pk);
                }
            }
            l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
            // value rows past the split's last cache key may hold anything (P is
            // zero there, but 0 * NaN is not): each warpgroup zeroes those of
            // its key half once V(t) has landed
            if (!blk && !whole) {
                const int v0 = max(64 * wg, min(64 * wg + 64, cend - tile_key0(t)));
                if (ok && v0 < 64 * wg + 64) {
                    ok = __all_sync(0xffffffffu, mbar_wait(vfull_bar(t % kVSlots), (t / kVSlots) & 1, abort_flag,
                                                           p.fault));
                    if (ok) {
                        uint8_t *vt = sbase + L::kOffV + (t % kVSlots) * kTileBytes;
                        for (int idx = r; idx < (64 * wg + 64 - v0) * 16; idx += 128) {
                            const int row = v0 + (idx >> 4), ch = idx & 15;
                            *reinterpret_cast<uint4 *>(vt + (ch >> 3) * (kBN * 128) + sw128_off(row, ch & 7)) =
                                make_uint4(0u, 0u, 0u, 0u);
                        }
                        fence_proxy_async_smem();
                    }
                }
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(pfull_bar(bi));
        }
        // ---- epilogue: normalise O, write this split's partial (or the output) ----
        const int last_t = n_tiles - 1;
        ok = __all_sync(0xffffffffu,
                        mbar_wait(pempty_bar(last_t % kSP), (last_t / kSP) & 1, abort_flag, p.fault)) && ok;
        if (!ok) { m_used = -INFINITY; l = 0.f; }
        tc_fence_before();
        // the last P.V, hence every MMA (and every copy they read), is complete
        // past this point: the rings are free for the staging
        named_sync(1, 256);
        xrow[wg * 128 + r] = l;
        named_sync(1, 256);
        const float Lsum = wg == 0 ? l + xrow[128 + r] : xrow[r] + l;  // same order in both
        const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
        const bool abort_seen = *abort_flag != 0;
        // stage the normalised rows in shared memory; warpgroup wg fills output
        // columns [64 wg, 64 wg + 64)
        float *ostage = reinterpret_cast<float *>(sbase + L::kOffOStage);
        if (!abort_seen) {
            tc_fence_after();
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                uint32_t oa[32];
                tmem_ld32_async(o_col + 32u * cc, oa);
                tmem_ld_wait();
                tmem_ld_bind(oa);
#pragma unroll
                for (int e = 0; e < 32; e += 4)
                    *reinterpret_cast<float4 *>(ostage + r * kOStride + 64 * wg + 32 * cc + e) =
                        make_float4(__uint_as_float(oa[e]) * inv, __uint_as_float(oa[e + 1]) * inv,
                                    __uint_as_float(oa[e + 2]) * inv, __uint_as_float(oa[e + 3]) * inv);
            }
            if (row_ok && wg == 0 && p.merge != 2) {
                const int h = g * G + r % G;
                p.lse_part[(long)s * rows_total + ((long)b * T + j) * p.Hq + h] =
                    Lsum > 0.f ? m_used * kLn2 + logf(Lsum) : -INFINITY;
            }
        }
        if (!abort_seen) fence_proxy_async_smem();   // the staged rows, for the copy engine
        tc_fence_before();
        named_sync(1, 256);
        if (!abort_seen && sidx < M) {
            // one 512-byte bulk copy per row, by the copy engine; the thread waits
            // for its copy to land before the CTA announces its partial
            const int rr = sidx;
            float *obase = p.merge == 2 ? p.out : p.o_part + (long)s * rows_total * 128;
            float *dst = obase + (((long)b * T + j0 + rr / G) * p.Hq + g * G + rr % G) * 128;
            bulk_store_s2g(dst, smem_u32(ostage + rr * kOStride), 128 * 4);
            bulk_store_wait_all();
        }
    }

    // teardown: every MMA has completed (drain above); free tensor memory
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                     : "memory");
    }
    if (p.merge == 1)
        merge_group(p, s, g, b, mb, j0, M, G, rows_total,
                    reinterpret_cast<volatile int *>(sbase + L::kOffMisc + 12), sbase + L::kOffK);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

// 5-D map over a [B, S, Hkv, D] bf16 cache with element strides kv, the D axis
// seen as (64 columns, 2 halves) and the halves placed outside the slots:
// dims (d % 64, slot, d / 64, kv head, sequence).  One box of 64 x 128 slots x 2
// lands as two [128 slots x 128 B] blocks, the layout the MMAs read.
bool make_map(CUtensorMap *m, const void *ptr, const sd_strides &kv, int S, int Hkv, int B) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[5] = {64, (cuuint64_t)S, 2, (cuuint64_t)Hkv, (cuuint64_t)B};
    cuuint64_t strides[4] = {(cuuint64_t)kv.s * 2, 128, (cuuint64_t)kv.h * 2, (cuuint64_t)kv.b * 2};
    cuuint32_t box[5] = {64, (cuuint32_t)kBN, 2, 1, 1}, estr[5] = {1, 1, 1, 1, 1};
    const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(ptr), dims, strides, box,
                          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 4-D map over the contiguous queries [B, T, Hq, D]; box: 64 d x G heads x
// mblk_nodes block rows x 1, which lands in shared memory as rows (j - j0)*G + hl
// of 128 bytes
bool make_q_map(CUtensorMap *m, const AttnParams &p) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn) return false;
    const int G = p.Hq / p.Hkv;
    cuuint64_t dims[4] = {128, (cuuint64_t)p.Hq, (cuuint64_t)p.T, (cuuint64_t)p.B};
    cuuint64_t strides[3] = {256, (cuuint64_t)p.Hq * 256, (cuuint64_t)p.T * p.Hq * 256};
    cuuint32_t box[4] = {64, (cuuint32_t)G, (cuuint32_t)p.mblk_nodes, 1}, estr[4] = {1, 1, 1, 1};
    const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(p.q), dims, strides, box,
                          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

int cache_slots(const AttnParams &p) { return p.mode == 1 ? p.max_ctx : p.max_ctx + p.T - 1; }

cudaError_t launch_tc(const AttnParams &p, cudaStream_t st) {
    alignas(64) CUtensorMap mq, mk, mv;
    if (!make_q_map(&mq, p)) return cudaErrorInvalidValue;
    if (!make_map(&mk, p.kc, p.kv, cache_slots(p), p.Hkv, p.B)) return cudaErrorInvalidValue;
    if (!make_map(&mv, p.vc, p.kv, cache_slots(p), p.Hkv, p.B)) return cudaErrorInvalidValue;
    constexpr int smem = Layout::kSmemBytes;
    static std::atomic<bool> opted_in[64];  // per device: shared-memory limit raised
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !opted_in[dev].load(std::memory_order_acquire)) {
        e = cudaFuncSetAttribute(attn_split_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) opted_in[dev].store(true, std::memory_order_release);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.n_splits, p.Hkv * p.n_mblk, p.B);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, attn_split_tc_kernel, mq, mk, mv, p);
}

}  // namespace

bool attn_tc_supported(const AttnParams &p) {
    if (p.dt != SD_BF16 || p.D != 128 || p.T < 1 || p.T > (p.mode == 2 ? kMaxTreeT : kMaxT)) return false;
    if (p.Hq / p.Hkv > 128) return false;   // a row block holds at least one block row
    if (!(p.scale > 0.f)) return false;      // the row max is taken on the raw scores
    if ((long)p.max_ctx + p.T > (1L << 30)) return false;
    if (!encode_fn()) return false;
    int dev = 0, optin = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return false;
    if (optin < Layout::kSmemBytes) return false;
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    return major == 10 && minor == 3;
}

size_t attn_tc_smem_bytes(const AttnParams &) { return Layout::kSmemBytes; }

cudaError_t launch_attn_tc(const AttnParams &p, cudaStream_t st) { return launch_tc(p, st); }

}  // namespace sdv
