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
//   warp 1           allocates tensor memory; one thread issues the S MMAs,
//                    up to three tiles ahead
//   warp 2           one thread issues each P.V as soon as its P and V are in
//                    (two issuing threads, so that neither waits behind the
//                    other's MMAs: an MMA issue blocks while the pipe is busy)
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
constexpr int kMmaWarp = 1;                 // tensor-memory allocation, S issue
constexpr int kPvWarp = 2;                  // P.V issue
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
    static constexpr int kOffPlan = kOffLo + 16;                            // the CtaPlan
    // epilogue, once every copy and MMA is done: the staged output rows, in the
    // (then idle) K ring
    static constexpr int kOffOStage = kOffK;
    static constexpr int kSmemBytes = kOffPlan + 48 + 1024;                 // + alignment slack (CtaPlan: 48 B)
    static_assert(128 * kOStride * 4 <= kKSlots * kTileBytes, "staging fits in the K ring");
    static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
};

// ---------------------------------------------------------------------------
// work plan: which keys of which (sequence, kv head, row block) this CTA takes
// ---------------------------------------------------------------------------
// The grid is one CTA per work slot.  Unit u = (b, g, mb) has tiles_u 128-key
// tiles (its sequence's cache keys, plus the block tile that leads a drafter
// unit) and gets n_u = ceil(tiles_u / L) splits, L the smallest load for which
// sum n_u fits the C slots, so long sequences get more CTAs than short ones and
// no CTA takes more than L tiles; split s of n takes tiles
// [ceil(s tiles / n), ceil((s + 1) tiles / n)), so that the shorter shares fall
// to the last splits, the last of which holds the masked edge tile.  A unit's
// CTAs are consecutive: slot0 is its first, and its partial slots are
// slot0 .. slot0 + n - 1.  CTAs past sum n_u are idle.  Every CTA derives the same plan from ctx_len, so no plan
// crosses the host.  With more units than kPlanUnits the grid holds one CTA
// per unit.
constexpr int kPlanUnits = 5 * 32;   // units a warp plans with its lanes' registers

struct CtaPlan {      // 48 bytes, held in shared memory at Layout::kOffPlan
    int b, g, mb;        // unit
    int s, n, slot0;     // split s of n; the unit's first slot
    int k0, k1;          // cache keys [k0, k1) of the sequence's key space (clipped later)
    int block_tile;      // the drafter's block tile leads this split
    int idle;
    int nb;              // the sequence's ctx_len, clamped to [1, max_ctx]
    int tiles;           // the unit's tiles (0: not yet read)
};
static_assert(sizeof(CtaPlan) == 48, "the plan's shared-memory slot");

// tiles of unit u: its sequence's cache keys, plus the drafter's block tile
__device__ __forceinline__ int unit_tiles(const AttnParams &p, int u) {
    int nb = p.nctx[u / (p.Hkv * p.n_mblk)];
    nb = max(1, min(nb, p.max_ctx));
    const int keys = p.mode == 1 ? nb : nb + p.T - 1;
    return (keys + kBN - 1) / kBN + (p.mode == 1 ? 1 : 0);
}

// ceil(t / d) for 0 <= t < 2^24, d >= 1: a float estimate, corrected by one
__device__ __forceinline__ int ceil_div_small(int t, int d, float inv_d) {
    int q = (int)ceilf((float)t * inv_d);
    if (q > 0 && (q - 1) * d >= t) --q;
    else if (q * d < t) ++q;
    return q;
}

// Which unit and split this CTA serves (warp-collective, one full warp).
// With one sequence every unit has the same length: the grid is (splits, units)
// and the assignment needs neither a global load nor a division.  Otherwise
// the grid is one CTA per work slot and the lanes search for the load L over
// the units' tiles, read from ctx_len.
__device__ CtaPlan plan_unit(const AttnParams &p) {
    const int lane = threadIdx.x & 31;
    const int U = p.B * p.Hkv * p.n_mblk;
    const int C = (int)gridDim.x;
    const int slot = (int)blockIdx.x;
    CtaPlan pl = {};
    pl.idle = 1;
    if (p.plan_static) {
        pl.idle = 0;
        pl.b = (int)blockIdx.y;                // the unit, split into (b, g, mb) below
        pl.s = slot;
        pl.n = C;
        pl.slot0 = (int)blockIdx.y * C;
    } else if (U > kPlanUnits || U >= C) {     // one CTA per unit
        if (slot < U) { pl.idle = 0; pl.b = slot; pl.s = 0; pl.n = 1; pl.slot0 = slot; }
    } else {
        const int kU = (U + 31) / 32;          // units per lane, <= kPlanUnits / 32
        int tl[kPlanUnits / 32];
        int tmax = 1;
        long tot = 0;
#pragma unroll
        for (int k = 0; k < kPlanUnits / 32; ++k) {
            const int u = lane + 32 * k;
            tl[k] = (k < kU && u < U) ? unit_tiles(p, u) : 0;
            tmax = max(tmax, tl[k]);
            tot += tl[k];
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            tmax = max(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
            tot += __shfl_xor_sync(0xffffffffu, tot, o);
        }
        // smallest L in [ceil(tot / C), tmax] with sum ceil(tiles_u / L) <= C:
        // each round the 32 lanes try 32 loads spread over the range at once
        // (the count falls as L grows, and L = tmax always fits: U <= C)
        int lo = (int)max(1L, (tot + C - 1) / C), hi = tmax;
        while (lo < hi) {
            const int span = hi - lo;
            const int cand = lo + (int)((long)lane * span / 31);   // lane 0: lo, lane 31: hi
            const float inv_c = 1.0f / (float)cand;
            int cnt = 0;
#pragma unroll
            for (int k = 0; k < kPlanUnits / 32; ++k) {
                if (k >= kU) break;
#pragma unroll 8
                for (int src = 0; src < 32; ++src) {
                    const int t = __shfl_sync(0xffffffffu, tl[k], src);   // 0 past the last unit
                    cnt += ceil_div_small(t, cand, inv_c);
                }
            }
            const unsigned fits = __ballot_sync(0xffffffffu, cnt <= C);
            const int f = __ffs((int)fits) - 1;                     // lane 31 (hi) always fits
            const int new_hi = __shfl_sync(0xffffffffu, cand, f);
            const int below = __shfl_sync(0xffffffffu, cand, max(f - 1, 0));
            lo = f > 0 ? below + 1 : lo;
            hi = new_hi;
        }
        const float inv = 1.0f / (float)lo;
        int base = 0;
#pragma unroll
        for (int k = 0; k < kPlanUnits / 32; ++k) {
            if (k >= kU) break;
            const int u = lane + 32 * k;
            const int nu = ceil_div_small(tl[k], lo, inv);   // 0 past the last unit
            int incl = nu;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            const int excl = base + incl - nu;
            const unsigned hit = __ballot_sync(0xffffffffu, u < U && slot >= excl && slot < excl + nu);
            if (hit) {
                const int src = __ffs((int)hit) - 1;
                pl.idle = 0;
                pl.b = 32 * k + src;   // the unit, split into (b, g, mb) below
                pl.n = __shfl_sync(0xffffffffu, nu, src);
                pl.slot0 = __shfl_sync(0xffffffffu, excl, src);
                pl.s = slot - pl.slot0;
                pl.tiles = __shfl_sync(0xffffffffu, tl[k], src);
                break;
            }
            base += __shfl_sync(0xffffffffu, incl, 31);
        }
    }
    if (!pl.idle) {
        const int u = pl.b;
        if (p.n_mblk == 1) {
            pl.b = p.B == 1 ? 0 : u / p.Hkv;
            pl.g = p.B == 1 ? u : u - pl.b * p.Hkv;
            pl.mb = 0;
        } else {
            pl.b = u / (p.Hkv * p.n_mblk);
            pl.g = (u / p.n_mblk) % p.Hkv;
            pl.mb = u % p.n_mblk;
        }
    }
    return pl;
}

// the split's cache keys, from its unit's tiles; ctx_b: ctx_len of the CTA's
// sequence, loaded by the caller
__device__ void plan_keys(const AttnParams &p, CtaPlan &pl, int ctx_b) {
    const int lead = p.mode == 1 ? 1 : 0;
    pl.nb = max(1, min(ctx_b, p.max_ctx));
    if (pl.tiles == 0) pl.tiles = ((p.mode == 1 ? pl.nb : pl.nb + p.T - 1) + kBN - 1) / kBN + lead;  // < 2^24
    const int tiles = pl.tiles;
    const int a = (pl.s * tiles + pl.n - 1) / pl.n;                                 // products < 2^31
    const int e = ((pl.s + 1) * tiles + pl.n - 1) / pl.n;
    pl.k0 = max(0, a - lead) * kBN;
    pl.k1 = max(0, e - lead) * kBN;
    pl.block_tile = lead && a == 0 && e > 0;   // an empty split [0, 0) takes nothing
}

// ---------------------------------------------------------------------------
// merge of the splits inside the kernel
// ---------------------------------------------------------------------------
// Bounded wait until the counter reaches `target`.
__device__ __noinline__ bool wait_count(const unsigned int *ctr, unsigned int target, unsigned long long limit_ns) {
    const unsigned long long t0 = global_timer();
    for (uint32_t it = 0;; ++it) {
        unsigned int v;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
        if (v >= target) return true;
        if ((it & 15u) == 15u && global_timer() - t0 > limit_ns) return false;
        __nanosleep(32);
    }
}

// Every split of unit (b, g, mb) has written its partial into its slot (rows
// normalised by their own sum, plus their log-sum-exp); once all n of them
// have arrived, split s combines rows s, s + n, s + 2n, ... of the unit's M
// rows (row rr is block row j0 + rr / G, query head g G + rr % G):
// out = sum_s w_s o_s / sum_s w_s with w_s = exp(lse_s - max).
// The whole grid is resident (at most one CTA per SM), so the wait ends.  The
// counter is returned to zero by the last split to finish merging.  `scratch`
// is idle shared memory (the K/V rings).
constexpr int kMergeBatch = 12;  // loads one merge thread keeps in flight
constexpr int kMergeSmall = 6;   // a chunk of at most this many splits takes the grouped path
constexpr int kMergeUnits = 3;   // units a merge thread loads together on that path
__device__ void merge_group(const AttnParams &p, const CtaPlan &pl, int j0, int M, int G, volatile int *go,
                            uint8_t *scratch) {
    const int s = pl.s, g = pl.g, b = pl.b;
    unsigned int *ctr = p.merge_ctr + (((long)b * p.Hkv + g) * p.n_mblk + pl.mb);
    const int n = pl.n;
    const int tid = threadIdx.x;
    // the arrival is a release by thread 0 after the CTA barrier: it covers
    // every thread's partial (the bulk copies each thread waited for, the
    // log-sum-exps) for whoever acquires the count
    __syncthreads();
    // every split takes a second ticket once its wait is over, whether or not
    // it succeeded, so the counter sees exactly 2n increments per launch and
    // the split holding the last of them returns it to zero (no split reads
    // it any more by then): a launch whose wait gave up (fault bit set, its
    // rows left unmerged) still leaves the workspace ready for the next call.
    // The ticket goes out now and its value is used only when the split ends,
    // so its round trip overlaps the merge.
    unsigned int ticket = 0u;
    if (tid == 0) {
        asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(ctr) : "memory");
        const bool ok = wait_count(ctr, (unsigned int)n + p.wt.extra, p.wt.limit_ns);
        if (!ok) set_fault(p.fault, FAULT_WAIT_TIMEOUT);
        *go = ok ? 1 : 0;
        ticket = atomicAdd(ctr, 1u);
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
        if (chunk <= kMergeSmall) {
            // few splits per chunk: a thread's units go kMergeUnits at a time,
            // every load of the group in flight together (one round trip for
            // up to kMergeUnits units instead of one each)
            for (int u0 = tid; u0 < K * R * 32; u0 += kMergeUnits * kTcThreads) {
                float4 v[kMergeUnits][kMergeSmall];
                float l[kMergeUnits][kMergeSmall];
#pragma unroll
                for (int q = 0; q < kMergeUnits; ++q) {
                    const int u = u0 + q * kTcThreads;
                    const bool live = u < K * R * 32;
                    const int uu = live ? u : u0;
                    const int k = uu / (R * 32), ri = (uu / 32) % R, c4 = uu & 31;
                    const int sp0 = k * chunk, sp1 = min(n, sp0 + chunk);
#pragma unroll
                    for (int e = 0; e < kMergeSmall; ++e) {
                        const long prow = (long)(pl.slot0 + min(sp0 + e, sp1 - 1)) * 128 + s + ri * n;
                        v[q][e] = live && sp0 + e < sp1
                                      ? __ldcg(reinterpret_cast<const float4 *>(p.o_part + prow * 128) + c4)
                                      : make_float4(0.f, 0.f, 0.f, 0.f);
                        l[q][e] = live && sp0 + e < sp1 ? __ldcg(p.lse_part + prow) : -INFINITY;
                    }
                }
#pragma unroll
                for (int q = 0; q < kMergeUnits; ++q) {
                    const int u = u0 + q * kTcThreads;
                    if (u >= K * R * 32) break;
                    float m_run = l[q][0];
#pragma unroll
                    for (int e = 1; e < kMergeSmall; ++e) m_run = fmaxf(m_run, l[q][e]);
                    float w_run = 0.f;
                    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (m_run != -INFINITY) {
#pragma unroll
                        for (int e = 0; e < kMergeSmall; ++e) {
                            const float w = __expf(l[q][e] - m_run);   // 0 for an empty or repeated split
                            w_run += w;
                            acc.x = fmaf(w, v[q][e].x, acc.x); acc.y = fmaf(w, v[q][e].y, acc.y);
                            acc.z = fmaf(w, v[q][e].z, acc.z); acc.w = fmaf(w, v[q][e].w, acc.w);
                        }
                    }
                    pacc[u] = acc;
                    pm[u] = m_run;
                    pw[u] = w_run;
                }
            }
        } else {
        for (int u = tid; u < K * R * 32; u += kTcThreads) {
            const int k = u / (R * 32), ri = (u / 32) % R, c4 = u & 31;
            const int sp0 = k * chunk, sp1 = min(n, sp0 + chunk);
            float m_run = -INFINITY, w_run = 0.f;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int sb = sp0; sb < sp1; sb += kMergeBatch) {
                // every load of the batch is issued before any is used, so
                // that all are in flight at once; past the chunk's end the
                // loads are predicated off (no traffic) and the entry carries
                // weight zero
                float4 v[kMergeBatch];
                float l[kMergeBatch];
#pragma unroll
                for (int e = 0; e < kMergeBatch; ++e) {
                    const long prow = (long)(pl.slot0 + min(sb + e, sp1 - 1)) * 128 + s + ri * n;  // slot, row
                    v[e] = sb + e < sp1 ? __ldcg(reinterpret_cast<const float4 *>(p.o_part + prow * 128) + c4)
                                        : make_float4(0.f, 0.f, 0.f, 0.f);
                    l[e] = sb + e < sp1 ? __ldcg(p.lse_part + prow) : -INFINITY;
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
    if (tid == 0 && ticket == 2u * (unsigned int)n - 1u) atomicExch(ctr, 0u);
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kTcThreads, 1)
attn_split_tc_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                     const __grid_constant__ CUtensorMap tmap_v, const __grid_constant__ CUtensorMap tmap_kb,
                     const __grid_constant__ CUtensorMap tmap_vb, const AttnParams p) {
    using L = Layout;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    const uint32_t base = (raw_u32 + 1023u) & ~1023u;
    uint8_t *sbase = smem_raw + (base - raw_u32);

    // grid: one CTA per work slot, or (split, unit) for one sequence (plan_unit)
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
    CtaPlan *plan_sh = reinterpret_cast<CtaPlan *>(sbase + L::kOffPlan);

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
        if (p.mode == 1) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_kb)) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_vb)) : "memory");
        }
    }
    if (warp == kMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_holder)), "r"(kTmemCols) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
#if __CUDA_ARCH__ >= 900
    // inputs of the upstream kernel are visible past the wait.  No early
    // trigger: the dependents launch as this kernel's CTAs exit (an early one
    // let the next kernel's CTAs occupy the idle SMs only to wait there, and
    // made a step of the five attention calls and the acceptance slower)
    asm volatile("griddepcontrol.wait;" ::: "memory");
#endif

    // the plan: warp 0 works it out, its lane 0 starts the Q copy and its
    // lanes the first K/V copies before the CTA-wide barrier; the other warps
    // read the plan after it
    const int T = p.T, G = p.Hq / p.Hkv;
    const int MQ = G * p.mblk_nodes;  // rows the Q copy writes (those past block row T - 1 as zeros)
    CtaPlan pl = {};
    if (warp == kProducerWarp) {
        pl = plan_unit(p);
        // the sequence's length, loaded ahead of the Q copy so that the two overlap
        const int ctx_b = pl.idle ? 1 : p.nctx[pl.b];
        if (producer && !pl.idle) {
            // Q first: rows r = (j - j0)*G + hl of this kv head, two 64-column halves;
            // the copy always moves the whole box (out-of-range rows are zero-filled)
            mbar_arrive_expect_tx(qready_bar, (uint32_t)(256 * MQ));
            tma_load_4d(sQ, &tmap_q, qready_bar, 0, pl.g * G, pl.mb * p.mblk_nodes, pl.b);
            tma_load_4d(sQ + 128 * 128, &tmap_q, qready_bar, 64, pl.g * G, pl.mb * p.mblk_nodes, pl.b);
        }
        if (!pl.idle) plan_keys(p, pl, ctx_b);
        if (lane == 0) *plan_sh = pl;
    }
    // a split's tiles: the cache keys [k0, cend) of its sequence, after the
    // drafter's block tile when it leads the split
    struct Tiles {
        int nb, k0, cend, n_tiles, lead_blk;
    };
    auto tiles_of = [&](const CtaPlan &q) {
        Tiles r;
        r.nb = q.nb;
        r.k0 = q.k0;
        r.cend = p.mode == 1 ? min(q.k1, r.nb) : min(q.k1, r.nb + T - 1);
        const int n_cache = r.cend > r.k0 ? (r.cend - r.k0 + kBN - 1) / kBN : 0;
        r.lead_blk = q.block_tile ? 1 : 0;   // tile 0 of the drafter's leading split is the block
        r.n_tiles = n_cache + r.lead_blk;
        return r;
    };
    // one copy per tile: map coordinates (d within a half, key, half, kv head,
    // sequence); the drafter's block tile comes from the [B, T, Hkv, D] block
    // keys / values, whose rows past T the copy fills with zeros
    auto issue_k = [&](const CtaPlan &q, const Tiles &r, int t) {
        const int sl = t % kKSlots;
        mbar_arrive_expect_tx(kfull_bar(sl), (uint32_t)kTileBytes);
        if (t < r.lead_blk) tma_load_5d(sK + sl * kTileBytes, &tmap_kb, kfull_bar(sl), 0, 0, 0, q.g, q.b);
        else tma_load_5d(sK + sl * kTileBytes, &tmap_k, kfull_bar(sl), 0, r.k0 + (t - r.lead_blk) * kBN, 0, q.g, q.b);
    };
    auto issue_v = [&](const CtaPlan &q, const Tiles &r, int t) {
        const int sl = t % kVSlots;
        mbar_arrive_expect_tx(vfull_bar(sl), (uint32_t)kTileBytes);
        if (t < r.lead_blk) tma_load_5d(sV + sl * kTileBytes, &tmap_vb, vfull_bar(sl), 0, 0, 0, q.g, q.b);
        else tma_load_5d(sV + sl * kTileBytes, &tmap_v, vfull_bar(sl), 0, r.k0 + (t - r.lead_blk) * kBN, 0, q.g, q.b);
    };
    // first wave, before the CTA-wide barrier: the first tile's K and V, one
    // copy per lane of the producer warp; the other slots fill after the
    // barrier (every CTA's first tile then comes back ahead of the rest of
    // the grid's second and third)
    constexpr int kFirstWave = 1;
    if (warp == kProducerWarp && !pl.idle) {
        const Tiles r = tiles_of(pl);
        const int w = min(r.n_tiles, kFirstWave);
        if (lane < w) issue_k(pl, r, lane);
        else if (lane >= 8 && lane - 8 < w) issue_v(pl, r, lane - 8);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp != kProducerWarp) pl = *plan_sh;
    if (pl.idle) {
        // no work for this slot: give the tensor memory back and leave
        if (warp == kMmaWarp) {
            tc_fence_after();
            asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(*tmem_holder),
                         "r"(kTmemCols) : "memory");
        }
        return;
    }
    const int g = pl.g, mb = pl.mb, b = pl.b;
    const int slot = pl.slot0 + pl.s;  // this split's partial slot
    const bool direct = pl.n == 1;  // a unit's only split writes the output itself
    // this CTA's rows: block rows [j0, j0 + Tb) of the G query heads of kv head g
    const int j0 = mb * p.mblk_nodes, Tb = min(p.mblk_nodes, T - j0), M = G * Tb;
    const bool drafter = p.mode == 1;
    if (tid == 0 && (p.nctx[b] < 1 || p.nctx[b] > p.max_ctx)) set_fault(p.fault, FAULT_BAD_CTX);
    const Tiles tr = tiles_of(pl);
    const int nb = tr.nb, cend = tr.cend, n_tiles = tr.n_tiles, lead_blk = tr.lead_blk;
    const bool has_block_tile = lead_blk != 0;
    auto tile_key0 = [&](int t) { return tr.k0 + (t - lead_blk) * kBN; };
    auto is_block_tile = [&](int t) { return has_block_tile && t == 0; };
    // keys every row of the block sees: the drafter's context, the target's
    // cache before the block (before the anchor for a tree)
    const bool tree = p.mode == 2;
    const int all_see = min(cend, tree ? nb - 1 : nb);
    // copies the first wave issued
    int next_k = min(n_tiles, kFirstWave), next_v = next_k;
    static_assert(kFirstWave <= kKSlots && kFirstWave <= kVSlots, "the first wave fits both rings");
    auto issue_k_t = [&](int t) { issue_k(pl, tr, t); };
    auto issue_v_t = [&](int t) { issue_v(pl, tr, t); };

    const uint32_t tmem = *tmem_holder;

    if (n_tiles == 0) {
        // nothing to read: an empty split (lse = -inf, zero partial) for the merge;
        // the Q copy issued above lands before the CTA exits
        if (producer) mbar_wait(qready_bar, 0, nullptr, p.fault);
        for (int idx = tid; idx < M * 32; idx += kTcThreads) {
            const int rr = idx >> 5, c4 = idx & 31;
            const long frow = ((long)b * T + j0 + rr / G) * p.Hq + g * G + rr % G;
            float *dst = direct ? p.out + frow * 128 : p.o_part + ((long)slot * 128 + rr) * 128;
            reinterpret_cast<float4 *>(dst)[c4] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (c4 == 0 && !direct) p.lse_part[(long)slot * 128 + rr] = -INFINITY;
        }
    } else if (warp == kProducerWarp) {
        // ------------------------------------------------------------------ producer
        if (lane == 0) {
            // whichever ring has a free slot first: a K slot frees when its S has
            // completed, a V slot when its P.V has, so neither waits behind the other
            unsigned long long t_last = global_timer();
            for (uint32_t spin = 0; next_k < n_tiles || next_v < n_tiles;) {
                if (next_k < n_tiles &&
                    (next_k < kKSlots || mbar_test(kempty_bar(next_k % kKSlots), ((next_k / kKSlots) - 1) & 1))) {
                    issue_k_t(next_k++);
                    t_last = global_timer();
                    continue;
                }
                if (next_v < n_tiles &&
                    (next_v < kVSlots || mbar_test(vempty_bar(next_v % kVSlots), ((next_v / kVSlots) - 1) & 1))) {
                    issue_v_t(next_v++);
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
                for (int u = max(0, next_k - kKSlots); u < next_k; ++u)
                    mbar_wait(kfull_bar(u % kKSlots), (u / kKSlots) & 1, nullptr, p.fault);
                for (int u = max(0, next_v - kVSlots); u < next_v; ++u)
                    mbar_wait(vfull_bar(u % kVSlots), (u / kVSlots) & 1, nullptr, p.fault);
            }
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------------ S issuer
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
            // S(ns) into S/P buffer ns % 3 as soon as its keys have landed and
            // P.V(ns - 3) has read the buffer: S runs up to three tiles ahead.
            // S and P.V go out from two threads, each waiting only for its own
            // inputs: one thread issuing both held every P.V behind the next S
            // (an MMA issue blocks while the tensor pipe is busy), and with it
            // the V slot the P.V frees
            const uint32_t idS = idesc_bf16(128, kBN, false);
            bool ok = mbar_wait(qready_bar, 0, abort_flag, p.fault);
            unsigned long long t_last = global_timer();
            int next_s = 0;
            for (uint32_t spin = 0; ok && next_s < n_tiles;) {
                const int ns = next_s;
                if (mbar_test(kfull_bar(ns % kKSlots), (ns / kKSlots) & 1) &&
                    (ns < kSP || mbar_test(pempty_bar(ns % kSP), ((ns / kSP) - 1) & 1))) {
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
                    ++next_s;
                    t_last = global_timer();
                    continue;
                }
                // nothing ready yet: poll again (the bound below still holds); a
                // back-off here only delays the reaction, the poll costs little
                if ((++spin & 15u) == 0) {
                    if (*abort_flag) ok = false;
                    else if (global_timer() - t_last > kWaitLimitNs) {
                        *abort_flag = 1;
                        set_fault(p.fault, FAULT_WAIT_TIMEOUT);
                        ok = false;
                    }
                }
            }
        }
        __syncwarp();
    } else if (warp == kPvWarp) {
        // ------------------------------------------------------------------ P.V issuer
        if (lane == 0) {
            const uint32_t idO = idesc_bf16(128, 128, true);
            bool ok = true;
            unsigned long long t_last = global_timer();
            int next_pv = 0;
            for (uint32_t spin = 0; ok && next_pv < n_tiles;) {
                const int npv = next_pv;
                if (mbar_test(pfull_bar(npv % kSP), (npv / kSP) & 1) &&
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
                    ++next_pv;
                    t_last = global_timer();
                    continue;
                }
                if ((++spin & 15u) == 0) {
                    if (*abort_flag) ok = false;
                    else if (global_timer() - t_last > kWaitLimitNs) {
                        *abort_flag = 1;
                        set_fault(p.fault, FAULT_WAIT_TIMEOUT);
                        ok = false;
                    }
                }
            }
            // every MMA has completed before tensor memory is freed: the last
            // P.V follows every S (its P needed S), and this thread issued it
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
        // this row's tree word, read once (the edge tiles use it)
        const uint64_t row_tm = tree && row_ok ? p.tree_mask[(long)b * T + j] : 0ull;
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
                    const uint64_t tm = row_tm;
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
            // the P arrival, by the P.V issuer
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
            // packed fp32 pairs (one instruction for two lanes' worth of FMA or
            // add): the argument of each exponential pair, and two pairs of
            // partial sums
            float2 ls2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
            const float2 qk2 = make_float2(qk, qk), nm2 = make_float2(neg_m, neg_m);
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
                        const float2 x = __ffma2_rn(make_float2(__uint_as_float(sq[2 * c]),
                                                                __uint_as_float(sq[2 * c + 1])), qk2, nm2);
                        const float p0 = ex2(x.x), p1 = ex2(x.y);
                        ls2[c & 1] = __fadd2_rn(ls2[c & 1], make_float2(p0, p1));
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
                        const float2 x = __ffma2_rn(make_float2(__uint_as_float(sq[2 * c]),
                                                                __uint_as_float(sq[2 * c + 1])), qk2, nm2);
                        const float p0 = ex2(x.x), p1 = ex2(x.y);
                        const __nv_bfloat162 h2 = __floats2bfloat162_rn(p0, p1);   // .x = p0 in the low half
                        const uint32_t h = *reinterpret_cast<const uint32_t *>(&h2);
                        pk[c] = h;
                        ls2[c & 1] = __fadd2_rn(ls2[c & 1], make_float2(__uint_as_float(h << 16),
                                                                        __uint_as_float(h & 0xffff0000u)));
                    }
                    tmem_st16(sp_col + 16u * q, pk);
                }
            }
            l += (ls2[0].x + ls2[1].x) + (ls2[0].y + ls2[1].y);
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
        // the row sum first (it needs no MMA), then the wait for the last P.V
        named_sync(1, 256);
        xrow[wg * 128 + r] = l;
        named_sync(1, 256);
        const int last_t = n_tiles - 1;
        ok = __all_sync(0xffffffffu,
                        mbar_wait(pempty_bar(last_t % kSP), (last_t / kSP) & 1, abort_flag, p.fault)) && ok;
        float Lsum = wg == 0 ? l + xrow[128 + r] : xrow[r] + l;  // same order in both
        if (!ok) { m_used = -INFINITY; l = 0.f; Lsum = 0.f; }
        tc_fence_before();
        // the last P.V, hence every MMA (and every copy they read), is complete
        // past this point: the rings are free for the staging
        named_sync(1, 256);
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
            if (row_ok && wg == 0 && !direct)
                p.lse_part[(long)slot * 128 + r] = Lsum > 0.f ? m_used * kLn2 + logf(Lsum) : -INFINITY;
        }
        if (!abort_seen) fence_proxy_async_smem();   // the staged rows, for the copy engine
        tc_fence_before();
        named_sync(1, 256);
        if (!abort_seen && sidx < M) {
            // one 512-byte bulk copy per row, by the copy engine; the thread waits
            // for its copy to land before the CTA announces its partial
            const int rr = sidx;
            float *dst = direct ? p.out + (((long)b * T + j0 + rr / G) * p.Hq + g * G + rr % G) * 128
                                : p.o_part + ((long)slot * 128 + rr) * 128;
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
    if (!direct)
        merge_group(p, pl, j0, M, G, reinterpret_cast<volatile int *>(sbase + L::kOffMisc + 12), sbase + L::kOffK);
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
    alignas(64) CUtensorMap mq, mk, mv, mkb, mvb;
    if (!make_q_map(&mq, p)) return cudaErrorInvalidValue;
    if (!make_map(&mk, p.kc, p.kv, cache_slots(p), p.Hkv, p.B)) return cudaErrorInvalidValue;
    if (!make_map(&mv, p.vc, p.kv, cache_slots(p), p.Hkv, p.B)) return cudaErrorInvalidValue;
    if (p.mode == 1) {
        // the drafter's block keys / values [B, T, Hkv, D], contiguous: T slots
        // per sequence, so a 128-slot box reads rows past T as zeros
        const sd_strides blk = {(int64_t)p.T * p.Hkv * 128, (int64_t)p.Hkv * 128, 128};
        if (!make_map(&mkb, p.kb, blk, p.T, p.Hkv, p.B)) return cudaErrorInvalidValue;
        if (!make_map(&mvb, p.vb, blk, p.T, p.Hkv, p.B)) return cudaErrorInvalidValue;
    } else {
        mkb = mk;   // not read
        mvb = mv;
    }
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
    // one CTA per work slot, or (splits, units) for one sequence (plan_unit)
    cfg.gridDim = p.plan_static ? dim3(p.n_splits / (p.B * p.Hkv * p.n_mblk), p.B * p.Hkv * p.n_mblk)
                                : dim3(p.n_splits);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    // the splits of a unit that merge inside the kernel wait for one another:
    // with at most one CTA per SM the grid goes out as a cooperative launch,
    // which makes every CTA resident at once; a device that cannot hold it (a
    // partitioned one) refuses the launch, and the caller takes the CUDA-core
    // kernel, whose splits never wait
    const bool coop = (long)cfg.gridDim.x * cfg.gridDim.y <= device_sm_count();
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeCooperative;
    attr[1].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = coop ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, attn_split_tc_kernel, mq, mk, mv, mkb, mvb, p);
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
