// Internal interface between the C-ABI layer (api.cu) and the kernel files.
// Not installed; callers use include/sd_verify.h.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/sd_verify.h"

namespace sdv {

// Fault word bits set by device-side guards (never a trap).
enum FaultBits : unsigned int {
    FAULT_BAD_CTX = 1u << 0,        // ctx_len / n_ctx outside [1, max_ctx]
    FAULT_BAD_DRAFT_ID = 1u << 1,   // draft id outside [0, V)
    FAULT_NAN_ROW = 1u << 2,        // argmax row without any ordered value (NaN)
    FAULT_WAIT_TIMEOUT = 1u << 3,   // a bounded mbarrier wait gave up
    FAULT_TMEM_ALLOC = 1u << 4,     // tensor-memory allocation returned out of range
    FAULT_BAD_TREE = 1u << 5,       // a tree node's parent outside [0, node)
    FAULT_BAD_COMMIT = 1u << 6,     // a commit with n_acc / path / lengths out of range (skipped)
};

constexpr int kMaxT = 16;           // block rows (anchor + 15 proposals)
constexpr int kMaxTreeT = 64;       // nodes of a draft tree (one 64-bit ancestor mask per node)
constexpr int kTileKeys = 64;       // keys per tile of the CUDA-core attention kernel
constexpr int kTcTileKeys = 128;    // keys per tile of the tensor-core attention kernel
constexpr int kMaxHeadBytes = 512;  // bytes of one (position, kv head) row the tree compaction moves

constexpr unsigned long long kBarrierWaitNs = 2000000000ull;   // an in-kernel barrier wait gives up after 2 s

// Failure-detection test hook (sd_set_wait_test): the in-kernel barriers
// (attention merge, one-launch sampled rule) wait for `extra` arrivals more
// than exist, giving up after `limit_ns`.  {0, kBarrierWaitNs} normally.
struct WaitTest {
    unsigned int extra;
    unsigned long long limit_ns;
};
WaitTest wait_test();

// Attention launch description (both the target verify and the drafter).
//  key index space of sequence b:
//   mode 0 (verify):  N_b = nctx[b] + T - 1 cache keys; row j sees [0, nctx[b] + j)
//   mode 1 (drafter): N_b = nctx[b] + T; keys [0, nctx[b]) from the cache,
//                     [nctx[b], N_b) from the block tensors; every row sees all
//   mode 2 (tree):    N_b = nctx[b] + T - 1 cache keys; row j sees
//                     [0, nctx[b] - 1) and block slot nctx[b] - 1 + k for every
//                     bit k set in tree_mask[b * T + j]
//  split s covers keys [s * keys_per_split, (s + 1) * keys_per_split) of that space.
//  The tensor-core kernel cuts a kv head's G*T query rows into n_mblk row
//  blocks of mblk_nodes whole block rows (G * mblk_nodes <= 128 rows each);
//  the blocks of one split read the same K/V tiles.
struct AttnParams {
    const void *q;                  // [B, T, Hq, D]
    const void *kc, *vc;            // [B, S, Hkv, D] with strides kv
    sd_strides kv;
    const int32_t *nctx;            // [B]
    int mode;
    const void *kb, *vb;            // [B, T, Hkv, D] (mode 1)
    const uint64_t *tree_mask;      // [B, T] (mode 2)
    float *out;                     // [B, T, Hq, D]
    int B, T, Hq, Hkv, D;
    sd_dtype dt;
    float scale;
    int max_ctx;                    // host bound of nctx
    int s_rows;                     // cache slots available per sequence (derived bound)
    int n_splits, keys_per_split;
    int n_mblk, mblk_nodes;         // tensor-core kernel: row blocks per kv head, block rows per row block
    int plan_static;                // tensor-core kernel: grid (splits, units) instead of one CTA per work slot
    float *o_part;                  // [n_splits, B*T*Hq, D]
    float *lse_part;                // [n_splits, B*T*Hq]
    // how the splits are combined: 0 a separate merge kernel, 1 merged inside
    // the split kernel once every split of a (sequence, kv head, row block) has
    // arrived (counters merge_ctr[B * Hkv * n_mblk], zero between calls), 2 a
    // single split that writes the output itself
    int merge;
    unsigned int *merge_ctr;
    WaitTest wt;
    unsigned int *fault;
};

// kernel launchers: return the launch error (cudaSuccess when enqueued)
cudaError_t launch_attn_generic(const AttnParams &p, cudaStream_t st);
cudaError_t launch_attn_tc(const AttnParams &p, cudaStream_t st);
cudaError_t launch_lse_merge(const AttnParams &p, cudaStream_t st);
bool attn_tc_supported(const AttnParams &p);
size_t attn_tc_smem_bytes(const AttnParams &p);

// Acceptance workspaces hold ticket counters that must be zero before the
// first call and are returned to zero by every completed call.
struct GreedyParams {
    const int32_t *draft;           // chain: [B, T-1] proposals; tree: [B, T] node tokens
    const int32_t *parents;         // tree only: [B, T], parents[b][0] = -1, parents[b][j] < j
    int32_t *path;                  // tree only: [B, T] accepted nodes at depth 1..n, then -1
    const void *logits;
    int B, T, V;
    sd_dtype dt;
    int32_t *n_acc, *corr;
    int chunk, n_chunks;
    unsigned int *counter;          // CTAs finished
    float *pval;                    // [B*T, n_chunks] chunk max
    int *pidx;                      // [B*T, n_chunks] its index
    unsigned int *fault;
};
cudaError_t launch_accept_greedy(const GreedyParams &p, cudaStream_t st);

struct SampleParams {
    const int32_t *draft;
    const float *q;
    const void *logits;
    int B, T, V;
    sd_dtype dt;
    float inv_tau;
    uint64_t seed;
    uint32_t offset;
    int32_t *n_acc, *next_id;
    int chunk, n_chunks;            // pass 1 chunks (streamed)
    int draw_chunk, n_draw_chunks;  // pass 2 chunks, draw_chunk <= kDrawChunkMax
    unsigned int *counters;         // [0]: CTAs of pass 1 finished
    unsigned int *row_counter;      // [B] CTAs of pass 2 finished per sequence
    float *pm;                      // [B*T, n_chunks] chunk max
    float2 *pz;                     // [B*T, n_chunks] chunk sum of exp (hi, lo: a float-float value)
    float2 *row_stats;              // [B*T] (logit, q) of the row's proposal
    float4 *state;                  // [B]: (n as int bits, M, Z, unused) of the deciding row
    float2 *rs;                     // [B, n_draw_chunks] chunk sums of the draw's weights (hi, lo)
    // the one-launch form: counters[1..2] its grid barrier (arrivals,
    // departures), row_counter [2B] the barriers of the sequences
    int seg, n_segs;                // the B*T*V logits as n_segs segments of seg (<= V) elements
    int fchunk, n_fchunks;          // chunks of the deciding row, one CTA each
    float4 *pp;                     // [n_segs, 2] (max, sum hi, sum lo, -) of a segment's two row pieces
    float4 *fs;                     // [B, n_fchunks] (residual sum hi, lo, p sum hi, lo) of each chunk
    WaitTest wt;
    unsigned int *fault;
};
constexpr int kMaxDevices = 64;          // devices whose per-device caches the library keeps
constexpr int kSampleFusedPerSm = 2;     // CTAs per SM of the one-launch sampled rule
constexpr int kDrawChunkMax = 4096;  // pass 2 chunk bound: 16 elements per thread of the in-chunk search
cudaError_t launch_accept_sample(const SampleParams &p, cudaStream_t st);
// the one-launch form: a cooperative grid of `grid` CTAs, all resident
cudaError_t launch_accept_sample_fused(const SampleParams &p, int grid, cudaStream_t st);
int sample_fused_per_sm(sd_dtype dt, int nv);   // its resident CTAs per SM (0: none)
int sample_vec_per_thread(sd_dtype dt, int chunk);

// Drafter K/V projector: k_out[n] = h[n] . wk^T, v_out[n] = h[n] . wv^T for
// rows n < N; h [N, Hd] row stride ld_h, wk / wv [Dout, Hd] contiguous,
// outputs row stride ld_out (elements).
struct ProjParams {
    const __nv_bfloat16 *h;
    const __nv_bfloat16 *wk, *wv;
    __nv_bfloat16 *k_out, *v_out;
    long ld_h, ld_out;
    int N, Hd, Dout;
    // commit-time append (launch_project_commit): sequence b's rows are
    // 0..n_acc[b] of its block (row r >= 1 is node path[b * T + r - 1] when
    // path is given), read at h + b * h_bstride, written to output rows
    // dst_row0[b] + r at k_out / v_out + b * out_bstride; max_rows bounds them
    const int32_t *n_acc, *path, *dst_row0;
    long h_bstride, out_bstride;
    int B, T, max_rows;
    unsigned int *fault;
};
constexpr int kProjSmallRows = 16;  // rows per CTA of the CUDA-core projector
constexpr size_t kProjSmallSmemMax = 200 * 1024;  // its hidden rows staged in shared memory
// path: 1 CUDA cores, 2 tensor cores (requires project_tc_supported())
cudaError_t launch_project(const ProjParams &p, int path, cudaStream_t st);
bool project_tc_supported();
bool project_small_supported(int rows_per_cta, int Hd);  // those rows of Hd fit its shared memory
cudaError_t launch_project_commit(const ProjParams &p, cudaStream_t st);

// Commit of a verified block: tokens and lengths (one warp per sequence) and,
// for trees, the move of the kept nodes' K/V rows to consecutive positions.
struct CommitParams {
    const int32_t *prop;            // [B, ps] proposals (chain drafts or tree node tokens)
    int ps;
    const int32_t *path;            // tree: [B, T] kept nodes by depth; chain: null
    const int32_t *n_acc, *next_tok;
    int B, T;
    int32_t *ctx_len;
    int ctx_cap;
    int32_t *draft_ctx;             // nullable
    int32_t *out_tokens;            // [B, out_cap]
    int32_t *out_len;
    int out_cap;
    int32_t *anchor;
    int32_t *status;                // nullable
    unsigned int *fault;
};
cudaError_t launch_commit_tokens(const CommitParams &p, cudaStream_t st);

// Results into pinned host memory by SM stores (16-byte vectors), through the
// host buffer's device-visible address.
struct HostStoreParams {
    const uint4 *src;               // device memory
    uint4 *dst;                     // device-visible address of pinned host memory
    int64_t n16;                    // 16-byte vectors
};
cudaError_t launch_store_to_host(const HostStoreParams &p, int sm_count, cudaStream_t st);

struct CompactParams {
    void *kc, *vc;                  // [B, S, Hkv, D] with strides kv (elements)
    sd_strides kv;
    int es;                         // bytes per element
    const int32_t *ctx_len, *path, *n_acc;
    int B, T, S, Hkv, D;
    unsigned int *fault;
};
cudaError_t launch_compact_tree_kv(const CompactParams &p, cudaStream_t st);

// SpecFLASH latent compressor: out[i] = softmax(q . f[i]^T) . f[i] per frame i.
constexpr int kLatentMaxQueries = 64;
constexpr int kLatentStageD = 256;  // d per stage of the scores kernel
struct LatentParams {
    const __nv_bfloat16 *q;         // [Cq, d] contiguous
    const __nv_bfloat16 *f;         // frame i, feature n at f + i * f_fstride + n * ld_f
    long ld_f, f_fstride;
    __nv_bfloat16 *out;             // frame i, query c at out + i * out_fstride + c * ld_out
    long ld_out, out_fstride;
    int frames, N, Cq, d;
    int n_tiles;                    // ceil(N / 128)
    int n_splits, ksteps_per_split; // slices of d in the scores kernel, kLatentStageD-wide stages each
    float *scores;                  // [n_splits, frames, 64, ld_s] partial S (fp32), ld_s = n_tiles * 128
    long ld_s;
    __nv_bfloat16 *probs;           // [frames, Cq, ld_p] P (bf16), ld_p = N rounded up to 8
    long ld_p;
    unsigned int *fault;
};
cudaError_t launch_latent(const LatentParams &p, cudaStream_t st);
bool latent_supported();

cudaError_t launch_philox(const uint32_t *ctr, uint64_t key, uint32_t *out, int64_t n,
                          cudaStream_t st);

int device_sm_count();              // SMs of the current device (cached)

// records `msg` as this thread's sd_last_error() and returns `s`
sd_status report_error(sd_status s, const char *msg);

}  // namespace sdv
