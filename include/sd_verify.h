/*
 * sd_verify.h -- C ABI of libsdverify.so: the GPU hot path of block
 * verification in lossless draft-then-verify speculative decoding.
 *
 * The method ("VFlash-FM: Flow-Trained One-Pass Drafting for Video Language
 * Models", project page, section "How VFlash-FM works" and the worked cycle
 * in its figure): a drafter proposes a block of 16 slots -- the anchor (the
 * last committed token) and 15 proposals -- in one forward; the frozen target
 * scores all 16 slots in one forward over its KV cache; the proposals equal to
 * the target's greedy picks are kept up to the first mismatch, where the
 * target's own pick is committed instead.  The sampled variant applies the
 * usual speculative accept/reject test ("SpecFLASH" README, inference
 * section), so the output follows the target distribution exactly.
 *
 * Conventions shared by every call
 *  - All tensor pointers are DEVICE pointers owned by the caller; the library
 *    allocates nothing and keeps no per-call state.  `workspace` is caller
 *    memory of at least the size the matching *_workspace_size() returns.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls only
 *    enqueue work and return; SD_OK means "validated and launched".  Faults
 *    of launched kernels surface at the caller's next synchronisation.
 *  - Argument errors are detected on the host before anything is launched
 *    and return SD_ERR_INVALID_ARG / SD_ERR_UNSUPPORTED / SD_ERR_WORKSPACE;
 *    sd_last_error() then holds a one-line reason (thread-local).  No C++
 *    exception crosses this boundary.
 *  - Device-side guards (bounded waits, index checks) never trap: they set
 *    the library's fault word, read with sd_fault_word().
 *  - Tensors are row-major and contiguous unless strides are passed.
 *  - Calls that share a workspace must be ordered on one stream.
 */
#ifndef SD_VERIFY_H
#define SD_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SD_OK = 0,
    SD_ERR_INVALID_ARG = 1,   /* null pointer, bad size, inconsistent shape */
    SD_ERR_UNSUPPORTED = 2,   /* valid but not implemented (e.g. D = 96)     */
    SD_ERR_WORKSPACE = 3,     /* workspace missing or too small              */
    SD_ERR_CUDA = 4           /* a CUDA runtime call failed (see sd_last_error) */
} sd_status;

typedef enum {
    SD_BF16 = 0,              /* bfloat16 storage, fp32 arithmetic */
    SD_FP32 = 1               /* float32 storage, fp32 arithmetic  */
} sd_dtype;

/* element strides of a [B, S, H, D] tensor whose D axis is contiguous */
typedef struct {
    int64_t b, s, h;
} sd_strides;

/* ------------------------------------------------------------------------
 * Target block-verify attention (split-KV, log-sum-exp merge)
 *
 * Source: "VFlash-FM" project page, "How VFlash-FM works": the target
 * verifies all 16 block slots in one forward with grouped-query attention
 * over a KV cache allocated up front.  Slot j of the block may only see what
 * precedes it, so row j attends to cache keys [0, ctx_len[b] + j): ctx_len
 * counts the anchor, whose K/V sits at slot ctx_len-1; block row j's own K/V
 * is at slot ctx_len-1+j and must already be written by the caller.  T = 1
 * is ordinary one-token decode attention.
 *
 *   q        [B, T, Hq, D]  contiguous, rotary embedding already applied
 *   k_cache, v_cache  [B, S_max, Hkv, D] with element strides `kv`; the D
 *            axis contiguous; base addresses 16-byte aligned
 *   ctx_len  device int32 [B], each in [1, max_ctx]
 *   max_ctx  host upper bound of ctx_len; the cache must hold at least
 *            max_ctx + T - 1 slots per sequence (caller's contract: slots
 *            beyond a sequence's ctx_len + T - 1 are never read into the
 *            result, whatever they hold)
 *   out      device fp32 [B, T, Hq, D] contiguous
 *   query head h reads kv head h / (Hq / Hkv)
 *   logits are scale * q.k; softmax and accumulation in fp32
 *   T in [1, 16]; D in {64, 128}; Hq % Hkv == 0; Hq <= 4096
 *
 * workspace: zero-filled before the first call on it.  It holds one counter
 * per (sequence, kv head) for the splits that merge inside the kernel; every
 * call returns them to zero when its kernel ends, including a call whose
 * bounded wait gave up (fault bit 3; its output is then incomplete), so the
 * workspace never needs clearing again.
 * ------------------------------------------------------------------------ */
sd_status sd_verify_attention(const void *q, const void *k_cache, const void *v_cache,
                              sd_strides kv, const int32_t *ctx_len, int max_ctx,
                              float *out, int B, int T, int Hq, int Hkv, int D,
                              sd_dtype dtype, float scale,
                              void *workspace, size_t workspace_bytes, void *stream);

size_t sd_verify_attention_workspace_size(int B, int T, int Hq, int Hkv, int D,
                                          int max_ctx, sd_dtype dtype);

/* ------------------------------------------------------------------------
 * Drafter block attention
 *
 * Source: "VFlash-FM" project page, "How VFlash-FM works" and its figure:
 * the drafter never reads the video; its keys and values are a linear map of
 * the hidden states the target cached for every context position, and its
 * block (anchor + 15 mask slots) is filled in one forward, so every block
 * query sees every context key and every block key (no causal mask).
 *
 *   q            [B, T, Hq, D] contiguous
 *   k_ctx, v_ctx [B, S_ctx, Hkv, D] projected context keys / values, strides `ctx`
 *   n_ctx        device int32 [B], context keys per sequence, each in [1, max_ctx]
 *   k_blk, v_blk [B, T, Hkv, D] contiguous keys / values of the block slots
 *   out          fp32 [B, T, Hq, D]
 *   every row attends to context keys [0, n_ctx[b]) followed by the T block keys
 *   limits as for sd_verify_attention
 *   workspace as for sd_verify_attention (zero-filled before its first call)
 * ------------------------------------------------------------------------ */
sd_status sd_draft_block_attention(const void *q, const void *k_ctx, const void *v_ctx,
                                   sd_strides ctx, const int32_t *n_ctx, int max_ctx,
                                   const void *k_blk, const void *v_blk, float *out,
                                   int B, int T, int Hq, int Hkv, int D, sd_dtype dtype,
                                   float scale, void *workspace, size_t workspace_bytes,
                                   void *stream);

size_t sd_draft_block_attention_workspace_size(int B, int T, int Hq, int Hkv, int D,
                                               int max_ctx, sd_dtype dtype);

/* ------------------------------------------------------------------------
 * Tree verify attention
 *
 * Source: "VFlash-FM" project page, speedup table: its fastest variant
 * verifies a draft tree ("Tree-60") rather than a chain.  The page gives no
 * layout; the one taken here: the block's T slots are the tree's nodes in
 * topological order, node 0 the anchor, their K/V at cache slots
 * ctx_len-1 .. ctx_len-2+T exactly as for sd_verify_attention.  Node j
 * attends to the cache keys [0, ctx_len-1) (the context before the anchor)
 * and to the slots ctx_len-1+k of every bit k set in tree_mask[b][j] (its
 * ancestors and itself).  A chain mask (bits 0..j) gives sd_verify_attention.
 *
 *   tree_mask  device uint64 [B, T], 8-byte aligned; bit k (k < T) of node j's
 *              word set when node j sees block slot k
 *   T          nodes, in [1, 64] (the page's "Tree-60" is about 60 nodes);
 *              the tensor-core kernel cuts a kv head's (Hq/Hkv)*T query rows
 *              into blocks of whole nodes of at most 128 rows, which read
 *              the same K/V tiles
 *   everything else as for sd_verify_attention; the workspace size comes
 *   from sd_verify_tree_attention_workspace_size
 * ------------------------------------------------------------------------ */
sd_status sd_verify_tree_attention(const void *q, const void *k_cache, const void *v_cache,
                                   sd_strides kv, const int32_t *ctx_len, int max_ctx,
                                   const uint64_t *tree_mask, float *out, int B, int T, int Hq,
                                   int Hkv, int D, sd_dtype dtype, float scale,
                                   void *workspace, size_t workspace_bytes, void *stream);

size_t sd_verify_tree_attention_workspace_size(int B, int T, int Hq, int Hkv, int D,
                                               int max_ctx, sd_dtype dtype);

/* ------------------------------------------------------------------------
 * Greedy acceptance
 *
 * Source: "VFlash-FM" project page, worked cycle: the target keeps the
 * proposals that equal its own greedy picks up to the first mismatch and
 * commits its own pick there (7 accepted + 1 correction = 8 tokens).
 *
 *   draft_ids     device int32 [B, T-1]; draft_ids[b][j] is the proposal for
 *                 the slot after block row j, checked against logits row j
 *   target_logits device [B, T, V] (bf16 or fp32), contiguous
 *   n_accepted    device int32 [B]: first j in [0, T-2] whose proposal is not
 *                 the row's argmax, else T-1
 *   correction_id device int32 [B]: argmax of row n_accepted (the target's
 *                 token at the first mismatch, or the bonus token)
 *   argmax ties go to the lowest index; values compare exactly in fp32
 *   workspace: zero-filled before the first call on it; each completed call
 *   leaves its counters zero again, so it stays reusable.
 * ------------------------------------------------------------------------ */
sd_status sd_accept_greedy(const int32_t *draft_ids, const void *target_logits,
                           int B, int T, int V, sd_dtype dtype,
                           int32_t *n_accepted, int32_t *correction_id,
                           void *workspace, size_t workspace_bytes, void *stream);

size_t sd_accept_greedy_workspace_size(int B, int T, int V, sd_dtype dtype);

/* ------------------------------------------------------------------------
 * Sampled (lossless) acceptance
 *
 * Source: "SpecFLASH" README, inference section: the drafted tokens are
 * checked under the standard speculative accept/reject rule, which leaves
 * the output distributed exactly as the target's.
 *
 *   p_j = softmax(target_logits[b, j] / temperature), fp32
 *   for j = 0 .. T-2:  u = U(seed; j, b, 0, offset);
 *                      accept draft_ids[b][j] = d iff u * q_j(d) < p_j(d)
 *   first reject at n: u' = U(seed; n, b, 1, offset); next_id = the smallest i
 *                      whose ascending inclusive cumulative sum of
 *                      r = max(p_n - q_n, 0) exceeds u' * sum(r)
 *                      (if sum(r) == 0: the same draw from p_n)
 *   all accepted:      next_id drawn the same way from p_{T-1} with u' from row T-1
 *   U(seed; c0, c1, c2, c3) = (word0 of Philox4x32-10 with key (seed lo32,
 *   seed hi32) and counter (c0, c1, c2, c3)) >> 8, times 2^-24.
 *
 *   draft_probs  device fp32 [B, T, V], rows 0..T-2 read (the drafter's
 *                normalised distributions)
 *   temperature  > 0 (temperature 0 is sd_accept_greedy)
 *   n_accepted, next_id  device int32 [B]
 *   workspace: zero-filled before the first call on it; each completed call
 *   leaves its counters zero again (a call whose bounded wait gave up
 *   included: the fault word says so).
 * ------------------------------------------------------------------------ */
sd_status sd_accept_sample(const int32_t *draft_ids, const float *draft_probs,
                           const void *target_logits, int B, int T, int V, sd_dtype dtype,
                           float temperature, uint64_t philox_seed, uint32_t philox_offset,
                           int32_t *n_accepted, int32_t *next_id,
                           void *workspace, size_t workspace_bytes, void *stream);

size_t sd_accept_sample_workspace_size(int B, int T, int V, sd_dtype dtype);

/* ------------------------------------------------------------------------
 * Greedy acceptance over a draft tree
 *
 * Source: "VFlash-FM" project page (speedup table, tree verification; the
 * greedy rule of the worked cycle).  With a_j the argmax of logits row j
 * (ties: lowest index), the anchor is accepted and node j >= 1 is accepted
 * when its parent is and tokens[b][j] == a_parent: the target's own greedy
 * pick after the parent.  The committed path ends at the accepted node of
 * greatest depth (the lowest index among equals), so a chain tree gives
 * sd_accept_greedy.
 *
 *   T              nodes, in [1, 64]
 *   tokens         device int32 [B, T]: tokens[b][j] is node j's proposal
 *                  (tokens[b][0], the anchor, is not read)
 *   parents        device int32 [B, T]: parents[b][0] = -1, parents[b][j] in
 *                  [0, j); anything else sets the fault word
 *   target_logits  [B, T, V] as for sd_accept_greedy
 *   n_accepted     device int32 [B]: depth of that node (proposals kept)
 *   correction_id  device int32 [B]: a_node (the target's next token)
 *   path           device int32 [B, T]: the kept nodes at depth 1..n, then -1
 *   workspace      at least sd_accept_tree_greedy_workspace_size bytes,
 *                  zero-filled before its first call (as for sd_accept_greedy)
 * ------------------------------------------------------------------------ */
sd_status sd_accept_tree_greedy(const int32_t *tokens, const int32_t *parents, const void *target_logits,
                                int B, int T, int V, sd_dtype dtype, int32_t *n_accepted,
                                int32_t *correction_id, int32_t *path, void *workspace,
                                size_t workspace_bytes, void *stream);

size_t sd_accept_tree_greedy_workspace_size(int B, int T, int V, sd_dtype dtype);

/* ------------------------------------------------------------------------
 * Drafter K/V projector
 *
 * Source: "VFlash-FM" project page, "How VFlash-FM works": the drafter reads
 * no pixels; the keys and values its block attends to are a learned linear
 * map of the hidden states the target already keeps for every context
 * position.  For rows n in [0, N):
 *   k_out[n][c] = sum_f hidden[n][f] * w_k[c][f]
 *   v_out[n][c] = sum_f hidden[n][f] * w_v[c][f]      (c < Dout, f < Hd)
 * fp32 accumulation, rounded once to bf16 (round to nearest even).  Run once
 * over the whole context (prefill) and then over the rows each cycle commits
 * (the incremental append), so the drafter's cache grows with the target's.
 *
 *   hidden      device bf16 [N, Hd], row stride ld_hidden elements
 *   w_k, w_v    device bf16 [Dout, Hd] contiguous (a linear layer's weight)
 *   k_out/v_out device bf16 [N, Dout], row stride ld_out elements: with a
 *               [B, S, Hkv, D] cache, Dout = Hkv * D and k_out points at the
 *               first row to write; rows outside [0, N) are not touched
 *   dtype       SD_BF16 (SD_FP32 returns SD_ERR_UNSUPPORTED)
 * Requires Hd % 8 == 0, Dout % 32 == 0, ld_hidden >= Hd and ld_out >= Dout,
 * both multiples of 8, every pointer 16-byte aligned, 0 <= N <= 2^21 (N = 0
 * launches nothing).  Up to 16 rows run on CUDA cores (the weights are read
 * once, the rows staged in shared memory: 16 * Hd * 2 bytes <= 200 KB, else
 * 8 rows per CTA); more rows run as a tensor-core GEMM.  No workspace.
 * ------------------------------------------------------------------------ */
sd_status sd_project_kv(const void *hidden, int64_t ld_hidden, const void *w_k, const void *w_v,
                        int N, int Hd, int Dout, void *k_out, void *v_out, int64_t ld_out,
                        sd_dtype dtype, void *stream);

/* ------------------------------------------------------------------------
 * Commit of a verified block, on the device
 *
 * Source: "VFlash-FM" project page, "How VFlash-FM works" and its worked
 * cycle: the accepted prefix and the target's own token at the first
 * disagreement are committed, the rest of the block is discarded, and the
 * next cycle starts from that token as its anchor.  These three calls read
 * the acceptance results from device memory, so a whole cycle -- draft,
 * verify, accept, append, commit -- can be enqueued (or captured in one CUDA
 * graph) and repeated with no host round trip.  Per cycle, in stream order:
 * sd_compact_tree_kv (trees only), sd_project_kv_commit, then
 * sd_commit_tokens (the first two read ctx_len / draft_ctx before the third
 * advances them).  Guards never trap: a sequence whose n_accepted, path or
 * lengths are out of range is skipped and bit 6 of the fault word is set.
 *
 * Conventions (those of the attention calls): ctx_len counts the anchor;
 * block slot k of sequence b is cache position ctx_len[b] - 1 + k; the
 * drafter's context is every position before the anchor (ctx_len - 1 rows).
 * T is the block's slot count: at most 16 for a chain, at most 64 for a tree.
 * ------------------------------------------------------------------------ */

/* Tokens and lengths.  With n = n_accepted[b]:
 *   kept proposal i < n: chain (path NULL) proposals[b * proposal_stride + i];
 *     tree proposals[b * proposal_stride + path[b * T + i]] (path as written
 *     by sd_accept_tree_greedy: the kept nodes by depth)
 *   out_tokens[b * out_cap + out_len[b] + i] = kept proposal i, then
 *   out_tokens[b * out_cap + out_len[b] + n] = next_token[b];
 *   out_len[b] += n + 1; ctx_len[b] += n + 1; draft_ctx[b] = ctx_len[b] - 1
 *   (if draft_ctx is not NULL); anchor[b] = next_token[b]; status[b] = 0.
 * A commit with n outside [0, T-1], a kept node outside [1, T), ctx_len + n + 1
 * > ctx_cap or out_len + n + 1 > out_cap leaves sequence b unchanged and sets
 * status[b] = 1 (if status is not NULL) and the fault word.
 *   proposals    device int32: chain [B, >= T-1] drafts, tree [B, >= T] node tokens
 *   n_accepted, next_token  device int32 [B] (sd_accept_* outputs; next_token
 *                is the correction or the sampled next id)
 *   ctx_len, draft_ctx, out_len, anchor, status  device int32 [B], updated in place
 *   out_tokens   device int32 [B, out_cap]
 *   ctx_cap      the largest ctx_len the caches can take (for a cache of S
 *                positions verified in T-slot blocks: S - T + 1) */
sd_status sd_commit_tokens(const int32_t *proposals, int proposal_stride, const int32_t *path,
                           const int32_t *n_accepted, const int32_t *next_token, int B, int T,
                           int32_t *ctx_len, int ctx_cap, int32_t *draft_ctx, int32_t *out_tokens,
                           int32_t *out_len, int out_cap, int32_t *anchor, int32_t *status, void *stream);

/* Tree rollback in the target's K/V cache: for depth d = 1..n_accepted[b],
 * position ctx_len[b]-1+d takes the row at position ctx_len[b]-1+path[b*T+d-1]
 * (every kv head, K and V, moved bit for bit); all other positions keep their
 * rows.  After it the cache holds the committed sequence in order and the
 * next block overwrites what follows.  ctx_len is read, not changed.
 *   k_cache, v_cache  [B, max_slots, Hkv, D] with element strides kv, D
 *                contiguous; D * element size a multiple of 16 bytes, <= 512
 *   path         device int32 [B, T] (sd_accept_tree_greedy's)
 * A sequence whose block passes max_slots is skipped (fault word). */
sd_status sd_compact_tree_kv(void *k_cache, void *v_cache, sd_strides kv, const int32_t *ctx_len,
                             const int32_t *path, const int32_t *n_accepted, int B, int T,
                             int max_slots, int Hkv, int D, sd_dtype dtype, void *stream);

/* The results a serving loop reads on the host each cycle (accepted counts and
 * next ids, the verified rows), stored into pinned host memory by the GPU's
 * own cores, after the stream's earlier work: for a few hundred KB this ends
 * sooner than a copy-engine transfer, whose set-up dominates at that size.
 * Once the stream's work up to this call has completed (an event or stream
 * synchronisation), host_dst[0, bytes) holds src[0, bytes).
 *   host_dst  pinned host memory (cudaHostAlloc, or cudaHostRegister'd), read
 *             by the host only after that synchronisation
 *   src       device memory
 *   bytes     a multiple of 16; both addresses 16-byte aligned; the caller
 *             keeps both ranges inside their allocations
 * Returns SD_ERR_INVALID_ARG (nothing enqueued) when host_dst is not pinned
 * host memory, src is not device memory, or the sizes are misaligned. */
sd_status sd_store_to_host(void *host_dst, const void *src, int64_t bytes, void *stream);

/* The drafter's context append for the committed rows (the incremental
 * append of sd_project_kv with the row count on the device): for r = 0..n
 * (n = n_accepted[b]), hidden row src = 0 (the anchor) or r (chain) or
 * path[b*T + r-1] (tree) of sequence b's block is projected (as in
 * sd_project_kv) into drafter context row draft_ctx[b] + r.
 *   hidden_block device bf16: row src of sequence b at
 *                hidden_block + b * hidden_bstride + src * ld_hidden
 *   k_ctx, v_ctx device bf16: row i of sequence b at + b * ctx_bstride +
 *                i * ld_out; rows past max_rows are never written (a commit
 *                that would pass it is skipped and sets the fault word)
 *   draft_ctx    device int32 [B]: the drafter's context length before the
 *                commit (sd_commit_tokens advances it afterwards)
 * Requirements as for sd_project_kv, and Hd <= 6400 (the rows go in groups of
 * 16 per CTA, staged in 200 KB of shared memory; else SD_ERR_UNSUPPORTED). */
sd_status sd_project_kv_commit(const void *hidden_block, int64_t ld_hidden, int64_t hidden_bstride,
                               const void *w_k, const void *w_v, int Hd, int Dout,
                               const int32_t *n_accepted, const int32_t *path, const int32_t *draft_ctx,
                               int B, int T, void *k_ctx, void *v_ctx, int64_t ctx_bstride, int64_t ld_out,
                               int max_rows, sd_dtype dtype, void *stream);

/* ------------------------------------------------------------------------
 * SpecFLASH latent visual compressor
 *
 * Source: "SpecFLASH" README, the first of the draft model's two components:
 * a learned set of Cq query vectors attends over the N visual features of
 * the target's second-to-top layer and compresses them into Cq latent
 * features (LLaVA-1.5: 576 -> 64; Qwen2.5-VL: 324 -> 36), per frame i:
 *   out[i] = softmax(Q . F[i]^T) . F[i]     (softmax over the N features;
 *                                             no scale on the scores)
 * Scores accumulate in fp32 on the tensor cores; the softmax weights are
 * rounded to bf16 for the second product, which accumulates in fp32 and is
 * rounded once to bf16.
 *
 *   queries    device bf16 [Cq, d] contiguous, 1 <= Cq <= 64
 *   features   device bf16: frame i, feature n at
 *              features + i * frame_stride + n * ld_features (d contiguous)
 *   out        device bf16: frame i, query c at out + i * out_frame_stride +
 *              c * ld_out (d contiguous)
 *   workspace  at least sd_latent_compress_workspace_size() bytes, 16-byte
 *              aligned, no initial contents needed (fp32 partial scores,
 *              one copy per slice of d, and the bf16 weights)
 * Requires d a multiple of 64 (<= 65536), 1 <= frames <= 65535, strides
 * multiples of 8 elements that cover a row / frame, 16-byte aligned
 * pointers, sm_103 (else SD_ERR_UNSUPPORTED).  Three kernel launches.
 * Deterministic: the scores kernel may slice d (how many slices depends on
 * the shape and the GPU's SM count) and the slices are summed in a fixed
 * order.
 * ------------------------------------------------------------------------ */
sd_status sd_latent_compress(const void *queries, const void *features, int64_t ld_features,
                             int64_t frame_stride, int frames, int N, int Cq, int d, void *out,
                             int64_t ld_out, int64_t out_frame_stride, sd_dtype dtype,
                             void *workspace, size_t workspace_bytes, void *stream);

size_t sd_latent_compress_workspace_size(int frames, int N, int Cq, int d);

/* ------------------------------------------------------------------------
 * Greedy acceptance without a caller workspace
 *
 * No counterpart in the method's pages: this is a convenience of the library.
 * For hosts that cannot hand the library device memory -- their own pool
 * allocator owns all of it and extensions may not call cudaMalloc, or only the
 * input and output buffers are at hand when the call is made.  Computes
 * exactly what sd_accept_greedy computes, with the same arguments minus the
 * workspace.  Scratch is a 1 MiB device array owned by the library (held on
 * every GPU that loads it until the process exits); shapes whose workspace
 * (sd_accept_greedy_workspace_size) exceeds 1 MiB return SD_ERR_WORKSPACE.
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) and keeps it for the process; make that first call
 * before any stream capture.  A cudaDeviceReset ends the context that address
 * belongs to: do not call this entry point on that device after one.
 * Every call clears and then uses the same array, so calls must not overlap
 * on the GPU: issue them on one stream (calls on different streams or from
 * different threads without ordering race).  Nothing on this path allocates.
 * ------------------------------------------------------------------------ */
sd_status sd_accept_greedy_noalloc(const int32_t *draft_ids, const void *target_logits,
                                   int B, int T, int V, sd_dtype dtype,
                                   int32_t *n_accepted, int32_t *correction_id, void *stream);

/* ------------------------------------------------------------------------
 * Philox4x32-10 (Salmon et al., "Parallel Random Numbers: As Easy as 1, 2,
 * 3", SC'11), the generator behind sd_accept_sample, exposed so callers can
 * check it: counters device uint32 [n, 4], out device uint32 [n, 4],
 * key = (key lo32, key hi32).
 * ------------------------------------------------------------------------ */
sd_status sd_philox4x32_10(const uint32_t *counters, uint64_t key, uint32_t *out,
                           int64_t n, void *stream);

/* ------------------------------------------------------------------------
 * Utilities
 * ------------------------------------------------------------------------ */
const char *sd_status_string(sd_status s);
const char *sd_last_error(void);        /* reason for the last non-OK status on this thread */
int sd_version(void);                   /* 100 * major + minor */

/* Device fault word: 0 while no kernel guard fired.  Reading synchronises the
 * current device; `clear` resets it to 0.  Bits: 0 ctx_len outside
 * [1, max_ctx]; 1 a draft id outside [0, V); 2 a logits row with no ordered
 * value (NaN); 3 a bounded wait gave up; 4 tensor-memory allocation failed;
 * 5 a tree parent outside [0, node); 6 a commit out of range (skipped). */
sd_status sd_fault_word(uint32_t *out, int clear);

/* Attention kernel selection, process-wide, for tests and measurement:
 * 0 = automatic (tensor-core kernel where it applies), 1 = force the
 * CUDA-core kernel, 2 = require the tensor-core kernel (calls it cannot
 * serve return SD_ERR_UNSUPPORTED).  Other values select 0.  Returns the
 * previous setting. */
int sd_set_attention_path(int path);

/* Which kernel the last attention call on this thread launched (1 or 2 as
 * above) and its split count: for the CUDA-core kernel the key splits of every
 * (sequence, kv head); for the tensor-core kernel the CTAs of its grid, which
 * the kernel spreads over the (sequence, kv head, row block) units by their
 * lengths (a unit left with one CTA writes its output itself). */
int sd_last_attention_path(int *n_splits);

/* How many kernels the last attention call on this thread launched: 1 when the
 * splits were merged inside the split kernel (or there was one split), 2 when
 * a separate merge kernel followed.  No counterpart on the pages: a count for
 * measurement. */
int sd_last_attention_launches(void);

/* Sampled-rule kernel selection, process-wide, for tests and measurement:
 * 0 = automatic (the one-launch form where its grid fits on the device at
 * once: 2 CTAs per SM, B*T and B at most that many, chunks of the deciding
 * row within 4 vectors per thread, logits 16-byte aligned; else two kernels),
 * 1 = force the two-kernel
 * form, 2 = require the one-launch form (calls it cannot serve return
 * SD_ERR_UNSUPPORTED).  Other values select 0.  Returns the previous setting.
 * Both forms compute the same rule; their float-float sums group terms
 * differently, so a draw may differ where it sits within rounding of a
 * boundary. */
int sd_set_sample_path(int path);

/* Which form the last sd_accept_sample on this thread launched: 1 two
 * kernels, 2 one cooperative launch, 0 none. */
int sd_last_sample_path(void);

/* Failure-detection test hook, process-wide.  The in-kernel barriers (the
 * tensor-core attention's merge of a unit's splits, the one-launch sampled
 * rule's grid and sequence barriers) wait for `extra_arrivals` more CTAs than
 * the grid has, giving up after `limit_ns` (0, or more than 2 s: 2 s, the
 * normal limit).  A call made meanwhile sets fault bit 3 (a bounded wait gave
 * up), returns with undefined outputs and leaves its counters zero, so the
 * next call on the same workspace is exact.  (0, 0) restores normal
 * operation.  SD_ERR_INVALID_ARG if extra_arrivals > 1024. */
sd_status sd_set_wait_test(uint32_t extra_arrivals, uint64_t limit_ns);

/* Projector kernel selection, process-wide, for tests and measurement:
 * 0 = automatic (above), 1 = CUDA cores for every N, 2 = tensor cores for
 * every N >= 1 (calls it cannot serve return SD_ERR_UNSUPPORTED).  Other
 * values select 0.  Returns the previous setting. */
int sd_set_projector_path(int path);

/* Which projector kernel the last sd_project_kv on this thread launched:
 * 1 or 2 as above, 0 if none. */
int sd_last_projector_path(void);

#ifdef __cplusplus
}
#endif

#endif /* SD_VERIFY_H */
