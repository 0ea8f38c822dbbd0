/*
 * Plain fp64 CPU oracle for block verification in lossless speculative
 * decoding.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the
 * benchmark's CPU-baseline leg call it; the GPU library never does, and the
 * two share no code.
 *
 * Every routine is the plainest statement of what the method computes, with
 * no blocking, fusion or reordering beyond its definition.  Sources:
 *
 *  - "VFlash-FM: Flow-Trained One-Pass Drafting for Video Language Models"
 *    (project page), section "How VFlash-FM works" and the worked cycle in its
 *    figure: a block has 16 slots (an anchor and 15 proposals) and the frozen
 *    target scores all of them in one forward, using grouped-query attention
 *    over a KV cache allocated up front.  The target keeps the longest run of
 *    proposals equal to its own greedy picks, adds its own pick at the first
 *    mismatch and drops everything after it.  The drafter gets its keys and
 *    values by a linear map of hidden states the target has already cached.
 *  - "SpecFLASH" README, section on inference: the target checks all drafted
 *    tokens at once under the usual speculative accept/reject test, which
 *    keeps the output distribution equal to the target's (lossless); and the
 *    first of its draft model's two components, the latent visual compressor
 *    softmax(C . F_V^T) . F_V over a frame's visual features.
 *  - Philox4x32-10: Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As
 *    Easy as 1, 2, 3", SC'11, section 3.2 (the Philox round and key schedule).
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *  - ctx counts the anchor; block row j attends to keys [0, ctx + j).
 *  - kv head of query head h is h / (Hq / Hkv).
 *  - draft[j] (j = 0..T-2) is checked against logits row j; row T-1 only
 *    supplies the bonus / correction token.
 *  - ties in argmax go to the lowest index.
 *  - sampled accept: accept iff u * q(d) < p(d); residual draw = smallest i
 *    whose inclusive ascending cumulative sum of max(p - q, 0) exceeds u' * S.
 *  - Philox counter = (row j, batch b, stream, offset), key = (seed lo, seed
 *    hi); the uniform is (word0 >> 8) * 2^-24.
 *  - a tree has at most 64 nodes; node j sees the context before the anchor
 *    and the block slots of its ancestors and itself; the committed path ends
 *    at the deepest accepted node (lowest index among equals).
 *  - commit: committed tokens = kept proposals + the next token, ctx_len
 *    advances by their count, the next token becomes the anchor; a tree's
 *    kept K/V rows move to consecutive positions after the anchor.
 *  - the compressor applies no scale to its scores (the formula has none).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Philox4x32-10 (Salmon et al. SC'11, section 3.2)                          */
/* ------------------------------------------------------------------------ */

#define PHILOX_M0 0xD2511F53u
#define PHILOX_M1 0xCD9E8D57u
#define PHILOX_W0 0x9E3779B9u
#define PHILOX_W1 0xBB67AE85u

static void mulhilo32(uint32_t a, uint32_t b, uint32_t *hi, uint32_t *lo) {
    uint64_t p = (uint64_t)a * (uint64_t)b;
    *hi = (uint32_t)(p >> 32);
    *lo = (uint32_t)p;
}

/* ten rounds; round r uses the key bumped r times by the Weyl constants */
void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
    uint32_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int r = 0; r < 10; ++r) {
        uint32_t hi0, lo0, hi1, lo1;
        mulhilo32(PHILOX_M0, x0, &hi0, &lo0);
        mulhilo32(PHILOX_M1, x2, &hi1, &lo1);
        uint32_t y0 = hi1 ^ x1 ^ k0;
        uint32_t y1 = lo1;
        uint32_t y2 = hi0 ^ x3 ^ k1;
        uint32_t y3 = lo0;
        x0 = y0; x1 = y1; x2 = y2; x3 = y3;
        k0 += PHILOX_W0;
        k1 += PHILOX_W1;
    }
    out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;
}

void oracle_philox4x32_10_batch(const uint32_t *ctr, const uint32_t key[2], uint32_t *out, long n) {
    for (long i = 0; i < n; ++i) oracle_philox4x32_10(ctr + 4 * i, key, out + 4 * i);
}

/* uniform in [0,1) from word 0: top 24 bits times 2^-24 (exact in fp32 and fp64) */
double oracle_uniform(uint64_t seed, uint32_t row, uint32_t batch, uint32_t stream, uint32_t offset) {
    uint32_t ctr[4] = {row, batch, stream, offset};
    uint32_t key[2] = {(uint32_t)(seed & 0xffffffffu), (uint32_t)(seed >> 32)};
    uint32_t out[4];
    oracle_philox4x32_10(ctr, key, out);
    return (double)(out[0] >> 8) * (1.0 / 16777216.0);
}

/* ------------------------------------------------------------------------ */
/* Attention                                                                 */
/* ------------------------------------------------------------------------ */

/*
 * Exact softmax attention of selected query rows, in fp64.
 *
 * q   [B, T, Hq, D]      queries (already rotary-embedded by the caller)
 * kc  [B, Sc, Hkv, D]    context / cache keys; vc the same for values
 * kb  [B, T, Hkv, D]     block keys (mode 1 only; NULL otherwise); vb values
 * nctx[B]                mode 0 (target verify): ctx_len, row j sees cache
 *                        keys [0, ctx + j) -- causal within the block;
 *                        mode 1 (drafter): number of context keys; every row
 *                        sees cache keys [0, n) followed by the T block keys.
 * lo, hi                 restrict to key indices in [lo, hi) of the row's key
 *                        sequence (hi < 0: no restriction) -- used to check the
 *                        split / log-sum-exp merge identity.
 * rows[n_rows]           flat row ids (b*T + j)*Hq + h; NULL = all rows in order
 * out [n_rows, D]        softmax(scale * q.k) weighted sum of v
 * lse [n_rows]           log of the softmax normaliser (natural log, including
 *                        the max), -inf where the row has no key; may be NULL
 * returns 0, or -1 on bad arguments / allocation failure
 */
int oracle_attention_rows(const double *q, const double *kc, const double *vc,
                          const double *kb, const double *vb, const int *nctx, int mode,
                          int B, int T, int Hq, int Hkv, int D, int Sc, double scale,
                          long lo, long hi, const long *rows, long n_rows,
                          double *out, double *lse) {
    if (B < 1 || T < 1 || Hq < 1 || Hkv < 1 || D < 1 || Hq % Hkv != 0) return -1;
    if (mode == 1 && (kb == NULL || vb == NULL)) return -1;
    const int G = Hq / Hkv;
    long total_rows = (long)B * T * Hq;
    if (rows == NULL) n_rows = total_rows;
    long max_keys = (long)Sc + T;
    double *s = (double *)malloc(sizeof(double) * (size_t)max_keys);
    const double **kp = (const double **)malloc(sizeof(double *) * (size_t)max_keys);
    const double **vp = (const double **)malloc(sizeof(double *) * (size_t)max_keys);
    if (!s || !kp || !vp) { free(s); free(kp); free(vp); return -1; }

    for (long r = 0; r < n_rows; ++r) {
        long flat = rows ? rows[r] : r;
        if (flat < 0 || flat >= total_rows) { free(s); free(kp); free(vp); return -1; }
        int h = (int)(flat % Hq);
        int j = (int)((flat / Hq) % T);
        int b = (int)(flat / ((long)Hq * T));
        int g = h / G;
        const double *qr = q + flat * D;

        /* the row's key sequence */
        long n = 0;
        if (mode == 0) {
            long L = (long)nctx[b] + j;
            if (L > Sc) { free(s); free(kp); free(vp); return -1; }
            for (long i = 0; i < L; ++i) {
                kp[n] = kc + (((long)b * Sc + i) * Hkv + g) * D;
                vp[n] = vc + (((long)b * Sc + i) * Hkv + g) * D;
                ++n;
            }
        } else {
            long L = nctx[b];
            if (L > Sc) { free(s); free(kp); free(vp); return -1; }
            for (long i = 0; i < L; ++i) {
                kp[n] = kc + (((long)b * Sc + i) * Hkv + g) * D;
                vp[n] = vc + (((long)b * Sc + i) * Hkv + g) * D;
                ++n;
            }
            for (long i = 0; i < T; ++i) {
                kp[n] = kb + (((long)b * T + i) * Hkv + g) * D;
                vp[n] = vb + (((long)b * T + i) * Hkv + g) * D;
                ++n;
            }
        }
        long k0 = lo < 0 ? 0 : lo;
        long k1 = (hi < 0 || hi > n) ? n : hi;

        double *o = out + r * D;
        for (int d = 0; d < D; ++d) o[d] = 0.0;
        if (k1 <= k0) {
            if (lse) lse[r] = -INFINITY;
            continue;
        }
        double m = -INFINITY;
        for (long i = k0; i < k1; ++i) {
            double acc = 0.0;
            for (int d = 0; d < D; ++d) acc += qr[d] * kp[i][d];
            s[i] = scale * acc;
            if (s[i] > m) m = s[i];
        }
        double denom = 0.0;
        for (long i = k0; i < k1; ++i) {
            double w = exp(s[i] - m);
            denom += w;
            for (int d = 0; d < D; ++d) o[d] += w * vp[i][d];
        }
        for (int d = 0; d < D; ++d) o[d] /= denom;
        if (lse) lse[r] = m + log(denom);
    }
    free(s); free(kp); free(vp);
    return 0;
}

/*
 * Tree verification (the "Tree-60" variant in the VFlash-FM speedup table):
 * the block's T slots are the nodes of a draft tree in topological order,
 * node 0 the anchor; their K/V sit at cache slots ctx-1 .. ctx-2+T as in the
 * chain case.  Node j attends to the context before the anchor, cache keys
 * [0, ctx-1), and to the block slots k whose bit is set in mask[b*T + j]
 * (its ancestors and itself), in increasing k; T <= 64, so a 64-bit word per
 * node holds its mask.  A chain mask (bits 0..j)
 * gives exactly the keys [0, ctx+j) of oracle_attention_rows, in the same
 * order.  Arguments as there; mask is [B*T].
 */
int oracle_tree_attention_rows(const double *q, const double *kc, const double *vc, const int *nctx,
                               const uint64_t *mask, int B, int T, int Hq, int Hkv, int D, int Sc,
                               double scale, const long *rows, long n_rows, double *out) {
    if (B < 1 || T < 1 || T > 64 || Hq < 1 || Hkv < 1 || D < 1 || Hq % Hkv != 0) return -1;
    const int G = Hq / Hkv;
    long total_rows = (long)B * T * Hq;
    if (rows == NULL) n_rows = total_rows;
    long max_keys = (long)Sc;
    double *s = (double *)malloc(sizeof(double) * (size_t)max_keys);
    long *ki = (long *)malloc(sizeof(long) * (size_t)max_keys);
    if (!s || !ki) { free(s); free(ki); return -1; }
    for (long r = 0; r < n_rows; ++r) {
        long flat = rows ? rows[r] : r;
        if (flat < 0 || flat >= total_rows) { free(s); free(ki); return -1; }
        int h = (int)(flat % Hq);
        int j = (int)((flat / Hq) % T);
        int b = (int)(flat / ((long)Hq * T));
        int g = h / G;
        const double *qr = q + flat * D;
        long c = nctx[b];
        if (c < 1 || c - 1 + T > Sc) { free(s); free(ki); return -1; }
        long n = 0;
        for (long i = 0; i < c - 1; ++i) ki[n++] = i;
        for (int k = 0; k < T; ++k)
            if ((mask[(long)b * T + j] >> k) & 1u) ki[n++] = c - 1 + k;   /* 64-bit mask, k < 64 */
        double *o = out + r * D;
        for (int d = 0; d < D; ++d) o[d] = 0.0;
        if (n == 0) continue;
        double m = -INFINITY;
        for (long i = 0; i < n; ++i) {
            const double *kr = kc + (((long)b * Sc + ki[i]) * Hkv + g) * D;
            double acc = 0.0;
            for (int d = 0; d < D; ++d) acc += qr[d] * kr[d];
            s[i] = scale * acc;
            if (s[i] > m) m = s[i];
        }
        double denom = 0.0;
        for (long i = 0; i < n; ++i) {
            const double *vr = vc + (((long)b * Sc + ki[i]) * Hkv + g) * D;
            double w = exp(s[i] - m);
            denom += w;
            for (int d = 0; d < D; ++d) o[d] += w * vr[d];
        }
        for (int d = 0; d < D; ++d) o[d] /= denom;
    }
    free(s); free(ki);
    return 0;
}

/*
 * Drafter K/V projector ("VFlash-FM" project page, "How VFlash-FM works":
 * the drafter's keys and values are a linear map of the hidden states the
 * target has cached).  For the selected rows r: out[i][c] = sum_k h[r][k] *
 * w[c][k], exact in fp64 (w is [Dout, Hd], the out-features x in-features
 * layout of a linear layer's weight).
 */
int oracle_project_rows(const double *h, const double *w, int N, int Hd, int Dout, const long *rows, long n_rows,
                        double *out) {
    if (N < 1 || Hd < 1 || Dout < 1) return -1;
    if (rows == NULL) n_rows = N;
    for (long i = 0; i < n_rows; ++i) {
        const long r = rows ? rows[i] : i;
        if (r < 0 || r >= N) return -1;
        for (int c = 0; c < Dout; ++c) {
            double acc = 0.0;
            for (int k = 0; k < Hd; ++k) acc += h[r * Hd + k] * w[(long)c * Hd + k];
            out[i * Dout + c] = acc;
        }
    }
    return 0;
}

/*
 * Log-sum-exp merge of attention over disjoint key ranges:
 * out = sum_s exp(lse_s - M) o_s / sum_s exp(lse_s - M), M = max_s lse_s;
 * ranges with lse = -inf hold no key and are skipped.
 * o [S, D], lse [S] -> out [D]; returns the merged lse.
 */
double oracle_lse_merge(const double *o, const double *lse, int S, int D, double *out) {
    double M = -INFINITY;
    for (int s = 0; s < S; ++s) if (lse[s] > M) M = lse[s];
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    if (M == -INFINITY) return -INFINITY;
    double wsum = 0.0;
    for (int s = 0; s < S; ++s) {
        if (lse[s] == -INFINITY) continue;
        double w = exp(lse[s] - M);
        wsum += w;
        for (int d = 0; d < D; ++d) out[d] += w * o[(long)s * D + d];
    }
    for (int d = 0; d < D; ++d) out[d] /= wsum;
    return M + log(wsum);
}

/* ------------------------------------------------------------------------ */
/* Greedy acceptance                                                         */
/* ------------------------------------------------------------------------ */

/* first index of the largest value (strictly-greater scan keeps the lowest) */
static int argmax_lowest(const double *x, int V) {
    int best = 0;
    for (int i = 1; i < V; ++i)
        if (x[i] > x[best]) best = i;
    return best;
}

/*
 * draft  [B, T-1]  draft[b][j] is the proposal checked against logits row j
 * logits [B, T, V]
 * n_acc[b]  = first j in [0, T-2] with draft[b][j] != argmax(row j), else T-1
 * corr[b]   = argmax of row n_acc[b] (the target's own token there)
 * amax [B, T] (optional) the per-row argmax
 */
int oracle_accept_greedy(const int *draft, const double *logits, int B, int T, int V,
                         int *n_acc, int *corr, int *amax) {
    if (B < 1 || T < 1 || V < 1) return -1;
    for (int b = 0; b < B; ++b) {
        int a[64];
        if (T > 64) return -1;
        for (int j = 0; j < T; ++j) {
            a[j] = argmax_lowest(logits + ((long)b * T + j) * V, V);
            if (amax) amax[b * T + j] = a[j];
        }
        int n = T - 1;
        for (int j = 0; j < T - 1; ++j) {
            if (draft[b * (T - 1) + j] != a[j]) { n = j; break; }
        }
        n_acc[b] = n;
        corr[b] = a[n];
    }
    return 0;
}

/*
 * Greedy acceptance over a draft tree (nodes in topological order, node 0 the
 * anchor; parent[b][j] < j, parent[b][0] = -1; token[b][j] is node j's
 * proposal, token[b][0] unused).  a_j = argmax of logits row j (ties: lowest
 * index).  The anchor is accepted; node j >= 1 is accepted when its parent
 * is and token[j] == a_parent(j) (the target's greedy pick after the
 * parent).  The committed path ends at the accepted node of greatest depth,
 * the lowest index among equals:
 *   n_acc[b]  its depth (proposals accepted), best[b] the node,
 *   corr[b]   a_best (the target's own next token),
 *   path[b]   the accepted nodes from depth 1 to n_acc, then -1.
 * A chain tree (parent j-1, token[j] = draft[j-1]) gives oracle_accept_greedy.
 */
int oracle_accept_tree_greedy(const int *token, const int *parent, const double *logits, int B, int T,
                              int V, int *n_acc, int *corr, int *best, int *path) {
    if (B < 1 || T < 1 || T > 64 || V < 1) return -1;
    for (int b = 0; b < B; ++b) {
        int a[64], acc[64], depth[64];
        for (int j = 0; j < T; ++j) a[j] = argmax_lowest(logits + ((long)b * T + j) * V, V);
        int bj = 0;
        for (int j = 0; j < T; ++j) {
            const int pj = parent[(long)b * T + j];
            if (j == 0) {
                if (pj != -1) return -1;
                acc[0] = 1; depth[0] = 0;
                continue;
            }
            if (pj < 0 || pj >= j) return -1;
            acc[j] = acc[pj] && token[(long)b * T + j] == a[pj];
            depth[j] = depth[pj] + 1;
            if (acc[j] && depth[j] > depth[bj]) bj = j;
        }
        n_acc[b] = depth[bj];
        corr[b] = a[bj];
        best[b] = bj;
        for (int k = 0; k < T; ++k) path[(long)b * T + k] = -1;
        for (int v = bj; v != 0; v = parent[(long)b * T + v]) path[(long)b * T + depth[v] - 1] = v;
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Sampled (lossless) acceptance                                             */
/* ------------------------------------------------------------------------ */

/* p = softmax(row / tau) in fp64 */
static void softmax_tau(const double *row, int V, double tau, double *p) {
    double m = row[0];
    for (int i = 1; i < V; ++i) if (row[i] > m) m = row[i];
    double z = 0.0;
    for (int i = 0; i < V; ++i) { p[i] = exp((row[i] - m) / tau); z += p[i]; }
    for (int i = 0; i < V; ++i) p[i] /= z;
}

/* smallest i with inclusive ascending cumsum C_i > x; reports C_{i-1}, C_i */
static int inverse_cdf(const double *w, int V, double x, double *c_prev, double *c_at) {
    double c = 0.0, prev = 0.0;
    int last_pos = -1;
    for (int i = 0; i < V; ++i) {
        prev = c;
        c += w[i];
        if (w[i] > 0.0) last_pos = i;
        if (c > x) { *c_prev = prev; *c_at = c; return i; }
    }
    /* only reachable if x >= the total through rounding: take the last
       index with positive weight */
    *c_prev = prev; *c_at = c;
    return last_pos < 0 ? V - 1 : last_pos;
}

/*
 * Standard speculative acceptance-rejection over one block.
 * draft [B, T-1], q [B, T, V] (rows 0..T-2 used; already normalised draft
 * distributions), logits [B, T, V], tau > 0.
 *  p_j = softmax(logits_j / tau)
 *  for j = 0..T-2: u_j = U(seed; j, b, stream 0, offset); accept d_j iff
 *                  u_j * q_j(d_j) < p_j(d_j); the first reject stops the scan.
 *  rejected at n: r = max(p_n - q_n, 0), S = sum r; u' = U(seed; n, b, 1, offset);
 *                 next = inverse cdf of r at u' * S (if S == 0, of p_n).
 *  all accepted:  next = inverse cdf of p_{T-1} at u' * sum p_{T-1}, u' from row T-1.
 * diag (optional) [B, 2*(T-1) + 6]: per b the u_j then p_j(d_j)/q_j(d_j) for the
 *  rows scanned (NaN for rows not scanned), then x = u' * S, S, C_{i-1}, C_i,
 *  the draw mode (0 residual, 1 p) and u'.
 */
int oracle_accept_sample(const int *draft, const double *q, const double *logits,
                         int B, int T, int V, double tau, uint64_t seed, uint32_t offset,
                         int *n_acc, int *next_id, double *diag) {
    if (B < 1 || T < 1 || V < 1 || !(tau > 0.0)) return -1;
    double *p = (double *)malloc(sizeof(double) * (size_t)V);
    double *r = (double *)malloc(sizeof(double) * (size_t)V);
    if (!p || !r) { free(p); free(r); return -1; }
    const int nd = 2 * (T - 1) + 6;
    for (int b = 0; b < B; ++b) {
        double *dg = diag ? diag + (long)b * nd : NULL;
        if (dg) for (int i = 0; i < nd; ++i) dg[i] = NAN;
        int n = T - 1;
        for (int j = 0; j < T - 1; ++j) {
            int d = draft[b * (T - 1) + j];
            if (d < 0 || d >= V) { free(p); free(r); return -1; }
            softmax_tau(logits + ((long)b * T + j) * V, V, tau, p);
            double qd = q[((long)b * T + j) * V + d];
            double u = oracle_uniform(seed, (uint32_t)j, (uint32_t)b, 0u, offset);
            if (dg) { dg[j] = u; dg[(T - 1) + j] = qd > 0.0 ? p[d] / qd : INFINITY; }
            if (!(u * qd < p[d])) { n = j; break; }
        }
        double u2 = oracle_uniform(seed, (uint32_t)n, (uint32_t)b, 1u, offset);
        softmax_tau(logits + ((long)b * T + n) * V, V, tau, p);
        const double *w = p;
        int mode = 1;
        if (n < T - 1) {
            const double *qn = q + ((long)b * T + n) * V;
            double S = 0.0;
            for (int i = 0; i < V; ++i) { r[i] = p[i] - qn[i] > 0.0 ? p[i] - qn[i] : 0.0; S += r[i]; }
            if (S > 0.0) { w = r; mode = 0; }
        }
        double S = 0.0;
        for (int i = 0; i < V; ++i) S += w[i];
        double x = u2 * S, c_prev = 0.0, c_at = 0.0;
        int id = inverse_cdf(w, V, x, &c_prev, &c_at);
        n_acc[b] = n;
        next_id[b] = id;
        if (dg) {
            dg[2 * (T - 1) + 0] = x;
            dg[2 * (T - 1) + 1] = S;
            dg[2 * (T - 1) + 2] = c_prev;
            dg[2 * (T - 1) + 3] = c_at;
            dg[2 * (T - 1) + 4] = (double)mode;
            dg[2 * (T - 1) + 5] = u2;
        }
    }
    free(p); free(r);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Commit / rollback                                                         */
/* ------------------------------------------------------------------------ */

/*
 * Commit of a verified block ("VFlash-FM" project page, "How VFlash-FM
 * works", the worked cycle: the accepted prefix and the target's own token at
 * the first disagreement are committed, everything after them is dropped,
 * and the next cycle starts from that token as its anchor).  Sequence b with
 * n = n_acc[b] kept proposals:
 *   kept proposal i (i < n): chain (path NULL) prop[b*ps + i]; tree
 *     prop[b*ps + path[b*T + i]] (path lists the kept nodes by depth)
 *   out_tokens[b*out_cap + out_len[b] + i] = kept proposal i, then
 *   out_tokens[b*out_cap + out_len[b] + n] = next_tok[b]; out_len[b] += n + 1
 *   ctx_len[b] += n + 1: ctx counts the anchor, so the new anchor (next_tok)
 *     sits at position ctx_len[b] - 1
 *   draft_ctx[b] = ctx_len[b] - 1 when given: the drafter's context is every
 *     position before the anchor
 *   anchor[b] = next_tok[b]
 * A sequence with n outside [0, T-1], a kept node outside [1, T), ctx_len < 1
 * (it counts the anchor), out_len < 0, or a commit that would pass ctx_cap or
 * out_cap is left as it was and gets status[b] = 1; the others get 0.
 */
int oracle_commit_tokens(const int *prop, int ps, const int *path, const int *n_acc, const int *next_tok,
                         int B, int T, int *ctx_len, int ctx_cap, int *draft_ctx, int *out_tokens, int *out_len,
                         int out_cap, int *anchor, int *status) {
    if (B < 1 || T < 1 || ps < 0) return -1;
    for (int b = 0; b < B; ++b) {
        const int n = n_acc[b];
        int ok = n >= 0 && n <= T - 1;
        if (ok && path)
            for (int i = 0; i < n; ++i)
                if (path[b * T + i] < 1 || path[b * T + i] >= T) ok = 0;
        if (ok && (ctx_len[b] < 1 || out_len[b] < 0)) ok = 0; /* ctx counts the anchor: at least 1 */
        if (ok && ((long)ctx_len[b] + n + 1 > ctx_cap || (long)out_len[b] + n + 1 > out_cap)) ok = 0;
        status[b] = ok ? 0 : 1;
        if (!ok) continue;
        int *dst = out_tokens + (long)b * out_cap + out_len[b];
        for (int i = 0; i < n; ++i) dst[i] = path ? prop[(long)b * ps + path[b * T + i]] : prop[(long)b * ps + i];
        dst[n] = next_tok[b];
        out_len[b] += n + 1;
        ctx_len[b] += n + 1;
        if (draft_ctx) draft_ctx[b] = ctx_len[b] - 1;
        anchor[b] = next_tok[b];
    }
    return 0;
}

/*
 * Tree commit in the target's KV cache (same passage: only the accepted path
 * survives and the next block follows it).  Block slot k of sequence b sits
 * at cache position ctx_len[b] - 1 + k (the anchor at k = 0), ctx_len taken
 * before the commit.  For depth d = 1..n_acc[b], position ctx-1+d receives
 * the row that was at position ctx-1+path[b*T + d-1] (every kv head, K and
 * V); every other position keeps its row.  Rows move as raw bytes: es bytes
 * per element, strides sb, ss, sh in elements, D contiguous.  A sequence whose
 * block does not fit the S positions, whose n is outside [0, T-1] or whose
 * kept node is outside [1, T) is left alone with status[b] = 1.
 */
int oracle_compact_tree_kv(uint8_t *kc, uint8_t *vc, long sb, long ss, long sh, int es, const int *ctx_len,
                           const int *path, const int *n_acc, int B, int T, int S, int Hkv, int D, int *status) {
    if (B < 1 || T < 1 || Hkv < 1 || D < 1 || es < 1) return -1;
    const long row = (long)D * es;
    uint8_t *tmp = (uint8_t *)malloc((size_t)T * Hkv * row + 1);
    if (!tmp) return -1;
    for (int b = 0; b < B; ++b) {
        const int n = n_acc[b], c = ctx_len[b];
        int ok = n >= 0 && n <= T - 1 && c >= 1 && (long)c - 1 + T <= S;
        for (int i = 0; ok && i < n; ++i)
            if (path[b * T + i] < 1 || path[b * T + i] >= T) ok = 0;
        status[b] = ok ? 0 : 1;
        if (!ok) continue;
        for (int pass = 0; pass < 2; ++pass) {
            uint8_t *cache = pass == 0 ? kc : vc;
            /* read every kept row first, then write them in depth order */
            for (int d = 1; d <= n; ++d)
                for (int h = 0; h < Hkv; ++h) {
                    const long src = ((long)b * sb + (long)(c - 1 + path[b * T + d - 1]) * ss + (long)h * sh) * es;
                    memcpy(tmp + ((long)(d - 1) * Hkv + h) * row, cache + src, (size_t)row);
                }
            for (int d = 1; d <= n; ++d)
                for (int h = 0; h < Hkv; ++h) {
                    const long dst = ((long)b * sb + (long)(c - 1 + d) * ss + (long)h * sh) * es;
                    memcpy(cache + dst, tmp + ((long)(d - 1) * Hkv + h) * row, (size_t)row);
                }
        }
    }
    free(tmp);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Latent visual compressor                                                  */
/* ------------------------------------------------------------------------ */

/*
 * SpecFLASH latent visual compressor ("SpecFLASH" README, the first of the
 * draft model's two components): a learned set of Cq query vectors attends
 * over the N visual features of the second-to-top layer and returns Cq latent
 * features, out = softmax(Q . F^T) . F, the softmax over the N features of
 * each query.  The formula applies no scale to the scores, so none is applied
 * here.  Keys and values are separate arguments (the method passes F for
 * both) so that the same routine also gives sum_n p_n |F_n|, the weighted
 * magnitude that bounds a kernel's rounding.
 *   q [Cq, d], k [N, d], v [N, d], out [Cq, d]; exact fp64, max-subtracted.
 */
int oracle_latent_compress(const double *q, const double *k, const double *v, int Cq, int N, int d, double *out) {
    if (Cq < 1 || N < 1 || d < 1) return -1;
    double *s = (double *)malloc(sizeof(double) * (size_t)N);
    if (!s) return -1;
    for (int c = 0; c < Cq; ++c) {
        double m = -INFINITY;
        for (int n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int i = 0; i < d; ++i) acc += q[(long)c * d + i] * k[(long)n * d + i];
            s[n] = acc;
            if (acc > m) m = acc;
        }
        double l = 0.0;
        for (int n = 0; n < N; ++n) { s[n] = exp(s[n] - m); l += s[n]; }
        for (int i = 0; i < d; ++i) {
            double acc = 0.0;
            for (int n = 0; n < N; ++n) acc += s[n] * v[(long)n * d + i];
            out[(long)c * d + i] = acc / l;
        }
    }
    free(s);
    return 0;
}
