/*
 * CPU oracle for the speculative-decoding verification row.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header or constant with the CUDA
 * library; it is plain, single-threaded C in double precision, written so that
 * each step can be read against the pages:
 *
 *   - softmax of logits / T ........ vLLM learning book, section 2 (algorithm
 *                                     flowchart: p and q are the target and
 *                                     draft distributions); TensorRT-LLM
 *                                     walkthrough, rejection-sampling section
 *                                     (target and draft filtered alike).
 *   - left-to-right accept scan .... vLLM anatomy page, "Speculative Decoding"
 *                                     (accept/reject steps); vLLM learning
 *                                     book, section 2 (r < min(1, p/q)).
 *   - residual / bonus sample ....... vLLM anatomy page, same list (rebalanced
 *                                     distribution max(0, p - q) normalised;
 *                                     bonus token from row k+1).
 *   - output row, -1 padded ........ TensorRT-LLM walkthrough, rejection-
 *                                     sampling section (accepted_tokens
 *                                     [batch, D+1]).
 *   - greedy verify ................. Kestrel article, section 3.3 (accept
 *                                     while argmax equals the draft; emit the
 *                                     target's own token).
 *   - tree verify ................... TensorRT-LLM deployment page, "Eagle-2"
 *                                     section (paths [batch, max_decoding_
 *                                     tokens, max_path_len]).
 *   - rollback lengths .............. TensorRT-LLM walkthrough, update_requests
 *                                     and rewind_cache sections (rewind =
 *                                     verified - accepted; cursor truncation).
 *   - top-k / top-p filtering ....... TensorRT-LLM walkthrough, rejection-
 *                                     sampling section (the target must be
 *                                     filtered exactly as the draft was:
 *                                     same temperature, top-k, top-p).
 *   - stochastic tree verify ........ TensorRT-LLM deployment page, "目标模型
 *                                     验证：树注意力与批量并行" (tree tokens judged
 *                                     by rejection sampling; children chosen by
 *                                     top-K, "Eagle-2" section).
 *   - per-request uniforms .......... TensorRT-LLM walkthrough, rejection-
 *                                     sampling section (a Philox state of
 *                                     seed and offset per request); the
 *                                     generator is Philox4x32-10 as defined by
 *                                     Salmon, Moraes, Dror and Shaw, "Parallel
 *                                     random numbers: as easy as 1, 2, 3"
 *                                     (SC'11).
 *
 * Readings taken where the pages are silent:
 *   target row i and draft row i both describe token x_i; row k is the bonus
 *   row; uniforms[b, 0..k-1] drive the accept tests and uniforms[b, k] drives
 *   the single final sample; accept iff r < p/q (q == 0 accepts); the inverse
 *   CDF picks the smallest t with C(t) > u*Z; argmax ties go to the lowest id.
 *
 * Precision: every logit is widened exactly to double, z = x / T in double,
 * exp() from libm, all sums sequential in token order.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_EINVAL (-1)
#define ORC_EBADINDEX (-2)
#define ORC_ENOMEM (-6)

#define ORC_F32 0
#define ORC_BF16 1

/* Near-tie windows: an accept test with |r - p/q| below ACCEPT_TIE, or a final
 * sample whose u*Z lies within SAMPLE_TIE*Z of a CDF boundary, is flagged. */
static const double ACCEPT_TIE = 1e-5;
static const double SAMPLE_TIE = 1e-6;

/* One stored logit, widened exactly to double. */
static double logit_at(const void *base, int dtype, size_t i)
{
    if (dtype == ORC_F32)
        return (double)((const float *)base)[i];
    uint32_t bits = (uint32_t)((const uint16_t *)base)[i] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* p(t) = exp(z_t - max z) / sum_s exp(z_s - max z), z = x / T. */
int oracle_softmax(const void *x, int dtype, double temperature, int V, double *p)
{
    if (!x || !p || V < 1 || !(temperature > 0.0) || (dtype != ORC_F32 && dtype != ORC_BF16))
        return ORC_EINVAL;
    double zmax = -INFINITY;
    for (int t = 0; t < V; ++t) {
        p[t] = logit_at(x, dtype, (size_t)t) / temperature;
        if (p[t] > zmax)
            zmax = p[t];
    }
    double sum = 0.0;
    for (int t = 0; t < V; ++t) {
        p[t] = exp(p[t] - zmax);
        sum += p[t];
    }
    for (int t = 0; t < V; ++t)
        p[t] /= sum;
    return ORC_OK;
}

/* Inverse-CDF draw from non-negative weights w[0..V).
 * Returns the smallest t with C(t) = w_0 + ... + w_t > u * Z, Z = C(V-1); when
 * rounding leaves no such t, the last t with w_t > 0.  Returns -1 if Z == 0.
 * *near_tie is set when u*Z lies within tol*Z of C(t) or of C(t-1). */
int oracle_inverse_cdf(const double *w, int V, double u, double tol, int32_t *near_tie)
{
    if (near_tie)
        *near_tie = 0;
    if (!w || V < 1)
        return ORC_EINVAL;
    double Z = 0.0;
    for (int t = 0; t < V; ++t)
        Z += w[t];
    if (!(Z > 0.0))
        return -1;
    double target = u * Z;
    double c_prev = 0.0, c = 0.0;
    int tok = -1;
    for (int t = 0; t < V; ++t) {
        c_prev = c;
        c += w[t];
        if (c > target) {
            tok = t;
            break;
        }
    }
    if (tok < 0) {
        for (int t = V - 1; t >= 0; --t)
            if (w[t] > 0.0) {
                tok = t;
                break;
            }
        c = Z;
        c_prev = Z - w[tok];
    }
    if (near_tie)
        *near_tie = (fabs(c - target) <= tol * Z) || (fabs(c_prev - target) <= tol * Z);
    return tok;
}

/* First index of the largest stored value (ties: lowest index). */
int oracle_argmax(const void *x, int dtype, int V)
{
    if (!x || V < 1)
        return ORC_EINVAL;
    int best = 0;
    double bv = logit_at(x, dtype, 0);
    for (int t = 1; t < V; ++t) {
        double v = logit_at(x, dtype, (size_t)t);
        if (v > bv) {
            bv = v;
            best = t;
        }
    }
    return best;
}

static void fail_closed_row(int32_t *row, int width, int32_t *n_acc)
{
    for (int i = 0; i < width; ++i)
        row[i] = -1;
    *n_acc = -1;
}

/* Chain rejection-sampling verify for B requests with up to k drafts each.
 *   target:  [B, k+1, V] logits (row k is the bonus row)
 *   draft:   [B, k, V] logits
 *   draft_tokens [B, k], uniforms [B, k+1] (column k drives the final sample)
 *   draft_lens [B] (nullable; NULL = k for every request): request b has
 *     k_b <= k real drafts in a buffer padded to k (TensorRT-LLM walkthrough,
 *     pad_draft_tokens_for_cuda_graph and the ragged verify_lens).  It is
 *     verified as a chain of k_b: accept tests on positions 0..k_b-1, column
 *     k_b of the uniforms drives the final sample, row k_b of the target is
 *     its bonus row; padded positions are neither read nor checked, and
 *     their probabilities are NaN.  A length outside [0, k] fails closed.
 *   out_tokens [B, k+1]: accepted drafts, then the corrected/bonus token, -1 pad
 *   out_num_accepted [B]: n_acc in [0, k]; -1 for a request whose draft token
 *     lies outside [0, V) (its row is all -1 and the call returns EBADINDEX)
 *   out_probs [B, k, 2] (nullable): p_i(x_i), q_i(x_i)
 *   out_flags [B, k+1] (nullable): 1 at each accept test that is a near-tie
 *     (positions 0..n_acc), and at column k when the final sample is one. */
int oracle_verify_chain(const void *target, const void *draft, int dtype,
                        const int32_t *draft_tokens, const float *uniforms,
                        const int32_t *draft_lens, float temperature, int B, int k, int V,
                        int32_t *out_tokens, int32_t *out_num_accepted,
                        double *out_probs, int32_t *out_flags)
{
    if (!target || !draft || !draft_tokens || !uniforms || !out_tokens || !out_num_accepted ||
        B < 1 || k < 1 || V < 2 || !(temperature > 0.0f) || !isfinite(temperature) ||
        (dtype != ORC_F32 && dtype != ORC_BF16))
        return ORC_EINVAL;
    const double T = (double)temperature;
    double *p = malloc(sizeof(double) * (size_t)V);
    double *q = malloc(sizeof(double) * (size_t)V);
    double *w = malloc(sizeof(double) * (size_t)V);
    double *ratio = malloc(sizeof(double) * (size_t)k);
    if (!p || !q || !w || !ratio) {
        free(p), free(q), free(w), free(ratio);
        return ORC_ENOMEM;
    }
    const size_t es = dtype == ORC_F32 ? 4 : 2;
    int rc = ORC_OK;
    for (int b = 0; b < B; ++b) {
        const char *tb = (const char *)target + (size_t)b * (size_t)(k + 1) * (size_t)V * es;
        const char *db = (const char *)draft + (size_t)b * (size_t)k * (size_t)V * es;
        const int32_t *x = draft_tokens + (size_t)b * k;
        const float *r = uniforms + (size_t)b * (k + 1);
        int32_t *out = out_tokens + (size_t)b * (k + 1);
        int32_t *flags = out_flags ? out_flags + (size_t)b * (k + 1) : NULL;
        if (flags)
            for (int i = 0; i <= k; ++i)
                flags[i] = 0;
        const int kb = draft_lens ? draft_lens[b] : k;
        int bad = kb < 0 || kb > k;
        for (int i = 0; !bad && i < kb; ++i)
            if (x[i] < 0 || x[i] >= V)
                bad = 1;
        if (bad) {
            fail_closed_row(out, k + 1, &out_num_accepted[b]);
            if (out_probs)
                for (int i = 0; i < 2 * k; ++i)
                    out_probs[(size_t)b * 2 * k + i] = NAN;
            rc = ORC_EBADINDEX;
            continue;
        }
        if (out_probs)
            for (int i = kb; i < k; ++i)
                out_probs[((size_t)b * k + i) * 2 + 0] = out_probs[((size_t)b * k + i) * 2 + 1] = NAN;
        /* p_i(x_i) and q_i(x_i) for every draft position. */
        for (int i = 0; i < kb; ++i) {
            oracle_softmax(tb + (size_t)i * V * es, dtype, T, V, p);
            oracle_softmax(db + (size_t)i * V * es, dtype, T, V, q);
            double pi = p[x[i]], qi = q[x[i]];
            if (out_probs) {
                out_probs[((size_t)b * k + i) * 2 + 0] = pi;
                out_probs[((size_t)b * k + i) * 2 + 1] = qi;
            }
            ratio[i] = qi > 0.0 ? pi / qi : INFINITY;
        }
        /* Left to right: accept x_i while r_i < p_i(x_i) / q_i(x_i). */
        int j = kb;
        for (int i = 0; i < kb; ++i) {
            if (flags && fabs((double)r[i] - ratio[i]) < ACCEPT_TIE)
                flags[i] = 1;
            if (!((double)r[i] < ratio[i])) {
                j = i;
                break;
            }
        }
        /* Final token: residual max(0, p_j - q_j) after a rejection, else the
         * bonus row p_{k_b}. */
        oracle_softmax(tb + (size_t)j * V * es, dtype, T, V, p);
        if (j < kb) {
            oracle_softmax(db + (size_t)j * V * es, dtype, T, V, q);
            for (int t = 0; t < V; ++t)
                w[t] = p[t] - q[t] > 0.0 ? p[t] - q[t] : 0.0;
        } else {
            memcpy(w, p, sizeof(double) * (size_t)V);
        }
        int32_t tie = 0;
        int tok = oracle_inverse_cdf(w, V, (double)r[kb], SAMPLE_TIE, &tie);
        if (tok < 0) /* residual mass vanished numerically: fall back to p_j */
            tok = oracle_inverse_cdf(p, V, (double)r[kb], SAMPLE_TIE, &tie);
        if (flags)
            flags[k] = tie;
        for (int i = 0; i < j; ++i)
            out[i] = x[i];
        out[j] = tok;
        for (int i = j + 1; i <= k; ++i)
            out[i] = -1;
        out_num_accepted[b] = j;
    }
    free(p), free(q), free(w), free(ratio);
    return rc;
}

/* Greedy chain verify: g_i = argmax target[b,i,:]; n_acc = the longest prefix
 * with g_i == d_i; output d_0..d_{n_acc-1}, g_{n_acc}, -1 pad.  draft_lens
 * (nullable) as for the chain: request b has k_b real drafts; a length
 * outside [0, k] fails closed. */
int oracle_verify_greedy(const void *target, int dtype, const int32_t *draft_tokens,
                         const int32_t *draft_lens, int B, int k, int V, int32_t *out_tokens,
                         int32_t *out_num_accepted)
{
    if (!target || !draft_tokens || !out_tokens || !out_num_accepted || B < 1 || k < 1 || V < 2 ||
        (dtype != ORC_F32 && dtype != ORC_BF16))
        return ORC_EINVAL;
    const size_t es = dtype == ORC_F32 ? 4 : 2;
    int rc = ORC_OK;
    for (int b = 0; b < B; ++b) {
        const char *tb = (const char *)target + (size_t)b * (size_t)(k + 1) * (size_t)V * es;
        const int32_t *d = draft_tokens + (size_t)b * k;
        int32_t *out = out_tokens + (size_t)b * (k + 1);
        const int kb = draft_lens ? draft_lens[b] : k;
        int bad = kb < 0 || kb > k;
        for (int i = 0; !bad && i < kb; ++i)
            if (d[i] < 0 || d[i] >= V)
                bad = 1;
        if (bad) {
            fail_closed_row(out, k + 1, &out_num_accepted[b]);
            rc = ORC_EBADINDEX;
            continue;
        }
        int j = 0;
        while (j < kb && oracle_argmax(tb + (size_t)j * V * es, dtype, V) == d[j])
            ++j;
        for (int i = 0; i < j; ++i)
            out[i] = d[i];
        out[j] = oracle_argmax(tb + (size_t)j * V * es, dtype, V);
        for (int i = j + 1; i <= k; ++i)
            out[i] = -1;
        out_num_accepted[b] = j;
    }
    return rc;
}

/* Greedy tree verify over EAGLE-style paths.
 *   target [B, N, V]: row n is the distribution after node n (node 0 = root)
 *   tree_tokens [B, N]: node n's token; paths [B, P, L]: root-to-leaf node
 *   lists, -1 padded; a path whose first entry is -1 is unused, a used path
 *   starts at node 0.
 * For each used path walk j = 1..L-1 while the node is >= 0 and its token
 * equals argmax of its parent's row; keep the path with the most accepted
 * steps (ties: lowest path index).  Outputs: out_tokens [B, L] = accepted
 * tokens then argmax of the last accepted node's row, -1 pad;
 * out_best_path [B] (nullable, -1 when no path is used);
 * out_accepted_nodes [B, L] (nullable) = root and accepted nodes, -1 pad.
 * A request with a node id outside [-1, N), a path that starts elsewhere than
 * 0 or -1, or a token outside [0, V) fails closed (n_acc -1, rows all -1). */
int oracle_verify_tree(const void *target, int dtype, const int32_t *tree_tokens,
                       const int32_t *paths, int B, int N, int P, int L, int V,
                       int32_t *out_tokens, int32_t *out_num_accepted,
                       int32_t *out_best_path, int32_t *out_accepted_nodes)
{
    if (!target || !tree_tokens || !paths || !out_tokens || !out_num_accepted || B < 1 ||
        N < 1 || P < 1 || L < 2 || V < 2 || (dtype != ORC_F32 && dtype != ORC_BF16))
        return ORC_EINVAL;
    const size_t es = dtype == ORC_F32 ? 4 : 2;
    int *g = malloc(sizeof(int) * (size_t)N);
    if (!g)
        return ORC_ENOMEM;
    int rc = ORC_OK;
    for (int b = 0; b < B; ++b) {
        const char *tb = (const char *)target + (size_t)b * (size_t)N * (size_t)V * es;
        const int32_t *tok = tree_tokens + (size_t)b * N;
        const int32_t *pb = paths + (size_t)b * P * L;
        int32_t *out = out_tokens + (size_t)b * L;
        int32_t *nodes = out_accepted_nodes ? out_accepted_nodes + (size_t)b * L : NULL;
        int bad = 0;
        for (int n = 0; n < N; ++n)
            if (tok[n] < 0 || tok[n] >= V)
                bad = 1;
        for (int pth = 0; pth < P; ++pth) {
            if (pb[(size_t)pth * L] != 0 && pb[(size_t)pth * L] != -1)
                bad = 1;
            for (int j = 0; j < L; ++j) {
                int32_t nd = pb[(size_t)pth * L + j];
                if (nd < -1 || nd >= N)
                    bad = 1;
            }
        }
        if (bad) {
            fail_closed_row(out, L, &out_num_accepted[b]);
            if (nodes)
                for (int j = 0; j < L; ++j)
                    nodes[j] = -1;
            if (out_best_path)
                out_best_path[b] = -1;
            rc = ORC_EBADINDEX;
            continue;
        }
        for (int n = 0; n < N; ++n)
            g[n] = oracle_argmax(tb + (size_t)n * V * es, dtype, V);
        int best = -1, best_acc = -1;
        for (int pth = 0; pth < P; ++pth) {
            const int32_t *path = pb + (size_t)pth * L;
            if (path[0] < 0)
                continue;
            int acc = 0;
            for (int j = 1; j < L; ++j) {
                int32_t node = path[j];
                if (node < 0 || tok[node] != g[path[j - 1]])
                    break;
                ++acc;
            }
            if (acc > best_acc) {
                best_acc = acc;
                best = pth;
            }
        }
        int n_acc = best < 0 ? 0 : best_acc;
        int last = best < 0 ? 0 : pb[(size_t)best * L + n_acc];
        for (int j = 0; j < n_acc; ++j)
            out[j] = tok[pb[(size_t)best * L + j + 1]];
        out[n_acc] = g[last];
        for (int j = n_acc + 1; j < L; ++j)
            out[j] = -1;
        if (nodes) {
            for (int j = 0; j <= n_acc; ++j)
                nodes[j] = best < 0 ? 0 : pb[(size_t)best * L + j];
            for (int j = n_acc + 1; j < L; ++j)
                nodes[j] = -1;
        }
        if (out_best_path)
            out_best_path[b] = best;
        out_num_accepted[b] = n_acc;
    }
    free(g);
    return rc;
}

/* KV cursor rollback: new_len = old_len + n_acc + 1 (the last committed token
 * plus the accepted drafts stay visible), rewind = k - n_acc (rows written by
 * the verify window but not kept).  An entry with n_acc outside [0, k] keeps
 * its length (new_len = old_len), its rewind reads -1 (the Kestrel article's
 * convention: an invalid result is reported as -1, section 3.1) and the call
 * returns EBADINDEX. */
int oracle_rollback(const int32_t *old_lens, const int32_t *num_accepted, int k, int B,
                    int32_t *new_lens, int32_t *rewind_lens)
{
    if (!old_lens || !num_accepted || !new_lens || B < 1 || k < 0)
        return ORC_EINVAL;
    int rc = ORC_OK;
    for (int b = 0; b < B; ++b) {
        int32_t n = num_accepted[b];
        if (n < 0 || n > k) {
            new_lens[b] = old_lens[b];
            if (rewind_lens)
                rewind_lens[b] = -1;
            rc = ORC_EBADINDEX;
            continue;
        }
        new_lens[b] = old_lens[b] + n + 1;
        if (rewind_lens)
            rewind_lens[b] = k - n;
    }
    return rc;
}

/* Philox4x32-10 (Salmon et al., SC'11): ten rounds on a 128-bit counter
 * (c0..c3) under a 64-bit key (k0, k1).  A round multiplies c0 by 0xD2511F53
 * and c2 by 0xCD9E8D57 into 64-bit products, and the new counter is
 * (hi(c2*M1) ^ c1 ^ k0, lo(c2*M1), hi(c0*M0) ^ c3 ^ k1, lo(c0*M0)).  The key is
 * bumped by the Weyl constants (0x9E3779B9, 0xBB67AE85) between rounds. */
void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4])
{
    uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        const uint64_t p0 = (uint64_t)0xD2511F53u * c0;
        const uint64_t p1 = (uint64_t)0xCD9E8D57u * c2;
        const uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;
        const uint32_t n1 = (uint32_t)p1;
        const uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
        const uint32_t n3 = (uint32_t)p0;
        c0 = n0;
        c1 = n1;
        c2 = n2;
        c3 = n3;
    }
    out[0] = c0;
    out[1] = c1;
    out[2] = c2;
    out[3] = c3;
}

/* The uniforms of request b, i = 0..n-1 (this library's reading of the
 * pages' per-request (seed, offset) state): Philox4x32-10 with key = seed_b
 * (low word first) and counter = (low and high word of offset_b, i / 4, 0);
 * uniform i = (word i % 4 >> 8) * 2^-24, in [0, 1). */
int oracle_philox_uniforms(const uint64_t *seeds, const uint64_t *offsets, int B, int n,
                           float *out)
{
    if (!seeds || !offsets || !out || B < 1 || n < 1)
        return ORC_EINVAL;
    for (int b = 0; b < B; ++b) {
        const uint32_t key[2] = {(uint32_t)seeds[b], (uint32_t)(seeds[b] >> 32)};
        for (int i = 0; i < n; ++i) {
            const uint32_t ctr[4] = {(uint32_t)offsets[b], (uint32_t)(offsets[b] >> 32),
                                     (uint32_t)(i / 4), 0u};
            uint32_t r[4];
            oracle_philox4x32_10(ctr, key, r);
            out[(size_t)b * n + i] = (float)((double)(r[i % 4] >> 8) * (1.0 / 16777216.0));
        }
    }
    return ORC_OK;
}

/* Paged rollback (TensorRT-LLM walkthrough, rewind_cache: the logical length
 * shrinks, the block count needed is recomputed from tokens_per_block and
 * only the whole surplus blocks are returned, nothing is zeroed; the vLLM
 * learning book's free_extra_blocks_for_request keeps ceil(tokens /
 * block_size) blocks likewise).  Per request: k_b = draft_lens[b] (or k when
 * NULL); new_len = old + n + 1, rewind = k_b - n, and, when blocks_held is
 * given, free_blocks = max(0, blocks_held - ceil(new_len / tokens_per_block)).
 * An entry with k_b outside [0, k] or n outside [0, k_b] keeps its length
 * (rewind -1, free 0) and the call returns EBADINDEX. */
int oracle_rollback_paged(const int32_t *old_lens, const int32_t *num_accepted,
                          const int32_t *draft_lens, int k, const int32_t *blocks_held,
                          int tokens_per_block, int B, int32_t *new_lens, int32_t *rewind_lens,
                          int32_t *free_blocks)
{
    if (!old_lens || !num_accepted || !new_lens || B < 1 || k < 0 || tokens_per_block < 1)
        return ORC_EINVAL;
    int rc = ORC_OK;
    for (int b = 0; b < B; ++b) {
        const int32_t kb = draft_lens ? draft_lens[b] : k;
        const int32_t n = num_accepted[b];
        if (kb < 0 || kb > k || n < 0 || n > kb) {
            new_lens[b] = old_lens[b];
            if (rewind_lens)
                rewind_lens[b] = -1;
            if (free_blocks)
                free_blocks[b] = 0;
            rc = ORC_EBADINDEX;
            continue;
        }
        const long long len = (long long)old_lens[b] + n + 1;
        new_lens[b] = (int32_t)len;
        if (rewind_lens)
            rewind_lens[b] = kb - n;
        if (free_blocks) {
            const long long need = (len + tokens_per_block - 1) / tokens_per_block;
            const long long spare = blocks_held ? (long long)blocks_held[b] - need : 0;
            free_blocks[b] = spare > 0 ? (int32_t)spare : 0;
        }
    }
    return rc;
}

/* One row's filtered distribution (TensorRT-LLM walkthrough, rejection-
 * sampling section: target and draft are filtered alike by temperature,
 * top-k, top-p and min_p, named in that order).  This library's reading,
 * applied in that order to z = x / T:
 *   top-k  the top_k tokens ordered by (logit descending, index ascending);
 *          top_k <= 0: every token, in that order;
 *   top-p  when top_p < 1, only the shortest prefix of that order whose
 *          probability under softmax(z) over the current set reaches top_p;
 *   min_p  when min_p > 0, only the tokens of the current set whose
 *          probability is at least min_p times the largest, that is
 *          exp(z_t - z_max) >= min_p (the normaliser cancels);
 * p[t] = exp(z_t - z_max) / sum over the kept set, 0 elsewhere.
 * *near_tie is set when the top-p cut lies within 1e-6 of top_p, or a kept
 * set token's exp(z_t - z_max) lies within 1e-6 * min_p of min_p. */
typedef struct {
    double x;
    int t;
} orc_item;

static int orc_item_order(const void *a, const void *b)
{
    const orc_item *u = (const orc_item *)a, *v = (const orc_item *)b;
    if (u->x > v->x)
        return -1;
    if (u->x < v->x)
        return 1;
    return u->t < v->t ? -1 : (u->t > v->t);
}

int oracle_filter_row(const void *x, int dtype, double temperature, int V, int top_k,
                      double top_p, double min_p, double *p, int32_t *near_tie)
{
    if (near_tie)
        *near_tie = 0;
    if (!x || !p || V < 1 || !(temperature > 0.0) || !(top_p > 0.0) || top_p > 1.0 ||
        !(min_p >= 0.0) || min_p > 1.0)
        return ORC_EINVAL;
    orc_item *it = malloc(sizeof(orc_item) * (size_t)V);
    if (!it)
        return ORC_ENOMEM;
    for (int t = 0; t < V; ++t) {
        it[t].x = logit_at(x, dtype, (size_t)t);
        it[t].t = t;
    }
    qsort(it, (size_t)V, sizeof(orc_item), orc_item_order);
    const int kk = top_k > 0 && top_k < V ? top_k : V;
    const double zmax = it[0].x / temperature;
    double sk = 0.0;
    for (int i = 0; i < kk; ++i)
        sk += exp(it[i].x / temperature - zmax);
    int m = kk;
    if (top_p < 1.0) {
        double cum = 0.0;
        for (int i = 0; i < kk; ++i) {
            const double pi = exp(it[i].x / temperature - zmax) / sk;
            const double before = cum;
            cum += pi;
            if (cum >= top_p) {
                m = i + 1;
                if (near_tie && (fabs(cum - top_p) < 1e-6 || fabs(before - top_p) < 1e-6))
                    *near_tie = 1;
                break;
            }
        }
    }
    if (min_p > 0.0) {
        int m2 = 0;
        for (int i = 0; i < m; ++i) {
            const double ratio = exp(it[i].x / temperature - zmax);
            if (near_tie && fabs(ratio - min_p) <= 1e-6 * min_p)
                *near_tie = 1;
            if (ratio >= min_p)
                m2 = i + 1;
        }
        m = m2;
    }
    for (int t = 0; t < V; ++t)
        p[t] = 0.0;
    double sm = 0.0;
    for (int i = 0; i < m; ++i)
        sm += exp(it[i].x / temperature - zmax);
    for (int i = 0; i < m; ++i)
        p[it[i].t] = exp(it[i].x / temperature - zmax) / sm;
    free(it);
    return ORC_OK;
}

/* top-k and top-p alone (min_p = 0); top_k <= 0 with top_p = 1 is the plain
 * softmax. */
int oracle_filtered_softmax(const void *x, int dtype, double temperature, int V, int top_k,
                            double top_p, double *p, int32_t *near_tie)
{
    return oracle_filter_row(x, dtype, temperature, V, top_k, top_p, 0.0, p, near_tie);
}

/* Chain verify on filtered distributions: oracle_verify_chain with every
 * target and draft row passed through oracle_filter_row(top_k, top_p, min_p)
 * before the accept tests and the final sample.  A near tie of a top-p cut in
 * a row that decides position i (its target or draft row) flags column i; one
 * in the rows of the final sample flags column k. */
int oracle_verify_chain_filtered(const void *target, const void *draft, int dtype,
                                 const int32_t *draft_tokens, const float *uniforms,
                                 float temperature, int top_k, double top_p, double min_p, int B,
                                 int k, int V,
                                 int32_t *out_tokens, int32_t *out_num_accepted,
                                 double *out_probs, int32_t *out_flags)
{
    if (!target || !draft || !draft_tokens || !uniforms || !out_tokens || !out_num_accepted ||
        B < 1 || k < 1 || V < 2 || top_k < 0 || !(temperature > 0.0f) || !isfinite(temperature) ||
        (dtype != ORC_F32 && dtype != ORC_BF16))
        return ORC_EINVAL;
    const double T = (double)temperature;
    double *p = malloc(sizeof(double) * (size_t)V);
    double *q = malloc(sizeof(double) * (size_t)V);
    double *w = malloc(sizeof(double) * (size_t)V);
    double *ratio = malloc(sizeof(double) * (size_t)k);
    int32_t *rowtie = malloc(sizeof(int32_t) * (size_t)k);
    if (!p || !q || !w || !ratio || !rowtie) {
        free(p), free(q), free(w), free(ratio), free(rowtie);
        return ORC_ENOMEM;
    }
    const size_t es = dtype == ORC_F32 ? 4 : 2;
    int rc = ORC_OK;
    for (int b = 0; b < B; ++b) {
        const char *tb = (const char *)target + (size_t)b * (size_t)(k + 1) * (size_t)V * es;
        const char *db = (const char *)draft + (size_t)b * (size_t)k * (size_t)V * es;
        const int32_t *x = draft_tokens + (size_t)b * k;
        const float *r = uniforms + (size_t)b * (k + 1);
        int32_t *out = out_tokens + (size_t)b * (k + 1);
        int32_t *flags = out_flags ? out_flags + (size_t)b * (k + 1) : NULL;
        if (flags)
            for (int i = 0; i <= k; ++i)
                flags[i] = 0;
        int bad = 0;
        for (int i = 0; i < k; ++i)
            if (x[i] < 0 || x[i] >= V)
                bad = 1;
        if (bad) {
            fail_closed_row(out, k + 1, &out_num_accepted[b]);
            if (out_probs)
                for (int i = 0; i < 2 * k; ++i)
                    out_probs[(size_t)b * 2 * k + i] = NAN;
            rc = ORC_EBADINDEX;
            continue;
        }
        for (int i = 0; i < k; ++i) {
            int32_t tp = 0, tq = 0;
            oracle_filter_row(tb + (size_t)i * V * es, dtype, T, V, top_k, top_p, min_p, p, &tp);
            oracle_filter_row(db + (size_t)i * V * es, dtype, T, V, top_k, top_p, min_p, q, &tq);
            const double pi = p[x[i]], qi = q[x[i]];
            if (out_probs) {
                out_probs[((size_t)b * k + i) * 2 + 0] = pi;
                out_probs[((size_t)b * k + i) * 2 + 1] = qi;
            }
            ratio[i] = qi > 0.0 ? pi / qi : INFINITY;
            rowtie[i] = tp || tq;
        }
        int j = k;
        for (int i = 0; i < k; ++i) {
            if (flags && (fabs((double)r[i] - ratio[i]) < ACCEPT_TIE || rowtie[i]))
                flags[i] = 1;
            if (!((double)r[i] < ratio[i])) {
                j = i;
                break;
            }
        }
        int32_t tp = 0, tq = 0;
        oracle_filter_row(tb + (size_t)j * V * es, dtype, T, V, top_k, top_p, min_p, p, &tp);
        if (j < k) {
            oracle_filter_row(db + (size_t)j * V * es, dtype, T, V, top_k, top_p, min_p, q, &tq);
            for (int t = 0; t < V; ++t)
                w[t] = p[t] - q[t] > 0.0 ? p[t] - q[t] : 0.0;
        } else {
            memcpy(w, p, sizeof(double) * (size_t)V);
        }
        int32_t tie = 0;
        int tok = oracle_inverse_cdf(w, V, (double)r[k], SAMPLE_TIE, &tie);
        if (tok < 0)
            tok = oracle_inverse_cdf(p, V, (double)r[k], SAMPLE_TIE, &tie);
        if (flags)
            flags[k] = tie || tp || tq;
        for (int i = 0; i < j; ++i)
            out[i] = x[i];
        out[j] = tok;
        for (int i = j + 1; i <= k; ++i)
            out[i] = -1;
        out_num_accepted[b] = j;
    }
    free(p), free(q), free(w), free(ratio), free(rowtie);
    return rc;
}

/* Stochastic tree verify (TensorRT-LLM deployment page, "目标模型验证：树注意力
 * 与批量并行": the draft tree's tokens are judged against the target logits by
 * rejection sampling; the tree itself is built by top-K selection per level,
 * "Eagle-2 多层级树状草稿生成").  This library's reading: a node's children are
 * chosen, not sampled, so each child c is a point-mass proposal on its token,
 * and the rejection-sampling rule (accept with min(1, p/q), else continue
 * from max(0, p - q) normalised; vLLM anatomy page, "Speculative Decoding")
 * with q = that point mass becomes: accept c with probability p'(tok c), the
 * current residual of the node's target distribution; on a rejection remove
 * tok c from the residual (its mass max(0, p - 1) = 0) and renormalise.
 * The emitted tokens are then distributed exactly as sampling from the
 * target rows in turn.
 *   target [B, N, V]: row n is the distribution after node n (node 0 = root);
 *   tree_tokens [B, N]; paths [B, P, L] as for oracle_verify_tree;
 *   uniforms [B, N]: uniforms[b, n] (n >= 1) is node n's accept test, used
 *     when n is tried as a child; uniforms[b, 0] drives the final draw.
 * Walk: the accepted prefix starts as (0).  Its candidates are the distinct
 * nodes paths[p][d + 1] >= 0 of the used paths p whose first d + 1 entries
 * equal the prefix (d = its depth), tried in increasing node id.  With p the
 * softmax of the current node's row at T and R the tokens rejected so far at
 * this node, candidate c is accepted iff u[c] < p'(tok c) = [tok c not in R]
 * p(tok c) / (1 - sum over R of p); then c joins the prefix (at most L - 1
 * steps).  When no candidate is accepted (or none exists) the final token is
 * the inverse-CDF draw at u[0] from w_t = p(t) [t not in R] (from p itself if
 * that total vanishes).  Outputs as for oracle_verify_tree; out_best_path is
 * the lowest used path whose first n_acc + 1 entries are the accepted nodes.
 *   out_flags [B, N] (nullable): column c = 1 when c's accept test is a near
 *     tie, |u[c] - p'| below 1e-5 / (1 - sum over R of p) (the residual's
 *     normaliser divides the precision of p' as well), column 0 when the
 *     final draw is one (u*Z within 1e-6*Z of a CDF boundary).
 * A request with a token outside [0, V), a node id outside [-1, N) or a path
 * starting elsewhere than 0 or -1 fails closed (n_acc -1, rows all -1). */
int oracle_verify_tree_sampled(const void *target, int dtype, const int32_t *tree_tokens,
                               const int32_t *paths, const float *uniforms, float temperature,
                               int B, int N, int P, int L, int V, int32_t *out_tokens,
                               int32_t *out_num_accepted, int32_t *out_best_path,
                               int32_t *out_accepted_nodes, int32_t *out_flags)
{
    if (!target || !tree_tokens || !paths || !uniforms || !out_tokens || !out_num_accepted ||
        B < 1 || N < 1 || P < 1 || L < 2 || V < 2 || !(temperature > 0.0f) ||
        !isfinite(temperature) || (dtype != ORC_F32 && dtype != ORC_BF16))
        return ORC_EINVAL;
    const size_t es = dtype == ORC_F32 ? 4 : 2;
    const double T = (double)temperature;
    double *p = malloc(sizeof(double) * (size_t)V);
    double *w = malloc(sizeof(double) * (size_t)V);
    int *alive = malloc(sizeof(int) * (size_t)P);
    int *cand = malloc(sizeof(int) * (size_t)P);
    int *prefix = malloc(sizeof(int) * (size_t)L);
    if (!p || !w || !alive || !cand || !prefix) {
        free(p), free(w), free(alive), free(cand), free(prefix);
        return ORC_ENOMEM;
    }
    int rc = ORC_OK;
    for (int b = 0; b < B; ++b) {
        const char *tb = (const char *)target + (size_t)b * (size_t)N * (size_t)V * es;
        const int32_t *tok = tree_tokens + (size_t)b * N;
        const int32_t *pb = paths + (size_t)b * P * L;
        const float *u = uniforms + (size_t)b * N;
        int32_t *out = out_tokens + (size_t)b * L;
        int32_t *nodes = out_accepted_nodes ? out_accepted_nodes + (size_t)b * L : NULL;
        int32_t *flags = out_flags ? out_flags + (size_t)b * N : NULL;
        if (flags)
            for (int n = 0; n < N; ++n)
                flags[n] = 0;
        int bad = 0;
        for (int n = 0; n < N; ++n)
            if (tok[n] < 0 || tok[n] >= V)
                bad = 1;
        for (int pth = 0; pth < P; ++pth) {
            if (pb[(size_t)pth * L] != 0 && pb[(size_t)pth * L] != -1)
                bad = 1;
            for (int j = 0; j < L; ++j)
                if (pb[(size_t)pth * L + j] < -1 || pb[(size_t)pth * L + j] >= N)
                    bad = 1;
        }
        if (bad) {
            fail_closed_row(out, L, &out_num_accepted[b]);
            if (nodes)
                for (int j = 0; j < L; ++j)
                    nodes[j] = -1;
            if (out_best_path)
                out_best_path[b] = -1;
            rc = ORC_EBADINDEX;
            continue;
        }
        for (int pth = 0; pth < P; ++pth)
            alive[pth] = pb[(size_t)pth * L] == 0;
        prefix[0] = 0;
        int d = 0, node = 0, final_tok = -1;
        for (;;) {
            oracle_softmax(tb + (size_t)node * V * es, dtype, T, V, p);
            /* candidates: distinct next nodes of the paths still on the prefix */
            int nc = 0;
            if (d + 1 < L)
                for (int pth = 0; pth < P; ++pth) {
                    if (!alive[pth])
                        continue;
                    const int c = pb[(size_t)pth * L + d + 1];
                    if (c < 0)
                        continue;
                    int seen = 0;
                    for (int i = 0; i < nc; ++i)
                        seen |= cand[i] == c;
                    if (!seen)
                        cand[nc++] = c;
                }
            for (int i = 1; i < nc; ++i) /* increasing node id */
                for (int j2 = i; j2 > 0 && cand[j2 - 1] > cand[j2]; --j2) {
                    const int t = cand[j2];
                    cand[j2] = cand[j2 - 1];
                    cand[j2 - 1] = t;
                }
            double removed = 0.0;
            int next = -1;
            for (int i = 0; i < nc; ++i) {
                const int c = cand[i];
                const double pc = p[tok[c]];
                const double ratio = (1.0 - removed) > 0.0 ? pc / (1.0 - removed) : 0.0;
                if (flags && (1.0 - removed) > 0.0 &&
                    fabs((double)u[c] - ratio) < ACCEPT_TIE / (1.0 - removed))
                    flags[c] = 1;
                if ((double)u[c] < ratio) {
                    next = c;
                    break;
                }
                removed += pc;
                p[tok[c]] = 0.0; /* the residual no longer holds tok c */
            }
            if (next < 0) {
                for (int t = 0; t < V; ++t)
                    w[t] = p[t];
                int32_t tie = 0;
                final_tok = oracle_inverse_cdf(w, V, (double)u[0], SAMPLE_TIE, &tie);
                if (final_tok < 0) { /* the residual vanished: draw from the row itself */
                    oracle_softmax(tb + (size_t)node * V * es, dtype, T, V, p);
                    final_tok = oracle_inverse_cdf(p, V, (double)u[0], SAMPLE_TIE, &tie);
                }
                if (flags)
                    flags[0] = tie;
                break;
            }
            ++d;
            prefix[d] = next;
            node = next;
            for (int pth = 0; pth < P; ++pth)
                alive[pth] = alive[pth] && pb[(size_t)pth * L + d] == next;
        }
        int best = -1;
        for (int pth = 0; pth < P && best < 0; ++pth) {
            int ok = pb[(size_t)pth * L] == 0;
            for (int j = 1; ok && j <= d; ++j)
                ok = pb[(size_t)pth * L + j] == prefix[j];
            if (ok)
                best = pth;
        }
        for (int j = 0; j < d; ++j)
            out[j] = tok[prefix[j + 1]];
        out[d] = final_tok;
        for (int j = d + 1; j < L; ++j)
            out[j] = -1;
        if (nodes)
            for (int j = 0; j < L; ++j)
                nodes[j] = j <= d ? prefix[j] : -1;
        if (out_best_path)
            out_best_path[b] = best;
        out_num_accepted[b] = d;
    }
    free(p), free(w), free(alive), free(cand), free(prefix);
    return rc;
}
