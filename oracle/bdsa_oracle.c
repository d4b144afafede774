/*
 * bdsa_oracle.c -- plain, slow, fp64 CPU oracle for one block-diffusion
 * draft/verify step over a paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file: only tests/, the smoke check and the CPU-baseline leg of
 * bench.py do.  It shares no code, header, table or constant with the CUDA
 * library; it is written directly from the definitions on the source pages:
 *
 *   [P1] "From DFlash to dLLM Self-Spec (IV): Self-Spec dLLM & AR Uni-Model",
 *        sections 4.3.1 (p/q acceptance) and 4.4.1 (LinearSpec block init,
 *        causal verify, greedy longest-prefix loop with bonus); sections 4.3,
 *        4.3.1 and 4.6 for the I-DLM Block-N round (2N-1 layout, verify of
 *        the carried specs, new specs from the MASK positions, KV trim).
 *   [P2] "Unlocking Lossless Speedups in LLMs via Discrete Diffusion",
 *        background on speculative decoding / rejection sampling and the
 *        Psi-Spec sampling step (first token always accepted, longest
 *        accepted prefix, residual resampling).
 *   [P3] "From DFlash to dLLM Self-Spec (II): SGLang Spec V2", sections 2.2.2
 *        (prepare block: block_ids / positions / cache_loc) and 2.2.5
 *        (greedy accept/bonus rule, commit_len = accept_len + 1).
 *   [P4] "SGLang dLLM / LLaDA 2.0", section "Attention Mask" (context query
 *        sees the whole cache; intra-block query is a rectangle in block
 *        diffusion, a token-causal trapezoid in chunked prefill).
 *   [P3] section 2.2.6 and the DFlash engineering notes of "From DFlash to
 *        dLLM Self-Spec" for the KV materialisation of the committed prefix
 *        (projection across draft layers, K norm, RoPE, paged write).
 *
 * Every floating-point quantity is computed in fp64 from inputs widened
 * exactly (bf16 -> fp64, fp32 -> fp64), except the two decisions whose
 * precision the boundary fixes in fp32: the acceptance ratio p/q and the
 * residual weights max(0, p - q).  Loops follow the definitions literally: no
 * blocking, no fusion, no reordering beyond an OpenMP split over independent
 * outputs.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* bf16 -> fp64, exact: a bf16 value is the top 16 bits of an IEEE fp32.     */
static double bf16_to_f64(uint16_t h) {
    uint32_t bits = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* ------------------------------------------------------------------------ */
/* prepare_block  [P3 2.2.2; P1 4.4.1 block init; P3 2.3.5 planning_len]
 *
 * For request r and block slot i in [0, B):
 *   block_ids[r,i] = verified_id[r] if i == 0 else mask_token_id
 *   positions[r,i] = L_r + i                       (L_r = seq_lens[r])
 *   cache_loc[r,i] = page * page_size + (L_r + i) % page_size,
 *                    page = block_table[r, (L_r + i) / page_size]
 * Returns the number of (r,i) whose page lookup was out of range (those get
 * cache_loc = -1).
 */
int oracle_prepare_block(const int32_t *verified_id, const int32_t *seq_lens,
                         const int32_t *block_table, int max_pages_per_req,
                         int num_pages, int bs, int B, int page_size,
                         int mask_token_id, int32_t *block_ids,
                         int32_t *positions, int32_t *cache_loc) {
    int bad = 0;
    for (int r = 0; r < bs; ++r) {
        for (int i = 0; i < B; ++i) {
            long pos = (long)seq_lens[r] + i;
            block_ids[r * B + i] = (i == 0) ? verified_id[r] : mask_token_id;
            positions[r * B + i] = (int32_t)pos;
            long page_idx = pos / page_size;
            int32_t loc = -1;
            if (seq_lens[r] >= 0 && page_idx < max_pages_per_req) {
                int32_t page = block_table[(long)r * max_pages_per_req + page_idx];
                if (page >= 0 && page < num_pages)
                    loc = (int32_t)((long)page * page_size + pos % page_size);
            }
            if (loc < 0) ++bad;
            cache_loc[r * B + i] = loc;
        }
    }
    return bad;
}

/* ------------------------------------------------------------------------ */
/* Block attention over a paged cache  [P4 "Attention Mask"; P1 4.4.1;
 * P3 2.2.3-2.2.4]
 *
 * One output row: request r, block row i, query head j.  KV head h = j / G
 * (G = Hq / Hkv, contiguous groups).  Keys t in [0, L_r + B); key t of
 * request r lives at cache slot block_table[r, t/ps] * ps + t % ps.
 *   allowed(i, t) = t < L_r  (context query: whole cache)
 *                   or mode == DRAFT (0)   (rectangular intra-block mask)
 *                   or (t - L_r) <= i      (VERIFY (1): token-causal)
 *   s_t = scale * <q[r,i,j], k[t,h]>
 *   o   = sum_t softmax(s)_t v[t,h],   lse = log sum_t exp(s_t)
 * Written as a two-pass softmax: scores, max, exp-sum, weighted sum.
 * Returns 0, or -1 if a needed page id is out of range.
 */
static int attn_one_row(const uint16_t *q, const uint16_t *k_cache,
                        const uint16_t *v_cache, const int32_t *block_table,
                        int max_pages_per_req, int num_pages,
                        const int32_t *seq_lens, int B, int Hq, int Hkv, int D,
                        int page_size, double scale, int mode, int r, int i,
                        int j, double *scores, double *out_row,
                        double *lse_out) {
    int G = Hq / Hkv;
    int h = j / G;
    long L = seq_lens[r];
    long n_keys = L + B;
    const uint16_t *qrow = q + (((long)r * B + i) * Hq + j) * D;

    double smax = -INFINITY;
    for (long t = 0; t < n_keys; ++t) {
        int allowed = (t < L) || (mode == 0) || (t - L <= i);
        if (!allowed) {
            scores[t] = -INFINITY;
            continue;
        }
        long page_idx = t / page_size;
        if (page_idx >= max_pages_per_req) return -1;
        int32_t page = block_table[(long)r * max_pages_per_req + page_idx];
        if (page < 0 || page >= num_pages) return -1;
        long slot = (long)page * page_size + t % page_size;
        const uint16_t *krow = k_cache + (slot * Hkv + h) * D;
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += bf16_to_f64(qrow[d]) * bf16_to_f64(krow[d]);
        scores[t] = scale * dot;
        if (scores[t] > smax) smax = scores[t];
    }
    double denom = 0.0;
    for (long t = 0; t < n_keys; ++t) {
        if (scores[t] == -INFINITY) continue;
        denom += exp(scores[t] - smax);
    }
    for (int d = 0; d < D; ++d) out_row[d] = 0.0;
    for (long t = 0; t < n_keys; ++t) {
        if (scores[t] == -INFINITY) continue;
        double w = exp(scores[t] - smax) / denom;
        long page_idx = t / page_size;
        int32_t page = block_table[(long)r * max_pages_per_req + page_idx];
        long slot = (long)page * page_size + t % page_size;
        const uint16_t *vrow = v_cache + (slot * Hkv + h) * D;
        for (int d = 0; d < D; ++d) out_row[d] += w * bf16_to_f64(vrow[d]);
    }
    if (lse_out) *lse_out = smax + log(denom);
    return 0;
}

/* Full attention: out is [bs*B, Hq, D] fp64, lse is [bs*B, Hq] fp64 (may be
 * NULL).  Requests are independent; OpenMP splits over (r, j) pairs when
 * nthreads > 1.  Returns the number of rows that hit an out-of-range page. */
int oracle_block_attn(const uint16_t *q, const uint16_t *k_cache,
                      const uint16_t *v_cache, const int32_t *block_table,
                      int max_pages_per_req, int num_pages,
                      const int32_t *seq_lens, int bs, int B, int Hq, int Hkv,
                      int D, int page_size, double scale, int mode,
                      double *out, double *lse, int nthreads) {
    long max_keys = 0;
    for (int r = 0; r < bs; ++r)
        if ((long)seq_lens[r] + B > max_keys) max_keys = (long)seq_lens[r] + B;
    int bad = 0;
    long units = (long)bs * Hq;
#ifdef _OPENMP
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel num_threads(nthreads) reduction(+ : bad)
#endif
    {
        double *scores = (double *)malloc(sizeof(double) * (size_t)(max_keys > 0 ? max_keys : 1));
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (long u = 0; u < units; ++u) {
            int r = (int)(u / Hq), j = (int)(u % Hq);
            for (int i = 0; i < B; ++i) {
                long row = ((long)r * B + i) * Hq + j;
                double l = 0.0;
                int rc = attn_one_row(q, k_cache, v_cache, block_table, max_pages_per_req,
                                      num_pages, seq_lens, B, Hq, Hkv, D, page_size, scale,
                                      mode, r, i, j, scores, out + row * D, &l);
                if (rc != 0) {
                    ++bad;
                    for (int d = 0; d < D; ++d) out[row * D + d] = NAN;
                    l = NAN;
                }
                if (lse) lse[row] = l;
            }
        }
        free(scores);
    }
    return bad;
}

/* ------------------------------------------------------------------------ */
/* Speculative acceptance  [P1 4.3.1; P2 background + Psi-Spec step;
 * P3 2.2.5; P1 4.4.1 greedy loop]
 *
 * Row r, draft tokens d_i = block_ids[r, i] for i = 1..B-1 (slot 0 is the
 * already verified token and is never tested: the first token is always
 * accepted).  p[r, i] is the verifier distribution for block slot i+1
 * (p[r, B-1] is the bonus distribution); q[r, i-1] is the draft distribution
 * d_i was drawn from.  Strides are in elements.
 *
 * Stochastic (q != NULL):
 *   accept d_i  iff  u_acc[r, i-1] < min(1, p[i-1][d_i] / q[i-1][d_i])
 *                (fp32 ratio, IEEE correctly rounded; q == 0 accepts iff p > 0)
 *   a = number of leading accepted drafts
 *   a <  B-1: token = InvCDF(max(0, p[a] - q[a]), u_samp)  (fp32 weights;
 *             if they sum to 0, sample p[a] instead)
 *   a == B-1: token = InvCDF(p[B-1], u_samp)              (bonus)
 * Greedy (q == NULL):
 *   a = number of leading i with d_i == argmax p[i-1]  (lowest index on ties)
 *   token = argmax p[a]
 * InvCDF(w, u) = smallest k with C_k > u * S, C_k = sum_{j<=k} w_j in index
 * order, S = C_{V-1}, all sums in fp64.
 * Outputs: accept_len = a, commit_len = a + 1, out_tokens[r] = d_1..d_a,
 * token, -1 padding; bonus_id = token; new_seq_lens = seq_lens + a + 1.
 * flags[r] (may be NULL) marks rows whose integer result is decided within
 * the fp rounding margin and so is not unique across summation orders:
 *   bit 0: some tested |p/q - u| < 1e-6 (fp64)
 *   bit 1: u*S within 1e-9*S of C_{k-1} or C_k for the chosen k (the fp64
 *          sequential sums here carry < 2e-11*S error, any other exact-to-
 *          1e-13 summation order can only disagree inside this band)
 *   bit 2: residual mass was zero, sampled from p
 *   bit 3: a draft id was outside [0, V) (treated as rejected)
 *   bit 4: greedy argmax had a tie at a deciding position
 */
static int inv_cdf_f32w(const float *w, int V, double u, int *flag_near) {
    double S = 0.0;
    for (int k = 0; k < V; ++k) S += (double)w[k];
    double T = u * S;
    double C = 0.0, Cprev = 0.0;
    int chosen = -1;
    for (int k = 0; k < V; ++k) {
        Cprev = C;
        C += (double)w[k];
        if (C > T) {
            chosen = k;
            break;
        }
    }
    if (chosen < 0) { /* rounding fallback: last positive-weight index */
        for (int k = V - 1; k >= 0; --k)
            if (w[k] > 0.0f) {
                chosen = k;
                break;
            }
        if (flag_near) *flag_near = 1;
        return chosen;
    }
    if (flag_near && ((T - Cprev) < 1e-9 * S || (C - T) < 1e-9 * S)) *flag_near = 1;
    return chosen;
}

static int argmax_lowest(const float *x, int V, int *tie) {
    int best = 0;
    for (int k = 1; k < V; ++k)
        if (x[k] > x[best]) best = k;
    if (tie) {
        *tie = 0;
        for (int k = 0; k < V; ++k)
            if (k != best && x[k] == x[best]) *tie = 1;
    }
    return best;
}

void oracle_spec_accept(const int32_t *block_ids, const float *p, int64_t p_stride_r,
                        int64_t p_stride_i, const float *q, int64_t q_stride_r,
                        int64_t q_stride_i, const float *u_acc, const float *u_samp,
                        const int32_t *seq_lens, int bs, int B, int V, int32_t *accept_len,
                        int32_t *commit_len, int32_t *out_tokens, int32_t *bonus_id,
                        int32_t *new_seq_lens, int32_t *flags, int nthreads) {
#ifdef _OPENMP
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel num_threads(nthreads)
#endif
    {
        float *w = (float *)malloc(sizeof(float) * (size_t)V);
#ifdef _OPENMP
#pragma omp for schedule(static)
#endif
        for (int r = 0; r < bs; ++r) {
            int flag = 0;
            const int32_t *ids = block_ids + (long)r * B;
            int a = 0, token = -1;
            if (q != NULL) {
                for (int i = 1; i < B; ++i) {
                    int d = ids[i];
                    if (d < 0 || d >= V) {
                        flag |= 8;
                        break;
                    }
                    float pv = p[(long)r * p_stride_r + (long)(i - 1) * p_stride_i + d];
                    float qv = q[(long)r * q_stride_r + (long)(i - 1) * q_stride_i + d];
                    float u = u_acc[(long)r * (B - 1) + (i - 1)];
                    int acc;
                    if (qv == 0.0f) {
                        acc = pv > 0.0f;
                    } else {
                        volatile float ratio = pv / qv; /* fp32, correctly rounded */
                        float lim = ratio < 1.0f ? ratio : 1.0f;
                        acc = u < lim;
                        if (fabs((double)pv / (double)qv - (double)u) < 1e-6) flag |= 1;
                    }
                    if (!acc) break;
                    ++a;
                }
                const float *pa = p + (long)r * p_stride_r + (long)a * p_stride_i;
                int near = 0;
                if (a < B - 1) {
                    const float *qa = q + (long)r * q_stride_r + (long)a * q_stride_i;
                    int any = 0;
                    for (int k = 0; k < V; ++k) {
                        float diff = pa[k] - qa[k]; /* fp32 */
                        w[k] = diff > 0.0f ? diff : 0.0f;
                        if (w[k] > 0.0f) any = 1;
                    }
                    if (!any) {
                        flag |= 4;
                        token = inv_cdf_f32w(pa, V, (double)u_samp[r], &near);
                    } else {
                        token = inv_cdf_f32w(w, V, (double)u_samp[r], &near);
                    }
                } else {
                    token = inv_cdf_f32w(pa, V, (double)u_samp[r], &near);
                }
                if (near) flag |= 2;
            } else {
                for (int i = 1; i < B; ++i) {
                    int tie = 0;
                    int tp = argmax_lowest(p + (long)r * p_stride_r + (long)(i - 1) * p_stride_i, V, &tie);
                    if (tie) flag |= 16;
                    if (ids[i] != tp) break;
                    ++a;
                }
                int tie = 0;
                token = argmax_lowest(p + (long)r * p_stride_r + (long)a * p_stride_i, V, &tie);
                if (tie) flag |= 16;
            }
            accept_len[r] = a;
            commit_len[r] = a + 1;
            for (int i = 0; i < B; ++i) {
                int32_t v = -1;
                if (i < a) v = ids[i + 1];
                else if (i == a) v = token;
                out_tokens[(long)r * B + i] = v;
            }
            bonus_id[r] = token;
            new_seq_lens[r] = seq_lens[r] + a + 1;
            if (flags) flags[r] = flag;
        }
        free(w);
    }
}

/* ------------------------------------------------------------------------ */
/* I-DLM Block-N round  [P1 4.3 (ISD: the specs drawn from MASK positions in
 * round t are verified in round t+1 against the causal view), 4.3.1 (the
 * Block-N layouts, p/q acceptance with a correction token, MASK KV freed
 * after the forward), 4.6 (KV trim info and the request's advance)]
 *
 * A round has blk = 2N-1 block slots per request.  Slot j's logits predict
 * the token at slot j+1 (the causal view with a logit shift), p[r, j] being
 * their distribution.
 *   verify (mode 1): [pending, spec_0 .. spec_{N-2}, M x (N-1)]
 *   cold   (mode 0): [pending, M x (2N-2)]
 * idlm_prepare writes that layout, positions L_r + j and cache_loc exactly as
 * prepare_block does for a block of blk slots.  Any mode other than 1 is laid
 * out as a cold start.
 */
int oracle_idlm_prepare(const int32_t *pending, const int32_t *specs, const int32_t *mode,
                        const int32_t *seq_lens, const int32_t *block_table,
                        int max_pages_per_req, int num_pages, int bs, int N, int page_size,
                        int mask_token_id, int32_t *block_ids, int32_t *positions,
                        int32_t *cache_loc) {
    const int blk = 2 * N - 1;
    int bad = 0;
    for (int r = 0; r < bs; ++r) {
        for (int j = 0; j < blk; ++j) {
            int32_t id = mask_token_id;
            if (j == 0) id = pending[r];
            else if (mode[r] == 1 && j <= N - 1) id = specs[(long)r * (N - 1) + (j - 1)];
            long pos = (long)seq_lens[r] + j;
            block_ids[(long)r * blk + j] = id;
            positions[(long)r * blk + j] = (int32_t)pos;
            long page_idx = pos / page_size;
            int32_t loc = -1;
            if (seq_lens[r] >= 0 && page_idx < max_pages_per_req) {
                int32_t page = block_table[(long)r * max_pages_per_req + page_idx];
                if (page >= 0 && page < num_pages)
                    loc = (int32_t)((long)page * page_size + pos % page_size);
            }
            if (loc < 0) ++bad;
            cache_loc[(long)r * blk + j] = loc;
        }
    }
    return bad;
}

/* The verify / sample / trim step of the round, stochastic.
 *
 * q_prev[r, q_slot[r] + k] is the distribution spec_k was drawn from in the
 * previous round (its p rows, kept by the caller); strides in elements.
 * verify (mode 1):
 *   spec_k (slot k+1) is tested against p[r, k]: accept iff
 *     u_acc[r, k] < min(1, p[k][s] / q_prev[q_slot + k][s])   (fp32 ratio;
 *     q == 0 accepts iff p > 0; an id outside [0, V) is rejected, flag bit 3)
 *   a = leading accepted specs.
 *   a < N-1: anchor = InvCDF(max(0, p[a] - q_prev[q_slot + a]), u_samp[r, 0])
 *            (from p[a] if that has no mass, flag bit 2); no new specs; next
 *            round is a cold start.
 *   a = N-1: anchor = InvCDF(p[N-1], u_samp[r, 0]) (the bonus); new specs
 *            spec'_j = InvCDF(p[N + j], u_samp[r, 1 + j]), j < N-1 (the MASK
 *            slots N..2N-2 predict the slots after the bonus); next round
 *            verifies them against q_slot' = N.
 * cold (mode 0, and mode 1 with q_slot outside [0, N], flag bit 5):
 *   a = 0; anchor = InvCDF(p[0], u_samp[r, 0]); spec'_j = InvCDF(p[1 + j],
 *   u_samp[r, 1 + j]); q_slot' = 1.
 * The KV rows kept are the pending token's and the accepted specs' (kv_keep =
 * a + 1 block rows from slot 0; every MASK row and rejected spec row, i.e.
 * cache_loc[r, kv_keep:], is freed); new_seq_lens = L + kv_keep.  The emitted
 * tokens are the accepted specs then the anchor (n_out = a + 1, -1 padding
 * to N); the anchor is the next round's pending token.  next_specs holds -1
 * and next_q_slot -1 when the next round is a cold start.  Any mode other
 * than 0 or 1 is a cold start with flag bit 6.
 * Flags as in oracle_spec_accept: bit 0 a tested ratio within 1e-6 of u, bit 1
 * a draw within 1e-9 * S of a boundary (any of the draws).
 */
void oracle_idlm_accept(const int32_t *block_ids, const int32_t *mode, const float *p,
                        int64_t p_stride_r, int64_t p_stride_i, const float *q_prev,
                        int64_t q_stride_r, int64_t q_stride_i, const int32_t *q_slot,
                        const float *u_acc, const float *u_samp, const int32_t *seq_lens, int bs,
                        int N, int V, int32_t *accept_len, int32_t *n_out, int32_t *out_tokens,
                        int32_t *next_mode, int32_t *next_pending, int32_t *next_specs,
                        int32_t *next_q_slot, int32_t *new_seq_lens, int32_t *kv_keep,
                        int32_t *flags, int nthreads) {
    const int blk = 2 * N - 1;
#ifdef _OPENMP
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel num_threads(nthreads)
#endif
    {
        float *w = (float *)malloc(sizeof(float) * (size_t)V);
#ifdef _OPENMP
#pragma omp for schedule(static)
#endif
        for (int r = 0; r < bs; ++r) {
            int flag = 0;
            const int32_t *ids = block_ids + (long)r * blk;
            const float *prow = p + (long)r * p_stride_r;
            int verify = mode[r] == 1;
            if (mode[r] != 0 && mode[r] != 1) flag |= 64;
            if (verify && (q_slot[r] < 0 || q_slot[r] > N)) {
                verify = 0;
                flag |= 32;
            }
            int a = 0, anchor, near = 0;
            int draw_specs;   /* slot of p holding spec'_0's distribution, or -1 */
            if (verify) {
                const float *qrow = q_prev + (long)r * q_stride_r + (long)q_slot[r] * q_stride_i;
                for (int k = 0; k < N - 1; ++k) {
                    int s = ids[1 + k];
                    if (s < 0 || s >= V) {
                        flag |= 8;
                        break;
                    }
                    float pv = prow[(long)k * p_stride_i + s];
                    float qv = qrow[(long)k * q_stride_i + s];
                    float u = u_acc[(long)r * (N - 1) + k];
                    int acc;
                    if (qv == 0.0f) {
                        acc = pv > 0.0f;
                    } else {
                        volatile float ratio = pv / qv; /* fp32, correctly rounded */
                        acc = u < fminf(1.0f, ratio);
                        if (fabs((double)ratio - (double)u) < 1e-6) flag |= 1;
                    }
                    if (!acc) break;
                    ++a;
                }
                if (a < N - 1) {
                    const float *pa = prow + (long)a * p_stride_i;
                    const float *qa = qrow + (long)a * q_stride_i;
                    double S = 0.0;
                    for (int k = 0; k < V; ++k) {
                        float d = pa[k] - qa[k];
                        w[k] = d > 0.0f ? d : 0.0f;
                        S += (double)w[k];
                    }
                    if (!(S > 0.0)) {
                        flag |= 4;
                        for (int k = 0; k < V; ++k) w[k] = pa[k];
                    }
                    anchor = inv_cdf_f32w(w, V, (double)u_samp[(long)r * N], &near);
                    draw_specs = -1;
                } else {
                    anchor = inv_cdf_f32w(prow + (long)(N - 1) * p_stride_i, V,
                                          (double)u_samp[(long)r * N], &near);
                    draw_specs = N;
                }
            } else {
                anchor = inv_cdf_f32w(prow, V, (double)u_samp[(long)r * N], &near);
                draw_specs = 1;
            }
            for (int j = 0; j < N - 1; ++j) {
                int32_t t = -1;
                if (draw_specs >= 0)
                    t = inv_cdf_f32w(prow + (long)(draw_specs + j) * p_stride_i, V,
                                     (double)u_samp[(long)r * N + 1 + j], &near);
                next_specs[(long)r * (N - 1) + j] = t;
            }
            if (near) flag |= 2;
            for (int i = 0; i < N; ++i) {
                int32_t v = -1;
                if (i < a) v = ids[1 + i];
                else if (i == a) v = anchor;
                out_tokens[(long)r * N + i] = v;
            }
            accept_len[r] = a;
            n_out[r] = a + 1;
            next_mode[r] = draw_specs >= 0 ? 1 : 0;
            next_pending[r] = anchor;
            next_q_slot[r] = draw_specs;
            kv_keep[r] = a + 1;
            new_seq_lens[r] = seq_lens[r] + a + 1;
            if (flags) flags[r] = flag;
        }
        free(w);
    }
}

/* ------------------------------------------------------------------------ */
/* KV materialisation of the committed prefix  [P3 2.2.6 (after verify, the
 * target hidden states of the committed prefix are written into the draft KV
 * cache at the verify step's cache locations); "From DFlash to dLLM
 * Self-Spec", DFlash engineering notes (KV injection is materialised right
 * before the draft forward: a batched linear projection across layers, then K
 * norm and RoPE, then the write into the KV pool)]
 *
 * Row (r, i) = r*B + i of `hidden` is committed when i < commit_len[r]
 * (commit_len clamped to [0, B]).  For every committed row x, draft layer l,
 * KV head h and d in [0, D):
 *   k[d] = sum_c W[l][0][h*D + d][c] * x[c]      (K projection)
 *   v[d] = sum_c W[l][1][h*D + d][c] * x[c]      (V projection)
 *   kn[d] = k[d] / sqrt(mean_d(k^2) + eps) * g[l][d]           (RMS K norm)
 *   for d < D/2, with c = cos_tab[pos][d], s = sin_tab[pos][d]:
 *     ko[d]       = kn[d] * c - kn[d + D/2] * s                 (RoPE, the
 *     ko[d + D/2] = kn[d + D/2] * c + kn[d] * s                  rotate-half pairing)
 * pos = positions[row].  Outputs, fp64: k_out / v_out [bs*B, L, Hkv, D] for the
 * committed rows; rows not written are left as they are.  status[row] = 1
 * for a written row, 0 for an uncommitted one, -1 for a committed row whose
 * cache_loc is outside [0, num_slots) or whose position is outside
 * [0, max_pos) (skipped).  Returns the number of such rows.
 */
int oracle_kv_materialize(const uint16_t *hidden, const int32_t *commit_len,
                          const int32_t *positions, const int32_t *cache_loc,
                          const uint16_t *w_kv, const uint16_t *k_norm_w, const float *cos_tab,
                          const float *sin_tab, int max_pos, double eps, int bs, int B, int H,
                          int n_layers, int Hkv, int D, int64_t num_slots, double *k_out,
                          double *v_out, int32_t *status, int nthreads) {
    const int half = D / 2;
    const long rows = (long)bs * B;
    int bad = 0;
    for (long row = 0; row < rows; ++row) {
        const int r = (int)(row / B), i = (int)(row % B);
        int cl = commit_len[r];
        if (cl < 0) cl = 0;
        if (cl > B) cl = B;
        if (i >= cl) {
            status[row] = 0;
            continue;
        }
        const int32_t loc = cache_loc[row], pos = positions[row];
        if (loc < 0 || (int64_t)loc >= num_slots || pos < 0 || pos >= max_pos) {
            status[row] = -1;
            ++bad;
            continue;
        }
        status[row] = 1;
    }
#ifdef _OPENMP
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel num_threads(nthreads)
#endif
    {
        double *x = (double *)malloc(sizeof(double) * (size_t)H);
        double *y = (double *)malloc(sizeof(double) * (size_t)D);
        double *kn = (double *)malloc(sizeof(double) * (size_t)D);
#ifdef _OPENMP
#pragma omp for schedule(dynamic)
#endif
        for (long row = 0; row < rows; ++row) {
            if (status[row] != 1) continue;
            for (int c = 0; c < H; ++c) x[c] = bf16_to_f64(hidden[row * H + c]);
            const int pos = positions[row];
            for (int l = 0; l < n_layers; ++l) {
                for (int kv = 0; kv < 2; ++kv) {
                    for (int h = 0; h < Hkv; ++h) {
                        for (int d = 0; d < D; ++d) {
                            const uint16_t *wr =
                                w_kv + ((((long)l * 2 + kv) * Hkv + h) * D + d) * (long)H;
                            double acc = 0.0;
                            for (int c = 0; c < H; ++c) acc += bf16_to_f64(wr[c]) * x[c];
                            y[d] = acc;
                        }
                        double *dst = (kv == 0 ? k_out : v_out) +
                                      (((row * n_layers + l) * Hkv + h) * (long)D);
                        if (kv == 1) {
                            for (int d = 0; d < D; ++d) dst[d] = y[d];
                            continue;
                        }
                        double ms = 0.0;
                        for (int d = 0; d < D; ++d) ms += y[d] * y[d];
                        ms /= (double)D;
                        const double inv = 1.0 / sqrt(ms + eps);
                        for (int d = 0; d < D; ++d)
                            kn[d] = y[d] * inv * bf16_to_f64(k_norm_w[(long)l * D + d]);
                        for (int d = 0; d < half; ++d) {
                            const double c = (double)cos_tab[(long)pos * half + d];
                            const double s = (double)sin_tab[(long)pos * half + d];
                            dst[d] = kn[d] * c - kn[d + half] * s;
                            dst[d + half] = kn[d + half] * c + kn[d] * s;
                        }
                    }
                }
            }
        }
        free(x);
        free(y);
        free(kn);
    }
    return bad;
}

/* ------------------------------------------------------------------------ */
/* Tree verify  ["Unlocking Lossless Speedups in LLMs via Discrete Diffusion",
 * Psi-Spec Tree sampler (per position the top-K tokens, the top-V prefixes by
 * log-probability kept, the tree verified in parallel with tree attention);
 * "SGLang dLLM / LLaDA 2.0", "Attention Mask" (the block's queries see the
 * whole context; inside the block the mask is set by the verify structure)]
 *
 * A request's block holds a token tree of B nodes in topological order: node 0
 * is the root (the verified token, parent -1), node i > 0 has a parent in
 * [0, i).  A parent outside that range makes the node a root of its own
 * (reported).  Node i sits at block slot i (cache position L + i) and at
 * sequence position L + depth(i).
 */
static int tree_parent(const int32_t *par, int i) {
    if (i <= 0) return -1;
    int p = par[i];
    return (p >= 0 && p < i) ? p : -1;
}

static int tree_is_ancestor(const int32_t *par, int j, int i) {  /* j == i counts */
    for (int k = i; k >= 0; k = tree_parent(par, k))
        if (k == j) return 1;
    return 0;
}

/* depth, positions L + depth, cache_loc of block slot i (as prepare_block),
 * and the ancestor-or-self set of node i as mask_words 64-bit words
 * (mask[(r * B + i) * mask_words + j / 64] has bit j % 64 set iff node j is
 * node i or one of its ancestors; mask_words >= ceil(B / 64), words past the
 * tree are 0).  Returns the number of invalid parents plus failed page
 * lookups, or -1 when mask_words is too small. */
int oracle_tree_prepare(const int32_t *parent, const int32_t *seq_lens,
                        const int32_t *block_table, int max_pages_per_req, int num_pages, int bs,
                        int B, int page_size, int32_t *depth, int32_t *positions,
                        int32_t *cache_loc, uint64_t *mask, int mask_words) {
    if (mask_words < (B + 63) / 64) return -1;
    int bad = 0;
    for (int r = 0; r < bs; ++r) {
        const int32_t *par = parent + (long)r * B;
        for (int i = 0; i < B; ++i) {
            const long row = (long)r * B + i;
            if (i == 0 ? par[0] != -1 : tree_parent(par, i) < 0) ++bad;
            uint64_t *m = mask + row * mask_words;
            for (int w = 0; w < mask_words; ++w) m[w] = 0;
            int d = -1;
            for (int k = i; k >= 0; k = tree_parent(par, k)) {
                ++d;
                m[k / 64] |= (uint64_t)1 << (k % 64);
            }
            depth[row] = d;
            const long L = seq_lens[r];
            positions[row] = (int32_t)(L + d);
            const long t = L + i;
            int32_t loc = -1;
            if (L >= 0 && t / page_size < max_pages_per_req) {
                int32_t page = block_table[(long)r * max_pages_per_req + t / page_size];
                if (page >= 0 && page < num_pages) loc = (int32_t)((long)page * page_size + t % page_size);
            }
            if (loc < 0) ++bad;
            cache_loc[row] = loc;
        }
    }
    return bad;
}

/* Tree attention: as oracle_block_attn, with the intra-block mask "block key
 * j is visible to block row i iff j is i or an ancestor of i". */
int oracle_block_attn_tree(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                           const int32_t *block_table, int max_pages_per_req, int num_pages,
                           const int32_t *seq_lens, const int32_t *parent, int bs, int B, int Hq,
                           int Hkv, int D, int page_size, double scale, double *out,
                           double *lse, int nthreads) {
    long max_keys = 0;
    for (int r = 0; r < bs; ++r)
        if ((long)seq_lens[r] + B > max_keys) max_keys = (long)seq_lens[r] + B;
    int bad = 0;
    const long units = (long)bs * Hq;
    const int G = Hq / Hkv;
#ifdef _OPENMP
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel num_threads(nthreads) reduction(+ : bad)
#endif
    {
        double *scores = (double *)malloc(sizeof(double) * (size_t)(max_keys > 0 ? max_keys : 1));
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (long u = 0; u < units; ++u) {
            const int r = (int)(u / Hq), j = (int)(u % Hq), h = j / G;
            const int32_t *par = parent + (long)r * B;
            const long L = seq_lens[r];
            for (int i = 0; i < B; ++i) {
                const long row = ((long)r * B + i) * Hq + j;
                const uint16_t *qrow = q + row * D;
                double smax = -INFINITY;
                int rc = 0;
                for (long t = 0; t < L + B; ++t) {
                    scores[t] = -INFINITY;
                    if (!(t < L || tree_is_ancestor(par, (int)(t - L), i))) continue;
                    const long page_idx = t / page_size;
                    int32_t page = page_idx < max_pages_per_req
                                       ? block_table[(long)r * max_pages_per_req + page_idx]
                                       : -1;
                    if (page < 0 || page >= num_pages) {
                        rc = -1;
                        break;
                    }
                    const uint16_t *krow = k_cache + (((long)page * page_size + t % page_size) * Hkv + h) * D;
                    double dot = 0.0;
                    for (int d = 0; d < D; ++d) dot += bf16_to_f64(qrow[d]) * bf16_to_f64(krow[d]);
                    scores[t] = scale * dot;
                    if (scores[t] > smax) smax = scores[t];
                }
                double *o = out + row * D;
                if (rc != 0) {
                    ++bad;
                    for (int d = 0; d < D; ++d) o[d] = NAN;
                    if (lse) lse[row] = NAN;
                    continue;
                }
                double denom = 0.0;
                for (long t = 0; t < L + B; ++t)
                    if (scores[t] != -INFINITY) denom += exp(scores[t] - smax);
                for (int d = 0; d < D; ++d) o[d] = 0.0;
                for (long t = 0; t < L + B; ++t) {
                    if (scores[t] == -INFINITY) continue;
                    const double w = exp(scores[t] - smax) / denom;
                    const int32_t page = block_table[(long)r * max_pages_per_req + t / page_size];
                    const uint16_t *vrow = v_cache + (((long)page * page_size + t % page_size) * Hkv + h) * D;
                    for (int d = 0; d < D; ++d) o[d] += w * bf16_to_f64(vrow[d]);
                }
                if (lse) lse[row] = smax + log(denom);
            }
        }
        free(scores);
    }
    return bad;
}

/* Tree acceptance.  p[r, n] (strides in elements) is the verifier's
 * distribution after node n, i.e. for n's children.  Walk from the root: at
 * node n of depth d draw x = InvCDF(p[r, n], u[r, d]) (stochastic) or x =
 * argmax p[r, n] (greedy, u == NULL; lowest index on ties); if a child of n
 * carries token x (the lowest-index such child) it is accepted and the walk
 * goes on from it, else x is emitted (the correction, or the bonus when n is a
 * leaf) and the walk ends.  With deterministic drafts (the tree's tokens are
 * chosen, not sampled) this is rejection sampling with one-hot draft
 * distributions: the emitted sequence follows the verifier exactly.
 * Outputs: accept_len = accepted nodes below the root; path[r] = node indices
 * root, accepted nodes, -1 padding; out_tokens[r] = accepted tokens then x,
 * -1 padding; bonus_id = x; new_seq_lens = L + accept_len + 1.
 * flags: bit 1 a draw within 1e-9 * S of a boundary of its token, bit 4 an
 * argmax tie (greedy). */
void oracle_tree_accept(const int32_t *block_ids, const int32_t *parent, const float *p,
                        int64_t p_stride_r, int64_t p_stride_n, const float *u,
                        const int32_t *seq_lens, int bs, int B, int V, int32_t *accept_len,
                        int32_t *path, int32_t *out_tokens, int32_t *bonus_id,
                        int32_t *new_seq_lens, int32_t *flags, int nthreads) {
#ifdef _OPENMP
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for num_threads(nthreads) schedule(static)
#endif
    for (int r = 0; r < bs; ++r) {
        const int32_t *ids = block_ids + (long)r * B;
        const int32_t *par = parent + (long)r * B;
        int flag = 0, n = 0, depth = 0, x = -1;
        for (int i = 0; i < B; ++i) {
            path[(long)r * B + i] = -1;
            out_tokens[(long)r * B + i] = -1;
        }
        path[(long)r * B] = 0;
        for (;;) {
            const float *pn = p + (long)r * p_stride_r + (long)n * p_stride_n;
            if (u != NULL) {
                int near = 0;
                x = inv_cdf_f32w(pn, V, (double)u[(long)r * B + depth], &near);
                if (near) flag |= 2;
            } else {
                int tie = 0;
                x = argmax_lowest(pn, V, &tie);
                if (tie) flag |= 16;
            }
            int child = -1;
            for (int c = n + 1; c < B; ++c)
                if (tree_parent(par, c) == n && ids[c] == x) {
                    child = c;
                    break;
                }
            out_tokens[(long)r * B + depth] = x;
            if (child < 0) break;
            ++depth;
            path[(long)r * B + depth] = child;
            n = child;
        }
        accept_len[r] = depth;
        bonus_id[r] = x;
        new_seq_lens[r] = seq_lens[r] + depth + 1;
        if (flags) flags[r] = flag;
    }
}

/* Exposed for tests of the sampling rule itself. */
int oracle_inv_cdf(const float *w, int V, double u, int32_t *flag_near) {
    int near = 0;
    int k = inv_cdf_f32w(w, V, u, &near);
    if (flag_near) *flag_near = near;
    return k;
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
