/*
 * bdsa.h -- C ABI of libbdsa.so: one draft/verify step of block-diffusion
 * self-speculative decoding over a paged KV cache, for NVIDIA GB300 (sm_103a).
 *
 * The step, in call order:
 *   bdsa_prepare_block     lay out each request's block (token ids, positions,
 *                          cache slots);
 *   bdsa_block_attn_paged  block attention of the B block queries over the
 *                          committed context plus the block itself, with a
 *                          bidirectional (draft) or token-causal (verify)
 *                          intra-block mask;
 *   bdsa_spec_accept       lossless speculative acceptance: longest accepted
 *                          prefix, then a residual correction or bonus token.
 *
 * Conventions for every call
 *   - All tensor pointers are DEVICE pointers owned by the caller.  The library
 *     allocates nothing: scratch comes from a caller-provided workspace sized by
 *     the matching *_workspace_bytes query.
 *   - Calls are asynchronous on `stream` (a cudaStream_t passed as void*; NULL
 *     is the legacy default stream) and never synchronise the device.
 *   - Tensors are dense row-major with the shapes given; int32 indices.
 *   - Host-side argument checks return a status synchronously and launch
 *     nothing.  Data errors that only the device can see (a page id outside the
 *     pool, a draft id outside the vocabulary, ...) are reported through the
 *     optional `dev_status` int32 device word: the first error code is stored
 *     with an atomic compare-and-swap from 0, the affected unit of work is
 *     skipped (its outputs are zero / -1), and the kernel never traps.  Callers
 *     zero *dev_status before the step and read it whenever convenient.
 *   - Bounded waits: every spin inside a kernel has a time limit; on expiry the
 *     kernel stores BDSA_DEVICE_TIMEOUT in dev_status and returns.
 *
 * Notation: bs requests, block size B, Hq query heads, Hkv KV heads, G = Hq/Hkv
 * (query head j reads KV head j / G), head dim D, page size ps, L_r = committed
 * context length of request r (keys already in the cache before the block),
 * V vocabulary size.
 */
#ifndef BDSA_H_
#define BDSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum bdsa_status {
    BDSA_OK = 0,
    BDSA_INVALID_ARG = 1,          /* null pointer, negative size, bad mode, ... */
    BDSA_UNSUPPORTED = 2,          /* a valid request this build does not handle (D, B, G*B) */
    BDSA_MISALIGNED = 3,           /* a pointer or stride breaks the alignment rules below */
    BDSA_WORKSPACE_TOO_SMALL = 4,
    BDSA_CUDA_ERROR = 5,           /* a CUDA runtime/driver call or launch failed */
    /* codes written to *dev_status by kernels */
    BDSA_DEVICE_OUT_OF_RANGE = 16, /* page id / slot / position / token id out of range */
    BDSA_DEVICE_TIMEOUT = 17       /* a bounded wait expired; outputs of that unit undefined */
} bdsa_status;

typedef struct bdsa_bf16 { uint16_t bits; } bdsa_bf16; /* IEEE bfloat16 storage */

enum { BDSA_MODE_DRAFT = 0, BDSA_MODE_VERIFY = 1, BDSA_MODE_TREE = 2 /* bdsa_block_attn_paged_tree */ };

/* Largest token tree (nodes per request) of the tree-verify calls: the
 * Psi-Spec Tree sampler's (B, K, V) = (16, 32, 32) keeps at most 32 prefixes
 * of 15 drafted tokens below the root, 481 nodes. */
enum { BDSA_TREE_MAX_NODES = 512 };

/* Human-readable name of a status code (static string, never NULL). */
const char *bdsa_status_string(int32_t status);

/* Library version as "major.minor.patch" (static string). */
const char *bdsa_version(void);

/* ------------------------------------------------------------------------ */
/* bdsa_prepare_block
 *
 * "From DFlash to dLLM Self-Spec (II): SGLang Spec V2", section 2.2.2 (the
 * block starts with the last verified token, the other slots are mask tokens;
 * positions and cache locations are prepared in the same kernel); "... (IV)",
 * section 4.4.1 (LinearSpec block init); section 2.3.5 of (II) (the caller has
 * reserved pages for at least L_r + B tokens).
 *
 * For r in [0, bs), i in [0, B):
 *   block_ids[r,i] = i == 0 ? verified_id[r] : mask_token_id
 *   positions[r,i] = L_r + i
 *   cache_loc[r,i] = block_table[r, (L_r+i)/ps] * ps + (L_r+i) % ps
 *
 * verified_id [bs], seq_lens [bs] (= L_r), block_table [bs, max_pages_per_req]
 * (page ids in [0, num_pages)); outputs block_ids / positions / cache_loc
 * [bs, B].  A lookup outside the table or the pool sets cache_loc = -1 and
 * dev_status = BDSA_DEVICE_OUT_OF_RANGE.  One launch.
 */
int32_t bdsa_prepare_block(const int32_t *verified_id, const int32_t *seq_lens,
                           const int32_t *block_table, int32_t max_pages_per_req,
                           int32_t num_pages, int32_t bs, int32_t B, int32_t page_size,
                           int32_t mask_token_id, int32_t *block_ids, int32_t *positions,
                           int32_t *cache_loc, int32_t *dev_status, void *stream);

/* ------------------------------------------------------------------------ */
/* bdsa_block_attn_paged
 *
 * "SGLang dLLM / LLaDA 2.0", section "Attention Mask": the block's queries see
 * the whole cached context (as in chunked prefill) and, inside the block, a
 * rectangle (block diffusion, DRAFT) or a token-causal trapezoid (chunked
 * prefill, VERIFY).  "From DFlash to dLLM Self-Spec (IV)", section 4.4.1: the
 * draft pass uses the bidirectional view, the verify pass the causal view over
 * the past KV; "... (II)", sections 2.2.3-2.2.4: both passes run a fixed block
 * of B tokens per request.
 *
 * For request r, block row i, query head j (KV head h = j / G):
 *   o[r*B+i, j] = sum_t softmax_t(scale * <q[r*B+i, j], k[t, h]>) v[t, h]
 *   over keys t in [0, L_r + B) with
 *   allowed(i, t) = t < L_r  or  mode == DRAFT  or  t - L_r <= i.
 * Key t of request r is cache slot block_table[r, t/ps] * ps + t % ps; the
 * block's own K/V (positions L_r..L_r+B-1) must already be in the cache.
 *
 * q        [bs*B, Hq, D] bf16 (post-RoPE)
 * k_cache, v_cache  [num_pages*ps, Hkv, D] bf16
 * out      [bs*B, Hq, D] bf16
 * lse      [bs*B, Hq] fp32 natural-log sum-exp of the scaled scores, or NULL
 * max_ctx_len  host-side upper bound on every L_r (the scheduler's planning
 *          length); checked to be >= 0.  The device-side schedule below reads
 *          the actual seq_lens and does not depend on it.
 * num_sms  number of persistent CTAs (0: the current device's SM count).
 * Schedule: one persistent CTA per SM takes an equal share of the concatenated
 * (request, KV head, 128-key tile) sequence, which each CTA derives from
 * seq_lens itself; a (request, KV head) unit cut between CTAs leaves partials.
 * With num_sms at most the device's SM count (every CTA resident at once) the
 * CTA holding a cut unit's first tile waits, boundedly, for the unit's other
 * partials and merges them: one launch per call.  With more CTAs than SMs a
 * second kernel merges them: two launches, chained with programmatic
 * dependent launch (no CTA of the first waits for another).
 * Pages: a request with L_r < 0, with L_r + B needing more pages than
 * max_pages_per_req, or with a page id it references (pages 0 ..
 * ceil((L_r+B)/ps) - 1 of its row) outside [0, num_pages) gets out = 0 and
 * lse = -inf on all its rows, and dev_status = BDSA_DEVICE_OUT_OF_RANGE.
 * softmax_scale must be finite and > 0.
 * Arithmetic: bf16 products, fp32 accumulation and softmax; P is rounded to
 * bf16 for the PV product.
 * Supported: D in {64, 128}; 1 <= B <= 64; G*B <= 128; page_size a power of two
 * >= 8; q, k_cache, v_cache, out 16-byte aligned.
 * Workspace: at least bdsa_block_attn_workspace_bytes(...) bytes of device
 * memory, 256-byte aligned: two partial slots per CTA (a flag, a 64-bit ready
 * word and G*B*(D+1) fp32 values).  Its contents need no initialisation and
 * are not meaningful after the call (each call stamps the slots it writes with
 * a ticket of its own; a call captured into a CUDA graph does not rely on
 * them); calls that share one workspace must be ordered on the same stream.
 */
size_t bdsa_block_attn_workspace_bytes(int32_t bs, int32_t B, int32_t Hq, int32_t Hkv, int32_t D,
                                       int32_t max_ctx_len, int32_t num_sms);

int32_t bdsa_block_attn_paged(const bdsa_bf16 *q, const bdsa_bf16 *k_cache,
                              const bdsa_bf16 *v_cache, const int32_t *block_table,
                              int32_t max_pages_per_req, int32_t num_pages,
                              const int32_t *seq_lens, int32_t max_ctx_len, int32_t bs,
                              int32_t B, int32_t Hq, int32_t Hkv, int32_t D, int32_t page_size,
                              float softmax_scale, int32_t mode, bdsa_bf16 *out, float *lse,
                              void *workspace, size_t workspace_bytes, int32_t num_sms,
                              int32_t *dev_status, void *stream);

/* ------------------------------------------------------------------------ */
/* bdsa_block_attn_paged_append
 *
 * "From DFlash to dLLM Self-Spec (II)", section 2.2.2 (the prepare step builds
 * the block's positions and the cache locations its K/V go to) and section
 * 2.2.4 (the verify forward over the block): the block's own keys and values
 * are written into the paged cache in the same launch as the block attention
 * that reads them, instead of by a separate write before it.
 *
 * k_new, v_new  [bs*B, Hkv, D] bf16: the block's keys (post-RoPE) and values,
 *          row r*B + i for position L_r + i.
 * For every r, i < B and KV head h:
 *   k_cache[slot, h, :] = k_new[r*B + i, h, :] and likewise v, with
 *   slot = block_table[r, (L_r+i)/ps] * ps + (L_r+i) % ps (the slot
 *   bdsa_prepare_block's cache_loc names); then the attention is exactly
 *   that of bdsa_block_attn_paged on the updated caches.
 * A position whose page is past max_pages_per_req or outside [0, num_pages) is
 * not written (the request's output is zeros as in bdsa_block_attn_paged);
 * nothing else in the caches changes.  Each new row is written by the CTA
 * whose share of the schedule holds it (by a warp of its own, before that
 * tile's load), so it is read back from the cache in the same launch.  No
 * other work may read or write the block's cache slots during the call.
 * Everything else (arguments, schedule, workspace, launches, errors) is as in
 * bdsa_block_attn_paged; k_new and v_new must be 16-byte aligned.
 */
int32_t bdsa_block_attn_paged_append(const bdsa_bf16 *q, const bdsa_bf16 *k_new,
                                     const bdsa_bf16 *v_new, bdsa_bf16 *k_cache,
                                     bdsa_bf16 *v_cache, const int32_t *block_table,
                                     int32_t max_pages_per_req, int32_t num_pages,
                                     const int32_t *seq_lens, int32_t max_ctx_len, int32_t bs,
                                     int32_t B, int32_t Hq, int32_t Hkv, int32_t D,
                                     int32_t page_size, float softmax_scale, int32_t mode,
                                     bdsa_bf16 *out, float *lse, void *workspace,
                                     size_t workspace_bytes, int32_t num_sms, int32_t *dev_status,
                                     void *stream);

/* ------------------------------------------------------------------------ */
/* bdsa_spec_accept
 *
 * "From DFlash to dLLM Self-Spec (IV)", section 4.3.1: a draft token is
 * accepted with probability min(1, p/q), and a rejection is corrected from the
 * verifier; "Unlocking Lossless Speedups in LLMs via Discrete Diffusion",
 * background on speculative decoding (keep the longest accepted prefix,
 * resample the first rejected position from the residual distribution; the
 * output distribution equals the verifier's) and the Psi-Spec step (the first
 * token is always accepted); "From DFlash to dLLM Self-Spec (II)", section
 * 2.2.5 (greedy rule: accept while the draft equals the verifier argmax, bonus
 * = verifier argmax at the first mismatch, commit_len = accept_len + 1, one
 * kernel emits accept_len, commit_lens, bonus ids, out tokens, new seq lens).
 *
 * Row r: block_ids[r] = [verified, d_1, ..., d_{B-1}].  p[r,i] is the verifier
 * distribution for block slot i+1 (p[r,B-1] is the bonus distribution); q[r,i-1]
 * is the draft distribution d_i was drawn from.  Element (r, i, k) of p is at
 * p[r*p_stride_r + i*p_stride_i + k] (likewise q); stride 0 broadcasts.
 *
 * Stochastic mode (q != NULL):
 *   a = number of leading i in 1..B-1 with u_acc[r,i-1] < min(1, p/q), where
 *       p/q = p[r,i-1][d_i] / q[r,i-1][d_i] is an IEEE fp32 divide (q == 0:
 *       accepted iff p > 0);
 *   a <  B-1: token = InvCDF(max(0, p[r,a] - q[r,a]), u_samp[r]) (fp32 weights;
 *             if they are all 0, InvCDF(p[r,a], u_samp[r]));
 *   a == B-1: token = InvCDF(p[r,B-1], u_samp[r]).
 * Greedy mode (q == NULL): a = number of leading i with d_i == argmax p[r,i-1]
 *   (lowest index on ties); token = argmax p[r,a].  u_acc / u_samp are unused.
 * InvCDF(w, u) = smallest k with C_k > u*S, C_k the cumulative weight in index
 *   order, S the total.  The kernel adds the fp32 weights with error-free
 *   transformations (TwoSum) and carries the running sums and S as
 *   float-float pairs (hi + lo, about 48 significant bits, all in fp32
 *   arithmetic); u*S is formed and compared as a float-float product too.  The
 *   sums are within ~1e-12*S of the exact ones, so the draw is the
 *   exact-arithmetic one unless u*S lies within that distance of a boundary.
 * Outputs: accept_len[r] = a, commit_len[r] = a+1,
 *   out_tokens[r] = [d_1..d_a, token, -1...] ([bs, B]), bonus_id[r] = token,
 *   new_seq_lens[r] = seq_lens[r] + a + 1.
 * p, q: fp32; u_acc [bs, B-1], u_samp [bs] fp32 in [0, 1); 1 <= B <= 64; 1 <= V.
 * With B = 1 there is no draft to test: q is never read but must still be a
 * non-null pointer to select the stochastic rule (the bonus is then sampled).
 * A draft id outside [0, V) counts as a rejection and sets dev_status.
 * Workspace: bdsa_spec_accept_workspace_bytes(...) bytes, 256-byte aligned.
 *   It is 0 for V <= 2^21: a row's partial sums then stay in the shared memory
 *   of the thread-block cluster that handles the row, and `workspace` may be
 *   NULL.  Larger vocabularies need global scratch (per-row float-float
 *   segment totals and a counter that each call clears with a memset).
 * Launches: one kernel (plus that memset above V = 2^21).
 */
size_t bdsa_spec_accept_workspace_bytes(int32_t bs, int32_t B, int32_t V, int32_t num_sms);

int32_t bdsa_spec_accept(const int32_t *block_ids, const float *p, int64_t p_stride_r,
                         int64_t p_stride_i, const float *q, int64_t q_stride_r,
                         int64_t q_stride_i, const float *u_acc, const float *u_samp,
                         const int32_t *seq_lens, int32_t bs, int32_t B, int32_t V,
                         int32_t *accept_len, int32_t *commit_len, int32_t *out_tokens,
                         int32_t *bonus_id, int32_t *new_seq_lens, void *workspace,
                         size_t workspace_bytes, int32_t num_sms, int32_t *dev_status,
                         void *stream);

/* ------------------------------------------------------------------------ */
/* bdsa_spec_accept_noalloc -- no counterpart on the source pages.
 *
 * The acceptance step of bdsa_spec_accept (same inputs, outputs, rules and
 * results) for callers that cannot give this library device memory for
 * scratch: a serving loop whose device memory is planned once at start-up and
 * may not grow afterwards, or a framework that owns the device allocator and
 * passes only the step's own tensors.  Instead of a workspace it uses a fixed
 * 8 MiB array in the library's device image (present on every GPU that loads
 * the library, and held there until the process exits).
 *   - Nothing is allocated: no cudaMalloc / cudaFree or allocating call.
 *   - Set-up: the first call on each device looks up the array's device
 *     address (cudaGetSymbolAddress, with that device current) and keeps it
 *     for the life of the process; make that first call before any stream
 *     capture.  A cudaDeviceReset later in the process is not supported.
 *   - All calls on a device share the array, and it keeps the last call's
 *     contents.  Calls whose kernels may overlap on the GPU (unordered
 *     streams) race on it; order them on one stream.  Problems with
 *     V <= 2^21 need no scratch: their kernels do not read or write the
 *     array.  Above that, each call clears the per-row counters it needs to
 *     zero (an asynchronous memset on `stream`) before its kernel runs; every
 *     other value it reads there is written earlier by the same call.
 *   - Argument errors are reported exactly as by bdsa_spec_accept.  Then it
 *     returns BDSA_WORKSPACE_TOO_SMALL, launching nothing, when the problem
 *     needs more than 8 MiB of scratch, i.e. when
 *     bdsa_spec_accept_workspace_bytes(bs, B, V, num_sms) > 8 MiB (for
 *     example 128 rows at V = 2^22).
 */
int32_t bdsa_spec_accept_noalloc(const int32_t *block_ids, const float *p, int64_t p_stride_r,
                                 int64_t p_stride_i, const float *q, int64_t q_stride_r,
                                 int64_t q_stride_i, const float *u_acc, const float *u_samp,
                                 const int32_t *seq_lens, int32_t bs, int32_t B, int32_t V,
                                 int32_t *accept_len, int32_t *commit_len, int32_t *out_tokens,
                                 int32_t *bonus_id, int32_t *new_seq_lens, int32_t num_sms,
                                 int32_t *dev_status, void *stream);

/* ------------------------------------------------------------------------ */
/* bdsa_idlm_prepare
 *
 * "From DFlash to dLLM Self-Spec (IV)", section 4.3.1: an I-DLM Block-N
 * round lays out blk = 2N-1 slots per request, [pending, spec_0 .. spec_{N-2},
 * M .. M] when it verifies the specs carried from the previous round (mode 1)
 * and [pending, M .. M] on a cold start (any other mode).
 *
 * pending [bs], mode [bs], specs [bs, N-1] (read only in mode 1; may be NULL
 * when N == 1), seq_lens [bs] (L_r, the committed length; the pending token's
 * KV is not yet in the cache), block_table [bs, max_pages_per_req].
 * Outputs [bs, blk]: block_ids as above, positions L_r + j, cache_loc exactly
 * as bdsa_prepare_block computes it for a block of blk slots (-1 and
 * *dev_status = BDSA_DEVICE_OUT_OF_RANGE where the page lookup fails).
 * Host checks: bs >= 0, 1 <= N, bs * blk <= INT32_MAX, page_size >= 1,
 * max_pages_per_req >= 1, num_pages >= 1, non-null buffers.  One launch.
 */
int32_t bdsa_idlm_prepare(const int32_t *pending, const int32_t *specs, const int32_t *mode,
                          const int32_t *seq_lens, const int32_t *block_table,
                          int32_t max_pages_per_req, int32_t num_pages, int32_t bs, int32_t N,
                          int32_t page_size, int32_t mask_token_id, int32_t *block_ids,
                          int32_t *positions, int32_t *cache_loc, int32_t *dev_status,
                          void *stream);

/* ------------------------------------------------------------------------ */
/* bdsa_idlm_accept
 *
 * "From DFlash to dLLM Self-Spec (IV)", sections 4.3 and 4.3.1 (the specs
 * drawn from MASK slots in one round are verified in the next against the
 * causal view with min(1, p/q), a rejection is corrected from the anchor
 * distribution and falls back to a cold start, the same forward drafts the
 * next specs) and 4.6 (which KV rows to free, how far the request advances).
 *
 * p [bs, 2N-1, V] fp32: p[r, j] (at p + r*p_stride_r + j*p_stride_i) is the
 *   distribution predicted at slot j, i.e. for slot j + 1's token.
 * q_prev: the previous round's p rows; spec_k of row r was drawn from
 *   q_prev[r, q_slot[r] + k] (at q_prev + r*q_stride_r + (q_slot[r]+k)*q_stride_i).
 * block_ids [bs, 2N-1] as written by bdsa_idlm_prepare; mode [bs];
 * u_acc [bs, N-1], u_samp [bs, N] fp32 uniforms in [0, 1); seq_lens [bs].
 * Row r, verify (mode 1 with 0 <= q_slot <= N):
 *   a = leading k with u_acc[r,k] < min(1, p[k][s_k] / q_prev[q_slot+k][s_k])
 *       (IEEE fp32 divide; q == 0 accepts iff p > 0; an id outside [0, V)
 *       rejects and sets *dev_status = BDSA_DEVICE_OUT_OF_RANGE);
 *   a < N-1: anchor = InvCDF(max(0, p[a] - q_prev[q_slot+a]), u_samp[r,0])
 *            (from p[a] if those weights are all 0); next round: cold start;
 *   a = N-1: anchor = InvCDF(p[N-1], u_samp[r,0]) (bonus); new specs
 *            next_specs[r,j] = InvCDF(p[N+j], u_samp[r,1+j]); next_q_slot = N.
 * Row r, cold start (mode 0; mode 1 with q_slot outside [0, N] and any other
 *   mode too, with *dev_status = BDSA_DEVICE_OUT_OF_RANGE): a = 0, anchor =
 *   InvCDF(p[0], u_samp[r,0]), next_specs[r,j] = InvCDF(p[1+j], u_samp[r,1+j]),
 *   next_q_slot = 1.
 * InvCDF(w, u) = smallest k with sum_{i<=k} w_i > u * sum_i w_i.
 * Outputs: accept_len = a; n_out = a + 1; out_tokens [bs, N] = s_0..s_{a-1},
 *   anchor, -1 padding; next_pending = anchor; next_mode = 1 if specs were
 *   drawn else 0; next_specs [bs, N-1] (-1 when not drawn; may be NULL when
 *   N == 1); next_q_slot (-1 when not drawn); kv_keep = a + 1, the block rows
 *   from slot 0 whose KV stays (cache_loc[r, kv_keep:] are freed: every MASK
 *   row and every rejected spec); new_seq_lens = seq_lens + kv_keep.
 * Limits: 1 <= N <= 32, V <= 2^21 (BDSA_UNSUPPORTED above).  No workspace.
 * Host checks: bs >= 0, V >= 1, non-negative strides, non-null buffers
 *   (q_prev, u_acc and next_specs may be NULL only when N == 1), p and q_prev
 *   4-byte aligned.  All buffers are device memory owned by the caller.
 * num_sms: SM count the vocabulary chunking is sized for (0: the current
 *   device's).  dev_status (nullable) receives BDSA_DEVICE_OUT_OF_RANGE by
 *   atomicCAS from 0 on the data errors above; the kernel never traps.
 * Launch: one kernel of bs * N thread-block clusters (one per row and draw),
 * each cluster = that draw's vocabulary chunks; draws that the row does not
 * need exit at once.  Asynchronous on `stream`.
 */
int32_t bdsa_idlm_accept(const int32_t *block_ids, const int32_t *mode, const float *p,
                         int64_t p_stride_r, int64_t p_stride_i, const float *q_prev,
                         int64_t q_stride_r, int64_t q_stride_i, const int32_t *q_slot,
                         const float *u_acc, const float *u_samp, const int32_t *seq_lens,
                         int32_t bs, int32_t N, int32_t V, int32_t *accept_len, int32_t *n_out,
                         int32_t *out_tokens, int32_t *next_mode, int32_t *next_pending,
                         int32_t *next_specs, int32_t *next_q_slot, int32_t *new_seq_lens,
                         int32_t *kv_keep, int32_t num_sms, int32_t *dev_status, void *stream);

/* ------------------------------------------------------------------------ */
/* bdsa_kv_materialize
 *
 * "From DFlash to dLLM Self-Spec (II): SGLang Spec V2", section 2.2.6: after
 * verify, the target hidden states of each request's committed prefix are
 * written into the draft model's KV cache at the verify step's cache
 * locations (DFlash KV injection); the DFlash engineering notes of "From
 * DFlash to dLLM Self-Spec": this is materialised right before the draft
 * forward as one batched linear projection across the draft layers followed
 * by K norm and RoPE, then the write into the KV pool.
 *
 * Row (r, i) = r*B + i of `hidden` is committed when i < commit_len[r]
 * (clamped to [0, B]).  For every committed row x, layer l, KV head h, d < D:
 *   k[d] = sum_c w_kv[l][0][h*D + d][c] x[c],  v[d] = sum_c w_kv[l][1][h*D + d][c] x[c]
 *   kn[d] = k[d] / sqrt(mean_d k^2 + rms_eps) * k_norm_w[l][d]
 *   for d < D/2, c = rope_cos[pos][d], s = rope_sin[pos][d], pos = positions[row]:
 *     k_cache[l][slot][h][d]       = kn[d] c - kn[d + D/2] s
 *     k_cache[l][slot][h][d + D/2] = kn[d + D/2] c + kn[d] s
 *   v_cache[l][slot][h][d] = v[d], slot = cache_loc[row].
 * Uncommitted rows write nothing.  A committed row whose slot is outside
 * [0, num_slots) or whose position is outside [0, max_pos) writes nothing and
 * sets *dev_status = BDSA_DEVICE_OUT_OF_RANGE.
 *
 * hidden      [bs*B, H] bf16, 16-byte aligned
 * commit_len  [bs] int32 (e.g. bdsa_spec_accept's commit_len)
 * positions, cache_loc  [bs*B] int32 (e.g. bdsa_prepare_block's outputs)
 * w_kv        [n_layers, 2, Hkv*D, H] bf16 (per layer: the K projection's
 *             rows, then the V projection's; row-major like a linear layer's
 *             weight), 16-byte aligned
 * k_norm_w    [n_layers, D] bf16
 * rope_cos, rope_sin  [max_pos, D/2] fp32: the rotary table (angle of pair d
 *             at position p)
 * k_cache, v_cache  [n_layers, num_slots, Hkv, D] bf16, 16-byte aligned
 * Arithmetic: bf16 products with fp32 accumulation on the tensor cores; norm
 * and rotation in fp32; one rounding to bf16 at the store.
 * Supported: D == 128, H a multiple of 128, bs*B <= 2^24.
 * Workspace: bdsa_kv_materialize_workspace_bytes(bs, B, H) bytes, 256-byte
 * aligned (the gathered rows: a count, (slot, position) per row and a dense
 * copy of each committed hidden row); no initialisation needed.
 * Launches: a gather kernel (four CTAs per request) and a projection kernel of
 * n_layers * 2 * Hkv thread-block clusters of 3 CTAs (the three split the
 * hidden dimension), chained with programmatic dependent launch.
 */
size_t bdsa_kv_materialize_workspace_bytes(int32_t bs, int32_t B, int32_t H);
int32_t bdsa_kv_materialize(const bdsa_bf16 *hidden, const int32_t *commit_len,
                            const int32_t *positions, const int32_t *cache_loc, int32_t bs,
                            int32_t B, int32_t H, const bdsa_bf16 *w_kv,
                            const bdsa_bf16 *k_norm_w, int32_t n_layers, int32_t Hkv, int32_t D,
                            const float *rope_cos, const float *rope_sin, int32_t max_pos,
                            float rms_eps, bdsa_bf16 *k_cache, bdsa_bf16 *v_cache,
                            int64_t num_slots, void *workspace, size_t workspace_bytes,
                            int32_t *dev_status, void *stream);

/* ------------------------------------------------------------------------ */
/* Tree verify
 *
 * "Unlocking Lossless Speedups in LLMs via Discrete Diffusion", the Psi-Spec
 * Tree sampler: a token tree drafted by keeping the top candidates per
 * position is verified in one forward with tree attention, and rejection
 * sampling keeps the verifier's output distribution; "SGLang dLLM / LLaDA
 * 2.0", section "Attention Mask": the block's queries see the whole context,
 * the intra-block mask follows the verify structure.
 *
 * A request's block holds a token tree of B <= BDSA_TREE_MAX_NODES nodes in
 * topological order: parent [bs, B] int32, node 0 the root (the last verified
 * token, parent -1), node i > 0 with a parent in [0, i).  A parent outside
 * that range makes the node a root of its own and sets
 * *dev_status = BDSA_DEVICE_OUT_OF_RANGE.
 *
 * bdsa_tree_prepare: node i sits at block slot i (cache_loc of position
 *   L_r + i, as bdsa_prepare_block computes it, -1 and OUT_OF_RANGE when the
 *   lookup fails) and at sequence position L_r + depth(i) (positions, for
 *   RoPE).  tree_mask [bs, B, W] uint64 (W = ceil(B / 64), 8-byte aligned)
 *   holds node i's ancestor-or-self set: bit j % 64 of word j / 64 of
 *   tree_mask[r, i] is set iff node j is node i or one of its ancestors (bits
 *   j >= B are 0).  Other outputs [bs, B].  One launch.
 *
 * bdsa_block_attn_paged_tree: bdsa_block_attn_paged with the intra-block mask
 *   "block key j is visible to block row i iff bit j of tree_mask[r, i] is
 *   set" (mode BDSA_MODE_TREE, tree_mask as bdsa_tree_prepare writes it);
 *   layouts, workspace, errors as bdsa_block_attn_paged.  Limits: B <=
 *   BDSA_TREE_MAX_NODES and G = Hq / Hkv <= 128.  A request's G * B query rows
 *   of one KV head are processed in 128-row tiles of floor(128 / G) whole
 *   nodes (one tile of G * B rows when G * B <= 128), each over the context
 *   and the block keys up to its last node; the workspace holds partials of
 *   those tiles.  With 128-row tiles the cut units are merged by a second
 *   launch (two launches per call); with a 64-row tile (G * B <= 64) as in
 *   bdsa_block_attn_paged.
 *
 * bdsa_tree_accept: p [bs, B, V] fp32 (p + r*p_stride_r + n*p_stride_n) is
 *   the verifier's distribution after node n, i.e. for n's children; u [bs, B]
 *   fp32 uniforms in [0, 1) indexed by depth, or NULL for greedy.  Walk from
 *   the root: at node n of depth d, x = InvCDF(p[r, n], u[r, d]) (the smallest
 *   k whose cumulative weight exceeds u times the total; -1 if p[r, n] has no
 *   mass) or x = argmax p[r, n] (lowest index on ties); the lowest-index child
 *   of n carrying token x is accepted and the walk continues from it,
 *   otherwise x is emitted (the correction, or the bonus at a leaf) and the
 *   walk ends.  The tree's tokens are chosen rather than sampled, so this is
 *   rejection sampling with one-hot draft distributions: lossless.
 *   Outputs: accept_len [bs] (accepted nodes below the root), path [bs, B]
 *   (node indices: the root, then the accepted nodes; -1 padding),
 *   out_tokens [bs, B] (the accepted nodes' tokens, then x; -1 padding),
 *   bonus_id [bs] = x, new_seq_lens [bs] = seq_lens + accept_len + 1.  The KV
 *   rows of the path's nodes are the ones to keep.
 *   Limits: B <= BDSA_TREE_MAX_NODES, V <= 2^21.  No workspace.  Launch: one thread-block
 *   cluster per request (its CTAs the vocabulary chunks; num_sms sizes them,
 *   0 = the current device's SM count); two cluster barriers per step of the
 *   walk, at most B steps.
 */
int32_t bdsa_tree_prepare(const int32_t *parent, const int32_t *seq_lens,
                          const int32_t *block_table, int32_t max_pages_per_req,
                          int32_t num_pages, int32_t bs, int32_t B, int32_t page_size,
                          int32_t *depth, int32_t *positions, int32_t *cache_loc,
                          uint64_t *tree_mask, int32_t *dev_status, void *stream);
int32_t bdsa_block_attn_paged_tree(const bdsa_bf16 *q, const bdsa_bf16 *k_cache,
                                   const bdsa_bf16 *v_cache, const int32_t *block_table,
                                   int32_t max_pages_per_req, int32_t num_pages,
                                   const int32_t *seq_lens, int32_t max_ctx_len, int32_t bs,
                                   int32_t B, int32_t Hq, int32_t Hkv, int32_t D,
                                   int32_t page_size, float softmax_scale,
                                   const uint64_t *tree_mask, bdsa_bf16 *out, float *lse,
                                   void *workspace, size_t workspace_bytes, int32_t num_sms,
                                   int32_t *dev_status, void *stream);
int32_t bdsa_tree_accept(const int32_t *block_ids, const int32_t *parent, const float *p,
                         int64_t p_stride_r, int64_t p_stride_n, const float *u,
                         const int32_t *seq_lens, int32_t bs, int32_t B, int32_t V,
                         int32_t *accept_len, int32_t *path, int32_t *out_tokens,
                         int32_t *bonus_id, int32_t *new_seq_lens, int32_t num_sms,
                         int32_t *dev_status, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* BDSA_H_ */
