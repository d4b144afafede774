// bdsa_api.cu -- the extern "C" boundary of libbdsa.so (declared in
// include/bdsa.h): synchronous host-side argument checks, workspace sizing and
// dispatch to the kernel launchers.  No call allocates device memory.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "../../include/bdsa.h"
#include "bdsa_internal.h"

namespace bdsa {

int device_num_sms(int requested) {
    if (requested > 0) return requested;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    static int cache[64] = {0};
    if (dev >= 0 && dev < 64 && cache[dev] > 0) return cache[dev];
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        n = 148;
    if (dev >= 0 && dev < 64) cache[dev] = n;
    return n;
}

}  // namespace bdsa

namespace {

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

}  // namespace

extern "C" {

const char *bdsa_status_string(int32_t status) {
    switch (status) {
        case BDSA_OK: return "BDSA_OK";
        case BDSA_INVALID_ARG: return "BDSA_INVALID_ARG: invalid argument";
        case BDSA_UNSUPPORTED: return "BDSA_UNSUPPORTED: shape not supported by this build";
        case BDSA_MISALIGNED: return "BDSA_MISALIGNED: pointer or stride alignment";
        case BDSA_WORKSPACE_TOO_SMALL: return "BDSA_WORKSPACE_TOO_SMALL";
        case BDSA_CUDA_ERROR: return "BDSA_CUDA_ERROR: CUDA call or launch failed";
        case BDSA_DEVICE_OUT_OF_RANGE: return "BDSA_DEVICE_OUT_OF_RANGE: index out of range on device";
        case BDSA_DEVICE_TIMEOUT: return "BDSA_DEVICE_TIMEOUT: bounded device wait expired";
        default: return "BDSA_UNKNOWN_STATUS";
    }
}

const char *bdsa_version(void) { return "0.1.0"; }

int32_t bdsa_prepare_block(const int32_t *verified_id, const int32_t *seq_lens,
                           const int32_t *block_table, int32_t max_pages_per_req,
                           int32_t num_pages, int32_t bs, int32_t B, int32_t page_size,
                           int32_t mask_token_id, int32_t *block_ids, int32_t *positions,
                           int32_t *cache_loc, int32_t *dev_status, void *stream) {
    if (bs < 0 || B < 1 || page_size < 1 || max_pages_per_req < 1 || num_pages < 1)
        return BDSA_INVALID_ARG;
    if (bs == 0) return BDSA_OK;
    if (!verified_id || !seq_lens || !block_table || !block_ids || !positions || !cache_loc)
        return BDSA_INVALID_ARG;
    if ((int64_t)bs * B > INT32_MAX) return BDSA_UNSUPPORTED;
    return bdsa::launch_prepare_block(verified_id, seq_lens, block_table, max_pages_per_req,
                                      num_pages, bs, B, page_size, mask_token_id, block_ids,
                                      positions, cache_loc, dev_status,
                                      static_cast<cudaStream_t>(stream));
}

size_t bdsa_block_attn_workspace_bytes(int32_t bs, int32_t B, int32_t Hq, int32_t Hkv, int32_t D,
                                       int32_t max_ctx_len, int32_t num_sms) {
    if (bs <= 0 || B <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || max_ctx_len < 0) return 0;
    return bdsa::attn_plan(bs, B, Hq, Hkv, D, max_ctx_len, bdsa::device_num_sms(num_sms))
        .workspace;
}

}  // extern "C"

namespace {

// Checks and dispatch shared by bdsa_block_attn_paged and
// bdsa_block_attn_paged_append (k_new / v_new null for the former).
int32_t attn_call(const bdsa_bf16 *q, const bdsa_bf16 *k_new, const bdsa_bf16 *v_new,
                  const bdsa_bf16 *k_cache, const bdsa_bf16 *v_cache, const int32_t *block_table,
                  int32_t max_pages_per_req, int32_t num_pages, const int32_t *seq_lens,
                  int32_t max_ctx_len, int32_t bs, int32_t B, int32_t Hq, int32_t Hkv, int32_t D,
                  int32_t page_size, float softmax_scale, int32_t mode, const uint64_t *tree_mask,
                  bdsa_bf16 *out, float *lse, void *workspace, size_t workspace_bytes,
                  int32_t num_sms, int32_t *dev_status, void *stream) {
    const bool mode_ok = tree_mask == nullptr
                             ? (mode == BDSA_MODE_DRAFT || mode == BDSA_MODE_VERIFY)
                             : mode == BDSA_MODE_TREE;
    if (bs < 0 || B < 1 || Hq < 1 || Hkv < 1 || max_pages_per_req < 1 || num_pages < 1 ||
        max_ctx_len < 0 || !isfinite(softmax_scale) || !(softmax_scale > 0.f) || !mode_ok)
        return BDSA_INVALID_ARG;
    if (bs == 0) return BDSA_OK;
    if (!q || !k_cache || !v_cache || !block_table || !seq_lens || !out) return BDSA_INVALID_ARG;
    if ((k_new == nullptr) != (v_new == nullptr)) return BDSA_INVALID_ARG;
    if (Hq % Hkv != 0) return BDSA_INVALID_ARG;
    if (D != 64 && D != 128) return BDSA_UNSUPPORTED;
    // DRAFT / VERIFY: one tile of G * B <= 128 query rows a (request, KV head);
    // TREE: trees of up to BDSA_TREE_MAX_NODES nodes in 128-row tiles
    if (tree_mask == nullptr ? (B > 64 || (Hq / Hkv) * B > 128)
                             : (B > BDSA_TREE_MAX_NODES || Hq / Hkv > 128))
        return BDSA_UNSUPPORTED;
    if (!pow2(page_size) || page_size < 8) return BDSA_UNSUPPORTED;
    if ((int64_t)num_pages * page_size > INT32_MAX) return BDSA_UNSUPPORTED;
    if ((int64_t)bs * B > INT32_MAX) return BDSA_UNSUPPORTED;
    if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
        (k_new && !aligned(k_new, 16)) || (v_new && !aligned(v_new, 16)) ||
        (lse && !aligned(lse, 4)) || (workspace && !aligned(workspace, 256)) ||
        (tree_mask && !aligned(tree_mask, 8)))
        return BDSA_MISALIGNED;
    bdsa::AttnArgs a;
    a.q = reinterpret_cast<const uint16_t *>(q);
    a.k_cache = reinterpret_cast<const uint16_t *>(k_cache);
    a.v_cache = reinterpret_cast<const uint16_t *>(v_cache);
    a.k_new = reinterpret_cast<const uint16_t *>(k_new);
    a.v_new = reinterpret_cast<const uint16_t *>(v_new);
    a.block_table = block_table;
    a.seq_lens = seq_lens;
    a.max_pages = max_pages_per_req;
    a.num_pages = num_pages;
    a.max_ctx_len = max_ctx_len;
    a.bs = bs;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.D = D;
    a.page_size = page_size;
    a.mode = mode;
    a.num_sms = bdsa::device_num_sms(num_sms);
    a.scale = softmax_scale;
    a.out = reinterpret_cast<uint16_t *>(out);
    a.lse = lse;
    a.tree_mask = tree_mask;
    a.workspace = workspace;
    a.workspace_bytes = workspace_bytes;
    a.dev_status = dev_status;
    return bdsa::launch_block_attn(a, static_cast<cudaStream_t>(stream));
}

}  // namespace

extern "C" {

int32_t bdsa_block_attn_paged(const bdsa_bf16 *q, const bdsa_bf16 *k_cache,
                              const bdsa_bf16 *v_cache, const int32_t *block_table,
                              int32_t max_pages_per_req, int32_t num_pages,
                              const int32_t *seq_lens, int32_t max_ctx_len, int32_t bs,
                              int32_t B, int32_t Hq, int32_t Hkv, int32_t D, int32_t page_size,
                              float softmax_scale, int32_t mode, bdsa_bf16 *out, float *lse,
                              void *workspace, size_t workspace_bytes, int32_t num_sms,
                              int32_t *dev_status, void *stream) {
    return attn_call(q, nullptr, nullptr, k_cache, v_cache, block_table, max_pages_per_req,
                     num_pages, seq_lens, max_ctx_len, bs, B, Hq, Hkv, D, page_size,
                     softmax_scale, mode, nullptr, out, lse, workspace, workspace_bytes, num_sms,
                     dev_status, stream);
}

int32_t bdsa_block_attn_paged_tree(const bdsa_bf16 *q, const bdsa_bf16 *k_cache,
                                   const bdsa_bf16 *v_cache, const int32_t *block_table,
                                   int32_t max_pages_per_req, int32_t num_pages,
                                   const int32_t *seq_lens, int32_t max_ctx_len, int32_t bs,
                                   int32_t B, int32_t Hq, int32_t Hkv, int32_t D,
                                   int32_t page_size, float softmax_scale,
                                   const uint64_t *tree_mask, bdsa_bf16 *out, float *lse,
                                   void *workspace, size_t workspace_bytes, int32_t num_sms,
                                   int32_t *dev_status, void *stream) {
    if (bs > 0 && !tree_mask) return BDSA_INVALID_ARG;
    return attn_call(q, nullptr, nullptr, k_cache, v_cache, block_table, max_pages_per_req,
                     num_pages, seq_lens, max_ctx_len, bs, B, Hq, Hkv, D, page_size,
                     softmax_scale, BDSA_MODE_TREE, tree_mask, out, lse, workspace,
                     workspace_bytes, num_sms, dev_status, stream);
}

int32_t bdsa_block_attn_paged_append(const bdsa_bf16 *q, const bdsa_bf16 *k_new,
                                     const bdsa_bf16 *v_new, bdsa_bf16 *k_cache,
                                     bdsa_bf16 *v_cache, const int32_t *block_table,
                                     int32_t max_pages_per_req, int32_t num_pages,
                                     const int32_t *seq_lens, int32_t max_ctx_len, int32_t bs,
                                     int32_t B, int32_t Hq, int32_t Hkv, int32_t D,
                                     int32_t page_size, float softmax_scale, int32_t mode,
                                     bdsa_bf16 *out, float *lse, void *workspace,
                                     size_t workspace_bytes, int32_t num_sms, int32_t *dev_status,
                                     void *stream) {
    if (bs > 0 && (!k_new || !v_new)) return BDSA_INVALID_ARG;
    return attn_call(q, k_new, v_new, k_cache, v_cache, block_table, max_pages_per_req, num_pages,
                     seq_lens, max_ctx_len, bs, B, Hq, Hkv, D, page_size, softmax_scale, mode,
                     nullptr, out, lse, workspace, workspace_bytes, num_sms, dev_status, stream);
}

int32_t bdsa_idlm_prepare(const int32_t *pending, const int32_t *specs, const int32_t *mode,
                          const int32_t *seq_lens, const int32_t *block_table,
                          int32_t max_pages_per_req, int32_t num_pages, int32_t bs, int32_t N,
                          int32_t page_size, int32_t mask_token_id, int32_t *block_ids,
                          int32_t *positions, int32_t *cache_loc, int32_t *dev_status,
                          void *stream) {
    if (bs < 0 || N < 1 || page_size < 1 || max_pages_per_req < 1 || num_pages < 1)
        return BDSA_INVALID_ARG;
    if (bs == 0) return BDSA_OK;
    if (!pending || !mode || !seq_lens || !block_table || !block_ids || !positions ||
        !cache_loc || (N > 1 && !specs))
        return BDSA_INVALID_ARG;
    if ((int64_t)bs * (2 * (int64_t)N - 1) > INT32_MAX) return BDSA_UNSUPPORTED;
    return bdsa::launch_idlm_prepare(pending, specs, mode, seq_lens, block_table,
                                     max_pages_per_req, num_pages, bs, N, page_size,
                                     mask_token_id, block_ids, positions, cache_loc, dev_status,
                                     static_cast<cudaStream_t>(stream));
}

int32_t bdsa_idlm_accept(const int32_t *block_ids, const int32_t *mode, const float *p,
                         int64_t p_stride_r, int64_t p_stride_i, const float *q_prev,
                         int64_t q_stride_r, int64_t q_stride_i, const int32_t *q_slot,
                         const float *u_acc, const float *u_samp, const int32_t *seq_lens,
                         int32_t bs, int32_t N, int32_t V, int32_t *accept_len, int32_t *n_out,
                         int32_t *out_tokens, int32_t *next_mode, int32_t *next_pending,
                         int32_t *next_specs, int32_t *next_q_slot, int32_t *new_seq_lens,
                         int32_t *kv_keep, int32_t num_sms, int32_t *dev_status, void *stream) {
    if (bs < 0 || N < 1 || V < 1 || p_stride_r < 0 || p_stride_i < 0 || q_stride_r < 0 ||
        q_stride_i < 0)
        return BDSA_INVALID_ARG;
    if (bs == 0) return BDSA_OK;
    if (N > 32 || V > (1 << 21)) return BDSA_UNSUPPORTED;
    if (!block_ids || !mode || !p || !q_slot || !u_samp || !seq_lens || !accept_len || !n_out ||
        !out_tokens || !next_mode || !next_pending || !next_q_slot || !new_seq_lens || !kv_keep)
        return BDSA_INVALID_ARG;
    if (N > 1 && (!q_prev || !u_acc || !next_specs)) return BDSA_INVALID_ARG;
    if (!aligned(p, 4) || (q_prev && !aligned(q_prev, 4))) return BDSA_MISALIGNED;
    bdsa::IdlmArgs a;
    a.block_ids = block_ids;
    a.mode = mode;
    a.q_slot = q_slot;
    a.seq_lens = seq_lens;
    a.p = p;
    a.q = q_prev;
    a.psr = p_stride_r;
    a.psi = p_stride_i;
    a.qsr = q_stride_r;
    a.qsi = q_stride_i;
    a.u_acc = u_acc;
    a.u_samp = u_samp;
    a.bs = bs;
    a.N = N;
    a.V = V;
    a.num_sms = bdsa::device_num_sms(num_sms);
    a.accept_len = accept_len;
    a.n_out = n_out;
    a.out_tokens = out_tokens;
    a.next_mode = next_mode;
    a.next_pending = next_pending;
    a.next_specs = next_specs;
    a.next_q_slot = next_q_slot;
    a.new_seq_lens = new_seq_lens;
    a.kv_keep = kv_keep;
    a.dev_status = dev_status;
    return bdsa::launch_idlm_accept(a, static_cast<cudaStream_t>(stream));
}

size_t bdsa_spec_accept_workspace_bytes(int32_t bs, int32_t B, int32_t V, int32_t num_sms) {
    if (bs <= 0 || B <= 0 || V <= 0) return 0;
    return bdsa::accept_plan(bs, B, V, bdsa::device_num_sms(num_sms)).workspace;
}

int32_t bdsa_spec_accept(const int32_t *block_ids, const float *p, int64_t p_stride_r,
                         int64_t p_stride_i, const float *q, int64_t q_stride_r,
                         int64_t q_stride_i, const float *u_acc, const float *u_samp,
                         const int32_t *seq_lens, int32_t bs, int32_t B, int32_t V,
                         int32_t *accept_len, int32_t *commit_len, int32_t *out_tokens,
                         int32_t *bonus_id, int32_t *new_seq_lens, void *workspace,
                         size_t workspace_bytes, int32_t num_sms, int32_t *dev_status,
                         void *stream) {
    if (bs < 0 || B < 1 || V < 1 || p_stride_r < 0 || p_stride_i < 0 || q_stride_r < 0 ||
        q_stride_i < 0)
        return BDSA_INVALID_ARG;
    if (bs == 0) return BDSA_OK;
    if (B > 64) return BDSA_UNSUPPORTED;
    if (!block_ids || !p || !seq_lens || !accept_len || !commit_len || !out_tokens || !bonus_id ||
        !new_seq_lens)
        return BDSA_INVALID_ARG;
    if (q != nullptr && (!u_samp || (B > 1 && !u_acc))) return BDSA_INVALID_ARG;
    if (!aligned(p, 4) || (q && !aligned(q, 4)) || (workspace && !aligned(workspace, 256)))
        return BDSA_MISALIGNED;
    bdsa::AcceptArgs a;
    a.block_ids = block_ids;
    a.p = p;
    a.q = q;
    a.psr = p_stride_r;
    a.psi = p_stride_i;
    a.qsr = q_stride_r;
    a.qsi = q_stride_i;
    a.u_acc = u_acc;
    a.u_samp = u_samp;
    a.seq_lens = seq_lens;
    a.bs = bs;
    a.B = B;
    a.V = V;
    a.num_sms = bdsa::device_num_sms(num_sms);
    a.accept_len = accept_len;
    a.commit_len = commit_len;
    a.out_tokens = out_tokens;
    a.bonus_id = bonus_id;
    a.new_seq_lens = new_seq_lens;
    a.workspace = workspace;
    a.workspace_bytes = workspace_bytes;
    a.dev_status = dev_status;
    return bdsa::launch_spec_accept(a, static_cast<cudaStream_t>(stream));
}

size_t bdsa_kv_materialize_workspace_bytes(int32_t bs, int32_t B, int32_t H) {
    if (bs <= 0 || B <= 0 || H <= 0) return 0;
    return bdsa::kvmat_workspace_bytes(bs, B, H);
}

int32_t bdsa_kv_materialize(const bdsa_bf16 *hidden, const int32_t *commit_len,
                            const int32_t *positions, const int32_t *cache_loc, int32_t bs,
                            int32_t B, int32_t H, const bdsa_bf16 *w_kv,
                            const bdsa_bf16 *k_norm_w, int32_t n_layers, int32_t Hkv, int32_t D,
                            const float *rope_cos, const float *rope_sin, int32_t max_pos,
                            float rms_eps, bdsa_bf16 *k_cache, bdsa_bf16 *v_cache,
                            int64_t num_slots, void *workspace, size_t workspace_bytes,
                            int32_t *dev_status, void *stream) {
    if (bs < 0 || B < 1 || H < 1 || n_layers < 1 || Hkv < 1 || D < 1 || max_pos < 1 ||
        num_slots < 1 || !(rms_eps >= 0.f) || !isfinite(rms_eps))
        return BDSA_INVALID_ARG;
    if (D != 128 || H % 128 != 0) return BDSA_UNSUPPORTED;
    if ((int64_t)bs * B > (1 << 24) || (int64_t)n_layers * 2 * Hkv * D > (1LL << 31) ||
        num_slots > (1LL << 31))
        return BDSA_UNSUPPORTED;
    if (bs == 0) return BDSA_OK;
    if (!hidden || !commit_len || !positions || !cache_loc || !w_kv || !k_norm_w || !rope_cos ||
        !rope_sin || !k_cache || !v_cache || !workspace)
        return BDSA_INVALID_ARG;
    if (!aligned(hidden, 16) || !aligned(w_kv, 16) || !aligned(k_cache, 16) ||
        !aligned(v_cache, 16) || !aligned(k_norm_w, 2) || !aligned(rope_cos, 4) ||
        !aligned(rope_sin, 4) || !aligned(workspace, 256))
        return BDSA_MISALIGNED;
    if (workspace_bytes < bdsa::kvmat_workspace_bytes(bs, B, H)) return BDSA_WORKSPACE_TOO_SMALL;
    bdsa::KvMatArgs a;
    a.hidden = reinterpret_cast<const uint16_t *>(hidden);
    a.commit_len = commit_len;
    a.positions = positions;
    a.cache_loc = cache_loc;
    a.w_kv = reinterpret_cast<const uint16_t *>(w_kv);
    a.k_norm_w = reinterpret_cast<const uint16_t *>(k_norm_w);
    a.cos_tab = rope_cos;
    a.sin_tab = rope_sin;
    a.max_pos = max_pos;
    a.eps = rms_eps;
    a.bs = bs;
    a.B = B;
    a.H = H;
    a.n_layers = n_layers;
    a.Hkv = Hkv;
    a.D = D;
    a.k_cache = reinterpret_cast<uint16_t *>(k_cache);
    a.v_cache = reinterpret_cast<uint16_t *>(v_cache);
    a.num_slots = num_slots;
    a.workspace = workspace;
    a.dev_status = dev_status;
    return bdsa::launch_kv_materialize(a, static_cast<cudaStream_t>(stream));
}

int32_t bdsa_tree_prepare(const int32_t *parent, const int32_t *seq_lens,
                          const int32_t *block_table, int32_t max_pages_per_req,
                          int32_t num_pages, int32_t bs, int32_t B, int32_t page_size,
                          int32_t *depth, int32_t *positions, int32_t *cache_loc,
                          uint64_t *tree_mask, int32_t *dev_status, void *stream) {
    if (bs < 0 || B < 1 || page_size < 1 || max_pages_per_req < 1 || num_pages < 1)
        return BDSA_INVALID_ARG;
    if (B > BDSA_TREE_MAX_NODES) return BDSA_UNSUPPORTED;
    if (bs == 0) return BDSA_OK;
    if (!parent || !seq_lens || !block_table || !depth || !positions || !cache_loc || !tree_mask)
        return BDSA_INVALID_ARG;
    if ((int64_t)bs * B > INT32_MAX) return BDSA_UNSUPPORTED;
    if (!aligned(tree_mask, 8)) return BDSA_MISALIGNED;
    return bdsa::launch_tree_prepare(parent, seq_lens, block_table, max_pages_per_req, num_pages,
                                     bs, B, page_size, depth, positions, cache_loc, tree_mask,
                                     dev_status, static_cast<cudaStream_t>(stream));
}

int32_t bdsa_tree_accept(const int32_t *block_ids, const int32_t *parent, const float *p,
                         int64_t p_stride_r, int64_t p_stride_n, const float *u,
                         const int32_t *seq_lens, int32_t bs, int32_t B, int32_t V,
                         int32_t *accept_len, int32_t *path, int32_t *out_tokens,
                         int32_t *bonus_id, int32_t *new_seq_lens, int32_t num_sms,
                         int32_t *dev_status, void *stream) {
    if (bs < 0 || B < 1 || V < 1 || p_stride_r < 0 || p_stride_n < 0) return BDSA_INVALID_ARG;
    if (B > BDSA_TREE_MAX_NODES || V > (1 << 21)) return BDSA_UNSUPPORTED;
    if (bs == 0) return BDSA_OK;
    if (!block_ids || !parent || !p || !seq_lens || !accept_len || !path || !out_tokens ||
        !bonus_id || !new_seq_lens)
        return BDSA_INVALID_ARG;
    if (!aligned(p, 4) || (u && !aligned(u, 4))) return BDSA_MISALIGNED;
    bdsa::TreeArgs a;
    a.block_ids = block_ids;
    a.parent = parent;
    a.seq_lens = seq_lens;
    a.p = p;
    a.psr = p_stride_r;
    a.psn = p_stride_n;
    a.u = u;
    a.bs = bs;
    a.B = B;
    a.V = V;
    a.num_sms = bdsa::device_num_sms(num_sms);
    a.accept_len = accept_len;
    a.path = path;
    a.out_tokens = out_tokens;
    a.bonus_id = bonus_id;
    a.new_seq_lens = new_seq_lens;
    a.dev_status = dev_status;
    return bdsa::launch_tree_accept(a, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
