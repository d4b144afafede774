// bdsa_internal.h -- host-side launch interfaces shared between the C ABI
// (bdsa_api.cu) and the kernel translation units.  Not installed.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace bdsa {

// ---------------------------------------------------------------- attention
// Persistent stream-K style schedule: `grid` CTAs share the concatenated
// (request, KV head, 128-key tile) sequence in equal contiguous ranges.  The
// workspace holds two partial slots per CTA for units cut between CTAs (a
// bad-page flag, the fp32 log2-sum-exp per row and the fp32 normalised output
// rows).
struct AttnPlan {
    int grid;
    int rows;             // packed query rows per unit (G * B)
    size_t off_part_bad, off_part_ready, off_part_o, off_part_lse;
    size_t workspace;     // total bytes
};

AttnPlan attn_plan(int bs, int B, int Hq, int Hkv, int D, int max_ctx_len, int num_sms);

struct AttnArgs {
    const uint16_t *q, *k_cache, *v_cache;
    const uint16_t *k_new, *v_new;  // fused append (bdsa_block_attn_paged_append), or null
    const int32_t *block_table, *seq_lens;
    int max_pages, num_pages, max_ctx_len, bs, B, Hq, Hkv, D, page_size, mode, num_sms;
    float scale;
    uint16_t *out;
    float *lse;
    const uint64_t *tree_mask;      // TREE mode only
    void *workspace;
    size_t workspace_bytes;
    int32_t *dev_status;
};

// Returns a bdsa_status code.
int launch_block_attn(const AttnArgs &a, cudaStream_t stream);

// ---------------------------------------------------------------- prepare
int launch_prepare_block(const int32_t *verified_id, const int32_t *seq_lens,
                         const int32_t *block_table, int max_pages, int num_pages, int bs, int B,
                         int page_size, int mask_token_id, int32_t *block_ids,
                         int32_t *positions, int32_t *cache_loc, int32_t *dev_status,
                         cudaStream_t stream);

// ---------------------------------------------------------------- accept
struct AcceptPlan {
    int nchunk;       // CTAs per row
    int nseg;         // 256-element segments per vocabulary row
    int spc;          // segments per chunk
    bool cluster;     // one thread-block cluster per row (no global scratch)
    bool prefetch;    // fewer CTAs than SMs: bulk-prefetch each chunk into L2
    size_t workspace; // bytes (0 on the cluster path)
};

AcceptPlan accept_plan(int bs, int B, int V, int num_sms);

struct AcceptArgs {
    const int32_t *block_ids;
    const float *p, *q;
    int64_t psr, psi, qsr, qsi;
    const float *u_acc, *u_samp;
    const int32_t *seq_lens;
    int bs, B, V, num_sms;
    int32_t *accept_len, *commit_len, *out_tokens, *bonus_id, *new_seq_lens;
    void *workspace;
    size_t workspace_bytes;
    int32_t *dev_status;
};

int launch_spec_accept(const AcceptArgs &a, cudaStream_t stream);

// I-DLM Block-N round: layout of 2N-1 slots, verify / sample / trim.
int launch_idlm_prepare(const int32_t *pending, const int32_t *specs, const int32_t *mode,
                        const int32_t *seq_lens, const int32_t *block_table, int max_pages,
                        int num_pages, int bs, int N, int page_size, int mask_token_id,
                        int32_t *block_ids, int32_t *positions, int32_t *cache_loc,
                        int32_t *dev_status, cudaStream_t stream);

struct IdlmArgs {
    const int32_t *block_ids, *mode, *q_slot, *seq_lens;
    const float *p, *q;
    int64_t psr, psi, qsr, qsi;
    const float *u_acc, *u_samp;
    int bs, N, V, num_sms;
    int32_t *accept_len, *n_out, *out_tokens, *next_mode, *next_pending, *next_specs,
        *next_q_slot, *new_seq_lens, *kv_keep;
    int32_t *dev_status;
};

int launch_idlm_accept(const IdlmArgs &a, cudaStream_t stream);

// ---------------------------------------------------------------- tree verify
int launch_tree_prepare(const int32_t *parent, const int32_t *seq_lens, const int32_t *block_table,
                        int max_pages, int num_pages, int bs, int B, int page_size,
                        int32_t *depth, int32_t *positions, int32_t *cache_loc,
                        uint64_t *tree_mask, int32_t *dev_status, cudaStream_t stream);

struct TreeArgs {
    const int32_t *block_ids, *parent, *seq_lens;
    const float *p;
    int64_t psr, psn;
    const float *u;  // [bs, B] uniforms by depth, or null for greedy
    int bs, B, V, num_sms;
    int32_t *accept_len, *path, *out_tokens, *bonus_id, *new_seq_lens;
    int32_t *dev_status;
};

int launch_tree_accept(const TreeArgs &a, cudaStream_t stream);

// ---------------------------------------------------------------- KV materialisation
// Committed rows of the verify block -> every draft layer's K (RMS norm, RoPE)
// and V at the rows' cache slots.  Workspace: the gathered row count, one
// (slot, position) pair and one dense copy of the hidden row per block row.
struct KvMatArgs {
    const uint16_t *hidden;    // [bs*B, H]
    const int32_t *commit_len, *positions, *cache_loc;
    const uint16_t *w_kv;      // [n_layers, 2, Hkv*D, H]
    const uint16_t *k_norm_w;  // [n_layers, D]
    const float *cos_tab, *sin_tab;
    int max_pos;
    float eps;
    int bs, B, H, n_layers, Hkv, D;
    uint16_t *k_cache, *v_cache;
    long long num_slots;
    void *workspace;
    int32_t *dev_status;
};

size_t kvmat_workspace_bytes(int bs, int B, int H);
int launch_kv_materialize(const KvMatArgs &a, cudaStream_t stream);

// ---------------------------------------------------------------- misc
int device_num_sms(int requested);

}  // namespace bdsa
