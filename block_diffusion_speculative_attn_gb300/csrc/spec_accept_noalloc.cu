// spec_accept_noalloc.cu -- bdsa_spec_accept for callers that cannot provide
// device memory for scratch.
//
// Some callers cannot allocate device memory when the step runs: a serving
// loop whose memory plan is fixed before start-up (every buffer comes from one
// pre-sized pool and nothing may be added later), code running while a CUDA
// graph is being captured (allocation calls are not allowed there), or a
// host framework that owns the allocator and hands this library only the
// step's own tensors.  This entry point takes the same inputs and outputs as
// bdsa_spec_accept but uses a fixed scratch array that lives in this
// library's device image instead of a caller-provided workspace.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/bdsa.h"
#include "bdsa_internal.h"

namespace {

// Fixed scratch: 8 MiB on every GPU that loads the library, held until the
// process exits.  Only vocabularies above 2^21 use scratch (about 60 rows at
// V = 2^22 fit); smaller ones need none.
constexpr size_t kScratchBytes = size_t(8) << 20;
static __device__ __align__(256) unsigned char g_accept_scratch[kScratchBytes];

// Device address of g_accept_scratch, resolved once per device.  In host code
// the symbol's name is only a handle; the kernels need this address.
constexpr int kMaxDevices = 64;
void *g_scratch_addr[kMaxDevices] = {nullptr};
std::mutex g_scratch_mu;

int scratch_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return BDSA_CUDA_ERROR;
    if (dev < 0 || dev >= kMaxDevices) return BDSA_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_accept_scratch) != cudaSuccess || p == nullptr)
            return BDSA_CUDA_ERROR;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return BDSA_OK;
}

}  // namespace

extern "C" int32_t bdsa_spec_accept_noalloc(const int32_t *block_ids, const float *p,
                                            int64_t p_stride_r, int64_t p_stride_i,
                                            const float *q, int64_t q_stride_r,
                                            int64_t q_stride_i, const float *u_acc,
                                            const float *u_samp, const int32_t *seq_lens,
                                            int32_t bs, int32_t B, int32_t V,
                                            int32_t *accept_len, int32_t *commit_len,
                                            int32_t *out_tokens, int32_t *bonus_id,
                                            int32_t *new_seq_lens, int32_t num_sms,
                                            int32_t *dev_status, void *stream) {
    if (bs < 0 || B < 1 || V < 1) return BDSA_INVALID_ARG;
    if (bs == 0) return BDSA_OK;
    // The scratch this problem needs must fit the fixed array.
    const size_t need = bdsa_spec_accept_workspace_bytes(bs, B, V, num_sms);
    if (need > kScratchBytes) return BDSA_WORKSPACE_TOO_SMALL;
    void *scratch = nullptr;
    const int st = scratch_address(&scratch);
    if (st != BDSA_OK) return st;
    // Same checks and kernels as bdsa_spec_accept; a launch that uses scratch
    // clears the per-row counters it needs at zero before the kernel runs.
    return bdsa_spec_accept(block_ids, p, p_stride_r, p_stride_i, q, q_stride_r, q_stride_i,
                            u_acc, u_samp, seq_lens, bs, B, V, accept_len, commit_len,
                            out_tokens, bonus_id, new_seq_lens, scratch, kScratchBytes, num_sms,
                            dev_status, stream);
}
