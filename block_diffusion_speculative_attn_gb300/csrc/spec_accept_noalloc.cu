// spec_accept_noalloc.cu -- bdsa_spec_accept for callers that cannot provide
// device memory for scratch.
//
// Some callers cannot allocate device memory when the step runs: a serving
// loop whose memory is planned once at start-up (every buffer comes from one
// pre-sized pool and nothing may be added later), or a host framework that
// owns the device allocator and hands this library only the step's own
// tensors.  This entry point takes the same inputs and outputs as
// bdsa_spec_accept but uses a fixed scratch array that lives in this
// library's device image instead of a caller-provided workspace.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/bdsa.h"
#include "bdsa_internal.h"

namespace {

// Fixed scratch: 8 MiB on every GPU that loads the library, held until the
// process exits.  Only vocabularies above 2^21 use scratch (for example up to
// about 60 rows at V = 2^22); smaller ones need none.
constexpr size_t kScratchBytes = size_t(8) << 20;
static __device__ __align__(256) unsigned char g_accept_scratch[kScratchBytes];

// Device address of g_accept_scratch, resolved once per device by the first
// call made with that device current.  In host code the symbol's name is only
// a host-side handle; the kernels need this address.  The cache is never
// invalidated, so a cudaDeviceReset later in the process is not supported.
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
    // The argument checks of bdsa_spec_accept, in its order, so that a bad
    // argument gets the same status from both entry points.
    if (bs < 0 || B < 1 || V < 1 || p_stride_r < 0 || p_stride_i < 0 || q_stride_r < 0 ||
        q_stride_i < 0)
        return BDSA_INVALID_ARG;
    if (bs == 0) return BDSA_OK;
    if (B > 64) return BDSA_UNSUPPORTED;
    if (!block_ids || !p || !seq_lens || !accept_len || !commit_len || !out_tokens || !bonus_id ||
        !new_seq_lens)
        return BDSA_INVALID_ARG;
    if (q != nullptr && (!u_samp || (B > 1 && !u_acc))) return BDSA_INVALID_ARG;
    // Set-up on the first call on this device, whatever its size: the
    // address lookup happens then, with the caller's device current.
    void *scratch = nullptr;
    const int st = scratch_address(&scratch);
    if (st != BDSA_OK) return st;
    // The scratch this problem needs must fit the fixed array.
    const size_t need = bdsa_spec_accept_workspace_bytes(bs, B, V, num_sms);
    if (need > kScratchBytes) return BDSA_WORKSPACE_TOO_SMALL;
    // Same kernels as bdsa_spec_accept.  A problem that needs no scratch
    // (V <= 2^21) is given none, so its kernels never touch the array; one
    // that does gets the array, and its per-row counters are cleared to zero
    // on `stream` before its kernel runs.
    return bdsa_spec_accept(block_ids, p, p_stride_r, p_stride_i, q, q_stride_r, q_stride_i,
                            u_acc, u_samp, seq_lens, bs, B, V, accept_len, commit_len,
                            out_tokens, bonus_id, new_seq_lens, need > 0 ? scratch : nullptr,
                            need > 0 ? kScratchBytes : 0, num_sms, dev_status, stream);
}
