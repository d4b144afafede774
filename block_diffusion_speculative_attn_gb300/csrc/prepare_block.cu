// prepare_block.cu -- per-round block layout in one launch.
//
// "From DFlash to dLLM Self-Spec (II): SGLang Spec V2", section 2.2.2: the
// block starts with the last verified token, every other slot holds the mask
// token, and positions / cache locations are prepared in the same kernel
// instead of a chain of small eager ops.  One thread per (request, slot).
//
// Each kernel lets the next kernel on the stream launch at once (it is the
// attention, launched with programmatic dependent launch, which waits for
// this grid's writes before it reads its inputs), and asks for the shared
// memory carve-out the attention runs with, so that the attention's CTAs can
// start their prologue on SMs still running this grid.
#include <cuda_runtime.h>

#include "bdsa_device.cuh"
#include "bdsa_internal.h"

namespace bdsa {
namespace {

template <typename K>
bool prefer_max_shared(K *kernel) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                cudaSharedmemCarveoutMaxShared) == cudaSuccess;
}

__global__ void __launch_bounds__(256)
    prepare_block_kernel(const int32_t *__restrict__ verified_id,
                         const int32_t *__restrict__ seq_lens,
                         const int32_t *__restrict__ block_table, int max_pages, int num_pages,
                         int bs, int B, int page_size, int mask_token_id,
                         int32_t *__restrict__ block_ids, int32_t *__restrict__ positions,
                         int32_t *__restrict__ cache_loc, int32_t *dev_status) {
    grid_launch_dependents();
    const long idx = (long)blockIdx.x * blockDim.x + threadIdx.x;
    // Pull the block table into L2 (one 128-byte line a thread, up to 2^16
    // entries), so that the attention that follows finds its first page ids
    // there: they are on its critical path, right after its schedule (the
    // Qwen3-8B-shaped verify call measured 64.2 -> 64.0 us, A/B means).  Here
    // the prefetches compete with nothing on that path.
    const long lines = ((long)bs * max_pages + 31) / 32;
    if (idx < lines && idx < 2048)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(block_table + idx * 32));
    if (idx >= (long)bs * B) return;
    const int r = (int)(idx / B), i = (int)(idx % B);
    const int L = seq_lens[r];
    const long pos = (long)L + i;
    block_ids[idx] = (i == 0) ? verified_id[r] : mask_token_id;
    positions[idx] = (int32_t)pos;
    int32_t loc = -1;
    const long page_idx = pos / page_size;
    if (L >= 0 && page_idx < max_pages) {
        const int32_t page = block_table[(long)r * max_pages + page_idx];
        if (page >= 0 && page < num_pages) loc = (int32_t)((long)page * page_size + pos % page_size);
    }
    if (loc < 0) report_status(dev_status, BDSA_DEVICE_OUT_OF_RANGE);
    cache_loc[idx] = loc;
}

// I-DLM Block-N layout ("From DFlash to dLLM Self-Spec (IV)", section 4.3.1):
// 2N-1 slots, [pending, spec_0 .. spec_{N-2}, mask ...] in verify mode (mode
// 1), [pending, mask ...] otherwise; positions and cache locations as above.
__global__ void __launch_bounds__(256)
    idlm_prepare_kernel(const int32_t *__restrict__ pending, const int32_t *__restrict__ specs,
                        const int32_t *__restrict__ mode, const int32_t *__restrict__ seq_lens,
                        const int32_t *__restrict__ block_table, int max_pages, int num_pages,
                        int bs, int N, int page_size, int mask_token_id,
                        int32_t *__restrict__ block_ids, int32_t *__restrict__ positions,
                        int32_t *__restrict__ cache_loc, int32_t *dev_status) {
    grid_launch_dependents();
    const int blk = 2 * N - 1;
    const long idx = (long)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (long)bs * blk) return;
    const int r = (int)(idx / blk), i = (int)(idx % blk);
    const int L = seq_lens[r];
    const long pos = (long)L + i;
    int32_t id = mask_token_id;
    if (i == 0) id = pending[r];
    else if (i < N && mode[r] == 1) id = specs[(long)r * (N - 1) + i - 1];
    block_ids[idx] = id;
    positions[idx] = (int32_t)pos;
    int32_t loc = -1;
    const long page_idx = pos / page_size;
    if (L >= 0 && page_idx < max_pages) {
        const int32_t page = block_table[(long)r * max_pages + page_idx];
        if (page >= 0 && page < num_pages) loc = (int32_t)((long)page * page_size + pos % page_size);
    }
    if (loc < 0) report_status(dev_status, BDSA_DEVICE_OUT_OF_RANGE);
    cache_loc[idx] = loc;
}

// Tree verify layout ("Unlocking Lossless Speedups in LLMs via Discrete
// Diffusion", Psi-Spec Tree sampler): node i of request r sits at block slot i
// (cache location of position L + i) and at sequence position L + depth(i);
// node i's ancestor-or-self set is W = ceil(B / 64) words at
// tree_mask[(r * B + i) * W], bit j % 64 of word j / 64 set iff node j is node
// i or one of its ancestors.  A parent outside [0, i) (or node 0's parent
// other than -1) makes the node a root and is reported.
__global__ void __launch_bounds__(256)
    tree_prepare_kernel(const int32_t *__restrict__ parent, const int32_t *__restrict__ seq_lens,
                        const int32_t *__restrict__ block_table, int max_pages, int num_pages,
                        int bs, int B, int page_size, int32_t *__restrict__ depth,
                        int32_t *__restrict__ positions, int32_t *__restrict__ cache_loc,
                        uint64_t *__restrict__ tree_mask, int32_t *dev_status) {
    grid_launch_dependents();
    const long idx = (long)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (long)bs * B) return;
    const int r = (int)(idx / B), i = (int)(idx % B);
    const int32_t *par = parent + (long)r * B;
    const int p_i = __ldg(par + i);
    if (i == 0 ? p_i != -1 : (p_i < 0 || p_i >= i)) report_status(dev_status, BDSA_DEVICE_OUT_OF_RANGE);
    // The walk visits decreasing node indices, so the word it sets never
    // moves up: one word is built in a register and written (with the empty
    // words the walk skips) each time the walk leaves it.
    const int W = (B + 63) >> 6;
    uint64_t *mrow = tree_mask + idx * W;
    int d = -1, cw = W - 1;
    uint64_t cur = 0;
    for (int k = i; k >= 0;) {
        ++d;
        const int w = k >> 6;
        for (; cw > w; --cw) {
            mrow[cw] = cur;
            cur = 0;
        }
        cur |= 1ull << (k & 63);
        const int pk = k > 0 ? __ldg(par + k) : -1;
        k = (pk >= 0 && pk < k) ? pk : -1;
    }
    for (; cw >= 0; --cw) {
        mrow[cw] = cur;
        cur = 0;
    }
    const int L = __ldg(seq_lens + r);
    depth[idx] = d;
    positions[idx] = L + d;
    const long t = (long)L + i;
    int32_t loc = -1;
    if (L >= 0 && t / page_size < max_pages) {
        const int32_t page = block_table[(long)r * max_pages + t / page_size];
        if (page >= 0 && page < num_pages) loc = (int32_t)((long)page * page_size + t % page_size);
    }
    if (loc < 0) report_status(dev_status, BDSA_DEVICE_OUT_OF_RANGE);
    cache_loc[idx] = loc;
}

}  // namespace

int launch_idlm_prepare(const int32_t *pending, const int32_t *specs, const int32_t *mode,
                        const int32_t *seq_lens, const int32_t *block_table, int max_pages,
                        int num_pages, int bs, int N, int page_size, int mask_token_id,
                        int32_t *block_ids, int32_t *positions, int32_t *cache_loc,
                        int32_t *dev_status, cudaStream_t stream) {
    const long n = (long)bs * (2 * N - 1);
    if (n == 0) return BDSA_OK;
    static const bool carve = prefer_max_shared(idlm_prepare_kernel);
    if (!carve) return BDSA_CUDA_ERROR;
    const unsigned grid = (unsigned)((n + 255) / 256);
    idlm_prepare_kernel<<<grid, 256, 0, stream>>>(pending, specs, mode, seq_lens, block_table,
                                                  max_pages, num_pages, bs, N, page_size,
                                                  mask_token_id, block_ids, positions, cache_loc,
                                                  dev_status);
    return cudaGetLastError() == cudaSuccess ? BDSA_OK : BDSA_CUDA_ERROR;
}

int launch_tree_prepare(const int32_t *parent, const int32_t *seq_lens, const int32_t *block_table,
                        int max_pages, int num_pages, int bs, int B, int page_size,
                        int32_t *depth, int32_t *positions, int32_t *cache_loc,
                        uint64_t *tree_mask, int32_t *dev_status, cudaStream_t stream) {
    const long n = (long)bs * B;
    if (n == 0) return BDSA_OK;
    static const bool carve = prefer_max_shared(tree_prepare_kernel);
    if (!carve) return BDSA_CUDA_ERROR;
    tree_prepare_kernel<<<(unsigned)((n + 255) / 256), 256, 0, stream>>>(
        parent, seq_lens, block_table, max_pages, num_pages, bs, B, page_size, depth, positions,
        cache_loc, tree_mask, dev_status);
    return cudaGetLastError() == cudaSuccess ? BDSA_OK : BDSA_CUDA_ERROR;
}

int launch_prepare_block(const int32_t *verified_id, const int32_t *seq_lens,
                         const int32_t *block_table, int max_pages, int num_pages, int bs, int B,
                         int page_size, int mask_token_id, int32_t *block_ids,
                         int32_t *positions, int32_t *cache_loc, int32_t *dev_status,
                         cudaStream_t stream) {
    const long n = (long)bs * B;
    if (n == 0) return BDSA_OK;
    static const bool carve = prefer_max_shared(prepare_block_kernel);
    if (!carve) return BDSA_CUDA_ERROR;
    const unsigned grid = (unsigned)((n + 255) / 256);
    prepare_block_kernel<<<grid, 256, 0, stream>>>(verified_id, seq_lens, block_table, max_pages,
                                                   num_pages, bs, B, page_size, mask_token_id,
                                                   block_ids, positions, cache_loc, dev_status);
    return cudaGetLastError() == cudaSuccess ? BDSA_OK : BDSA_CUDA_ERROR;
}

}  // namespace bdsa
