// spec_accept.cu -- lossless speculative acceptance over the vocabulary.
//
// Rules ("From DFlash to dLLM Self-Spec (IV)", section 4.3.1; "Unlocking
// Lossless Speedups in LLMs via Discrete Diffusion", background on speculative
// decoding and the Psi-Spec step; "From DFlash to dLLM Self-Spec (II)", section
// 2.2.5 for the greedy rule and the emitted tensors):
//   accept d_i while u_acc < min(1, p(d_i) / q(d_i))   (IEEE fp32 divide)
//   first rejection at a: token ~ max(0, p[a] - q[a]) (fp32 weights)
//   no rejection:         token ~ p[B-1]              (bonus)
//   greedy:               accept while d_i == argmax p[i-1]; token = argmax p[a]
// A draw is the smallest k whose cumulative weight exceeds u * total.
//
// Layout of the work: a row's vocabulary is cut into `nchunk` chunks of
// 256-element segments and each chunk is one CTA, so even a handful of rows
// spreads over the whole GPU.  Every CTA recomputes the accepted length a
// (B - 1 gathered probability pairs), sweeps its chunk once with 16-byte loads
// and stores one fp64 total per segment (error-free TwoSum pairwise sums of 8
// elements per lane, fp64 across lanes).  The last CTA of a row to finish
// (atomic counter; nothing ever waits) scans the segment totals, re-reads the
// one segment that holds the crossing point and resolves the token to a single
// index.  Cumulative sums stay within ~1e-13 relative of the exact sums, far
// inside the 1e-9 band within which the fp64 oracle flags a draw as
// order-dependent.
#include <cuda_runtime.h>
#include <limits.h>

#include "bdsa_device.cuh"
#include "bdsa_internal.h"

namespace bdsa {
namespace {

constexpr int kSeg = 256;  // vocabulary elements per segment (32 lanes x 8)
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

struct Params {
    const int32_t *block_ids;
    const float *p;
    const float *q;
    int64_t psr, psi, qsr, qsi;
    const float *u_acc;
    const float *u_samp;
    const int32_t *seq_lens;
    int bs, B, V, nchunk, nseg, spc;
    int32_t *accept_len, *commit_len, *out_tokens, *bonus_id, *new_seq_lens;
    double *seg_sum;   // [bs, nseg]
    int32_t *counter;  // [bs], zeroed before the launch
    float *am_val;     // [bs, B, nchunk]  (greedy)
    int32_t *am_idx;   // [bs, B, nchunk]  (greedy)
    int32_t *dev_status;
};

// The 8 weights of one lane: max(0, p - q) (residual) or p (q == nullptr).
__device__ __forceinline__ void load_weights(const float *prow, const float *qrow, long e0, int V,
                                             float (&w)[8]) {
    const bool vec = (e0 + 8 <= V) && ((reinterpret_cast<uintptr_t>(prow + e0) & 15) == 0) &&
                     (qrow == nullptr || (reinterpret_cast<uintptr_t>(qrow + e0) & 15) == 0);
    float pv[8], qv[8];
    if (vec) {
        const float4 a = __ldg(reinterpret_cast<const float4 *>(prow + e0));
        const float4 b = __ldg(reinterpret_cast<const float4 *>(prow + e0 + 4));
        pv[0] = a.x; pv[1] = a.y; pv[2] = a.z; pv[3] = a.w;
        pv[4] = b.x; pv[5] = b.y; pv[6] = b.z; pv[7] = b.w;
        if (qrow != nullptr) {
            const float4 c = __ldg(reinterpret_cast<const float4 *>(qrow + e0));
            const float4 d = __ldg(reinterpret_cast<const float4 *>(qrow + e0 + 4));
            qv[0] = c.x; qv[1] = c.y; qv[2] = c.z; qv[3] = c.w;
            qv[4] = d.x; qv[5] = d.y; qv[6] = d.z; qv[7] = d.w;
        }
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const long k = e0 + e;
            pv[e] = k < V ? __ldg(prow + k) : 0.f;
            qv[e] = (qrow != nullptr && k < V) ? __ldg(qrow + k) : 0.f;
        }
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        if (qrow != nullptr) {
            const float d = __fsub_rn(pv[e], qv[e]);
            w[e] = d > 0.f ? d : 0.f;
        } else {
            w[e] = pv[e];
        }
    }
}

// Error-free fp32 addition (Knuth's TwoSum): a + b == s + e exactly.
__device__ __forceinline__ float two_sum(float a, float b, float &e) {
    const float s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
    return s;
}

// Sum of 8 weights as an fp64 value within ~2^-46 relative of the exact sum: a
// pairwise tree of TwoSums keeps every rounding error, and only the (tiny) sum
// of those errors is rounded.  Fixed order; the sweep and the resolve step
// both use it.
__device__ __forceinline__ double group_sum(const float (&w)[8]) {
    float e0, e1, e2, e3, e4, e5, e6;
    const float s01 = two_sum(w[0], w[1], e0);
    const float s23 = two_sum(w[2], w[3], e1);
    const float s45 = two_sum(w[4], w[5], e2);
    const float s67 = two_sum(w[6], w[7], e3);
    const float s03 = two_sum(s01, s23, e4);
    const float s47 = two_sum(s45, s67, e5);
    const float s07 = two_sum(s03, s47, e6);
    const float err = __fadd_rn(__fadd_rn(__fadd_rn(e0, e1), __fadd_rn(e2, e3)),
                                __fadd_rn(__fadd_rn(e4, e5), e6));
    return (double)s07 + (double)err;
}

__device__ __forceinline__ double warp_sum_f64(double v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Accepted draft count for row r (stochastic mode), computed by one warp.
__device__ int accepted_len(const Params &P, int r, int lane, bool &bad_id) {
    const int B = P.B;
    bool bad_any = false;
    int a = -1;
    for (int base = 1; base < B; base += 32) {
        const int i = base + lane;
        bool rej = false;
        bad_id = false;
        if (i < B) {
            const int d = P.block_ids[(long)r * B + i];
            if (d < 0 || d >= P.V) {
                rej = true;
                bad_id = true;
            } else {
                const float pv = __ldg(P.p + r * P.psr + (i - 1) * P.psi + d);
                const float qv = __ldg(P.q + r * P.qsr + (i - 1) * P.qsi + d);
                const float u = __ldg(P.u_acc + (long)r * (B - 1) + (i - 1));
                bool acc;
                if (qv == 0.f) {
                    acc = pv > 0.f;
                } else {
                    const float ratio = __fdiv_rn(pv, qv);
                    acc = u < fminf(1.f, ratio);
                }
                rej = !acc;
            }
        }
        // any draft id outside the vocabulary is a data error, tested or not
        bad_any = bad_any || __any_sync(0xffffffffu, bad_id);
        const unsigned m = __ballot_sync(0xffffffffu, rej);
        if (m != 0u && a < 0) a = base + (__ffs(m) - 1) - 1;
    }
    bad_id = bad_any;
    return a < 0 ? B - 1 : a;
}

// Segment totals of this CTA's chunk for the chosen distribution.
__device__ void sweep_chunk(const Params &P, int r, const float *prow, const float *qrow,
                            int seg_begin, int seg_end, int warp, int lane) {
    for (int seg = seg_begin + warp; seg < seg_end; seg += kWarps) {
        float w[8];
        load_weights(prow, qrow, (long)seg * kSeg + lane * 8, P.V, w);
        const double t = warp_sum_f64(group_sum(w));
        if (lane == 0) P.seg_sum[(long)r * P.nseg + seg] = t;
    }
}

// Resolve the draw InvCDF(w, u) from the segment totals; executed by warp 0.
// Returns the token index (or -1 when the weights are all zero).
__device__ int resolve_draw(const Params &P, int r, const float *prow, const float *qrow,
                            float u, int lane) {
    const int nseg = P.nseg;
    const int per = (nseg + 31) / 32;
    const int s0 = min(nseg, lane * per), s1 = min(nseg, s0 + per);
    const double *seg = P.seg_sum + (long)r * nseg;
    double loc = 0.0;
    for (int s = s0; s < s1; ++s) loc += __ldcg(seg + s);
    double inc = loc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const double t = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += t;
    }
    double excl = __shfl_up_sync(0xffffffffu, inc, 1);
    if (lane == 0) excl = 0.0;
    const double S = __shfl_sync(0xffffffffu, inc, 31);
    if (!(S > 0.0)) return -1;
    double T = (double)u * S;

    // first segment whose cumulative total exceeds T
    int found = -1;
    double run = excl;
    for (int s = s0; s < s1; ++s) {
        const double v = __ldcg(seg + s);
        if (run + v > T) {
            found = s;
            break;
        }
        run += v;
    }
    const unsigned any = __ballot_sync(0xffffffffu, found >= 0);
    int seg_star;
    double base_seg;
    if (any != 0u) {
        const int leader = __ffs(any) - 1;
        seg_star = __shfl_sync(0xffffffffu, found, leader);
        base_seg = __shfl_sync(0xffffffffu, run, leader);
    } else {
        // rounding fallback: the last segment with positive mass, no crossing inside it
        int last = -1;
        for (int s = s0; s < s1; ++s)
            if (__ldcg(seg + s) > 0.0) last = s;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) last = max(last, __shfl_xor_sync(0xffffffffu, last, o));
        seg_star = last;
        base_seg = 0.0;
        T = INFINITY;
    }
    // within the segment: one 8-element group per lane
    float w[8];
    const long e0 = (long)seg_star * kSeg + lane * 8;
    load_weights(prow, qrow, e0, P.V, w);
    const double g = group_sum(w);
    double ginc = g;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const double t = __shfl_up_sync(0xffffffffu, ginc, o);
        if (lane >= o) ginc += t;
    }
    double gexcl = __shfl_up_sync(0xffffffffu, ginc, 1);
    if (lane == 0) gexcl = 0.0;
    const double gb = base_seg + gexcl;
    const unsigned cross = __ballot_sync(0xffffffffu, gb + g > T);
    int lane_star;
    double cum;
    bool use_cross;
    if (cross != 0u) {
        lane_star = __ffs(cross) - 1;
        use_cross = true;
    } else {
        const unsigned pos = __ballot_sync(0xffffffffu, g > 0.0);
        lane_star = pos ? 31 - __clz(pos) : 0;
        use_cross = false;
    }
    cum = __shfl_sync(0xffffffffu, gb, lane_star);
    int k = -1;
    if (lane == lane_star) {
        int last_pos = -1;
        for (int e = 0; e < 8; ++e) {
            if (w[e] > 0.f) last_pos = e;
            cum += (double)w[e];
            if (use_cross && cum > T) {
                k = e;
                break;
            }
        }
        if (k < 0) k = last_pos;
        if (k >= 0) k += (int)e0;
    }
    return __shfl_sync(0xffffffffu, k, lane_star);
}

__device__ void write_outputs(const Params &P, int r, int a, int token) {
    const int B = P.B;
    for (int i = threadIdx.x; i < B; i += blockDim.x) {
        int32_t v = -1;
        if (i < a) v = P.block_ids[(long)r * B + i + 1];
        else if (i == a) v = token;
        P.out_tokens[(long)r * B + i] = v;
    }
    if (threadIdx.x == 0) {
        P.accept_len[r] = a;
        P.commit_len[r] = a + 1;
        P.bonus_id[r] = token;
        P.new_seq_lens[r] = P.seq_lens[r] + a + 1;
        P.counter[r] = 0;
    }
}

// True in exactly one CTA per row: the last one to finish its chunk.
__device__ bool last_cta_of_row(const Params &P, int r) {
    __shared__ int s_last;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = (atomicAdd(P.counter + r, 1) == P.nchunk - 1);
    __syncthreads();
    if (s_last) __threadfence();
    return s_last != 0;
}

__global__ void __launch_bounds__(kThreads) accept_stochastic_kernel(const Params P) {
    const int r = blockIdx.x / P.nchunk, chunk = blockIdx.x % P.nchunk;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __shared__ int s_a;
    if (warp == 0) {
        bool bad = false;
        const int a = accepted_len(P, r, lane, bad);
        if (lane == 0) {
            s_a = a;
            if (bad && chunk == 0) report_status(P.dev_status, BDSA_DEVICE_OUT_OF_RANGE);
        }
    }
    __syncthreads();
    const int a = s_a;
    const float *prow = P.p + r * P.psr + a * P.psi;
    const float *qrow = (a < P.B - 1) ? P.q + r * P.qsr + a * P.qsi : nullptr;
    const int sb = chunk * P.spc, se = min(P.nseg, sb + P.spc);
    sweep_chunk(P, r, prow, qrow, sb, se, warp, lane);
    if (!last_cta_of_row(P, r)) return;

    __shared__ int s_tok;
    const float u = __ldg(P.u_samp + r);
    if (warp == 0) {
        const int t = resolve_draw(P, r, prow, qrow, u, lane);
        if (lane == 0) s_tok = t;
    }
    __syncthreads();
    if (s_tok < 0 && qrow != nullptr) {
        // residual has no mass (p <= q everywhere in fp32): draw from p instead
        __syncthreads();
        sweep_chunk(P, r, prow, nullptr, 0, P.nseg, warp, lane);
        __threadfence_block();
        __syncthreads();
        if (warp == 0) {
            const int t = resolve_draw(P, r, prow, nullptr, u, lane);
            if (lane == 0) s_tok = t;
        }
        __syncthreads();
    }
    write_outputs(P, r, a, s_tok);
}

__device__ __forceinline__ void better(float &bv, int &bi, float v, int i) {
    if (v > bv || (v == bv && i < bi)) {
        bv = v;
        bi = i;
    }
}

__global__ void __launch_bounds__(kThreads) accept_greedy_kernel(const Params P) {
    const int r = blockIdx.x / P.nchunk, chunk = blockIdx.x % P.nchunk;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __shared__ float s_v[kWarps];
    __shared__ int s_i[kWarps];
    const int sb = chunk * P.spc, se = min(P.nseg, sb + P.spc);
    for (int i = 0; i < P.B; ++i) {
        const float *prow = P.p + r * P.psr + (long)i * P.psi;
        float bv = -INFINITY;
        int bi = INT_MAX;
        for (int seg = sb + warp; seg < se; seg += kWarps) {
            float w[8];
            const long e0 = (long)seg * kSeg + lane * 8;
            load_weights(prow, nullptr, e0, P.V, w);
#pragma unroll
            for (int e = 0; e < 8; ++e)
                if (e0 + e < P.V) better(bv, bi, w[e], (int)(e0 + e));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            better(bv, bi, ov, oi);
        }
        if (lane == 0) {
            s_v[warp] = bv;
            s_i[warp] = bi;
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            for (int w = 1; w < kWarps; ++w) better(bv, bi, s_v[w], s_i[w]);
            const long o = ((long)r * P.B + i) * P.nchunk + chunk;
            P.am_val[o] = bv;
            P.am_idx[o] = bi;
        }
        __syncthreads();
    }
    if (!last_cta_of_row(P, r)) return;
    __shared__ int s_tp[64];
    for (int i = threadIdx.x; i < P.B; i += blockDim.x) {
        float bv = -INFINITY;
        int bi = INT_MAX;
        for (int c = 0; c < P.nchunk; ++c) {
            const long o = ((long)r * P.B + i) * P.nchunk + c;
            better(bv, bi, __ldcg(P.am_val + o), __ldcg(P.am_idx + o));
        }
        s_tp[i] = (bi == INT_MAX) ? 0 : bi;
    }
    __syncthreads();
    __shared__ int s_a;
    if (threadIdx.x == 0) {
        int a = 0;
        while (a < P.B - 1 && P.block_ids[(long)r * P.B + a + 1] == s_tp[a]) ++a;
        s_a = a;
    }
    __syncthreads();
    write_outputs(P, r, s_a, s_tp[s_a]);
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

AcceptPlan accept_plan(int bs, int B, int V, int num_sms) {
    AcceptPlan p;
    p.nseg = (V + kSeg - 1) / kSeg;
    long nchunk = bs > 0 ? (2L * num_sms + bs - 1) / bs : 1;
    const long cap = (p.nseg + 7) / 8;  // at least 8 segments (2048 elements) per CTA
    if (nchunk > cap) nchunk = cap;
    if (nchunk < 1) nchunk = 1;
    const long spc = (p.nseg + nchunk - 1) / nchunk;
    nchunk = (p.nseg + spc - 1) / spc;
    p.nchunk = (int)nchunk;
    p.workspace = align256((size_t)bs * sizeof(int32_t)) +
                  align256((size_t)bs * p.nseg * sizeof(double)) +
                  2 * align256((size_t)bs * B * p.nchunk * 4);
    return p;
}

int launch_spec_accept(const AcceptArgs &a, cudaStream_t stream) {
    if (a.bs == 0) return BDSA_OK;
    const AcceptPlan plan = accept_plan(a.bs, a.B, a.V, a.num_sms);
    if (a.workspace == nullptr || a.workspace_bytes < plan.workspace)
        return BDSA_WORKSPACE_TOO_SMALL;
    Params P;
    P.block_ids = a.block_ids;
    P.p = a.p;
    P.q = a.q;
    P.psr = a.psr;
    P.psi = a.psi;
    P.qsr = a.qsr;
    P.qsi = a.qsi;
    P.u_acc = a.u_acc;
    P.u_samp = a.u_samp;
    P.seq_lens = a.seq_lens;
    P.bs = a.bs;
    P.B = a.B;
    P.V = a.V;
    P.nchunk = plan.nchunk;
    P.nseg = plan.nseg;
    P.spc = (plan.nseg + plan.nchunk - 1) / plan.nchunk;
    P.accept_len = a.accept_len;
    P.commit_len = a.commit_len;
    P.out_tokens = a.out_tokens;
    P.bonus_id = a.bonus_id;
    P.new_seq_lens = a.new_seq_lens;
    P.dev_status = a.dev_status;
    char *ws = static_cast<char *>(a.workspace);
    P.counter = reinterpret_cast<int32_t *>(ws);
    ws += align256((size_t)a.bs * sizeof(int32_t));
    P.seg_sum = reinterpret_cast<double *>(ws);
    ws += align256((size_t)a.bs * plan.nseg * sizeof(double));
    P.am_val = reinterpret_cast<float *>(ws);
    ws += align256((size_t)a.bs * a.B * plan.nchunk * 4);
    P.am_idx = reinterpret_cast<int32_t *>(ws);
    if (cudaMemsetAsync(P.counter, 0, (size_t)a.bs * sizeof(int32_t), stream) != cudaSuccess)
        return BDSA_CUDA_ERROR;
    const long nblocks = (long)plan.nchunk * a.bs;
    if (nblocks > 0x7fffffffL) return BDSA_UNSUPPORTED;
    const unsigned grid = (unsigned)nblocks;
    if (a.q != nullptr)
        accept_stochastic_kernel<<<grid, kThreads, 0, stream>>>(P);
    else
        accept_greedy_kernel<<<grid, kThreads, 0, stream>>>(P);
    return cudaGetLastError() == cudaSuccess ? BDSA_OK : BDSA_CUDA_ERROR;
}

}  // namespace bdsa
