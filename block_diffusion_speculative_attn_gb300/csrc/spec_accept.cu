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
// (B - 1 gathered probability pairs) and sweeps its chunk once with 16-byte
// loads, reducing each segment to a float-float total (error-free TwoSum
// sums, about 48 significant bits, all in fp32 arithmetic).  One CTA per row
// then scans the segment totals, re-reads the one segment that holds the
// crossing point and resolves the token to a single index.  Cumulative sums
// stay within ~1e-12 relative of the exact sums, far inside the 1e-9 band
// within which the fp64 oracle flags a draw as order-dependent.
//
// Two ways to bring a row's chunks together:
//   cluster path (nseg <= kClusterMaxSeg): the row's CTAs form one thread-block
//     cluster; each writes its segment totals (or greedy chunk maxima) straight
//     into the shared memory of the cluster's first CTA, a hardware cluster
//     barrier publishes them and that CTA resolves.  No global scratch, no
//     atomics, no memset.
//   global path (larger vocabularies): totals go to the caller's workspace and
//     the last CTA of the row to finish (atomic counter, nothing ever waits)
//     resolves.
#include <cuda_runtime.h>
#include <limits.h>

#include <atomic>

#include "bdsa_device.cuh"
#include "bdsa_internal.h"

namespace bdsa {
namespace {

constexpr int kSeg = 256;  // vocabulary elements per segment (32 lanes x 8)
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxB = 64;
// Up to 16 CTAs a cluster: beyond the portable 8, enabled per kernel with
// cudaFuncAttributeNonPortableClusterSizeAllowed.  Against 8: 20.5 -> 18.4 us
// for the Qwen3-8B-shaped stochastic acceptance, 92 -> 80 us greedy.
constexpr int kMaxCluster = 16;
constexpr int kClusterMaxSeg = 8192;   // V <= 2^21 on the cluster path (64 KB of totals)

struct Params {
    const int32_t *block_ids;
    const float *p;
    const float *q;
    int64_t psr, psi, qsr, qsi;
    const float *u_acc;
    const float *u_samp;
    const int32_t *seq_lens;
    int bs, B, V, nchunk, nseg, spc;
    int prefetch;  // bulk-prefetch each chunk into L2 (grids smaller than the GPU)
    int32_t *accept_len, *commit_len, *out_tokens, *bonus_id, *new_seq_lens;
    float2 *seg_tot;   // global path: [bs, nseg] float-float totals
    int32_t *counter;  // global path: [bs], zeroed before the launch
    float *am_val;     // global path, greedy: [bs, B, nchunk]
    int32_t *am_idx;   // global path, greedy: [bs, B, nchunk]
    int32_t *dev_status;
};

// ------------------------------------------------------------ cluster helpers
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive_release() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Generic address of the same shared-memory object in cluster CTA `rank`.
template <class T>
__device__ __forceinline__ T *map_to_rank(T *p, uint32_t rank) {
    uint64_t out;
    asm volatile("mapa.u64 %0, %1, %2;"
                 : "=l"(out)
                 : "l"(reinterpret_cast<uint64_t>(p)), "r"(rank));
    return reinterpret_cast<T *>(out);
}

// ------------------------------------------------------------------ weights
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

// --------------------------------------------------------- float-float sums
// Error-free fp32 addition (Knuth's TwoSum): a + b == s + e exactly.
__device__ __forceinline__ float two_sum(float a, float b, float &e) {
    const float s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
    return s;
}

// A float-float value hi + lo (|lo| <= ulp(hi) / 2): about 48 significant bits
// from fp32 arithmetic alone (fp64 throughput on this GPU is a small fraction
// of fp32's).  Stored as float2 {hi, lo}.
__device__ __forceinline__ float2 ff_add(float2 a, float2 b) {
    float e;
    const float s = two_sum(a.x, b.x, e);
    const float lo = __fadd_rn(__fadd_rn(a.y, b.y), e);
    const float hi = __fadd_rn(s, lo);  // renormalise (Fast2Sum, |s| >= |lo|)
    return make_float2(hi, __fsub_rn(lo, __fsub_rn(hi, s)));
}

// Sum of 8 weights as a float-float: a pairwise tree of TwoSums keeps every
// rounding error; only the sum of those tiny errors is rounded.
__device__ __forceinline__ float2 group_sum_ff(const float (&w)[8]) {
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
    const float hi = __fadd_rn(s07, err);
    return make_float2(hi, __fsub_rn(err, __fsub_rn(hi, s07)));
}

__device__ __forceinline__ float2 shfl_xor_ff(float2 v, int o) {
    return make_float2(__shfl_xor_sync(0xffffffffu, v.x, o), __shfl_xor_sync(0xffffffffu, v.y, o));
}
__device__ __forceinline__ float2 shfl_up_ff(float2 v, int o) {
    return make_float2(__shfl_up_sync(0xffffffffu, v.x, o), __shfl_up_sync(0xffffffffu, v.y, o));
}
__device__ __forceinline__ float2 shfl_ff(float2 v, int src) {
    return make_float2(__shfl_sync(0xffffffffu, v.x, src), __shfl_sync(0xffffffffu, v.y, src));
}

// Warp total (butterfly; every lane gets the total).
__device__ __forceinline__ float2 warp_sum_ff(float2 v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = ff_add(v, shfl_xor_ff(v, o));
    return v;
}

// Warp inclusive prefix sum.
__device__ __forceinline__ float2 warp_scan_ff(float2 v, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float2 t = shfl_up_ff(v, o);
        if (lane >= o) v = ff_add(v, t);
    }
    return v;
}

// Warp totals of four values at once: the first two butterfly levels halve
// the number of values a lane carries (each lane sends the half it gives
// away), so four totals cost 12 shuffles and 6 additions instead of 40 and
// 20.  Lane l ends with the total of g[l >> 3].
__device__ __forceinline__ float2 warp_sum4_ff(const float2 (&g)[4], int lane) {
    const bool h16 = (lane & 16) != 0, h8 = (lane & 8) != 0;
    const float2 k0 = ff_add(h16 ? g[2] : g[0], shfl_xor_ff(h16 ? g[0] : g[2], 16));
    const float2 k1 = ff_add(h16 ? g[3] : g[1], shfl_xor_ff(h16 ? g[1] : g[3], 16));
    float2 k = ff_add(h8 ? k1 : k0, shfl_xor_ff(h8 ? k0 : k1, 8));
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) k = ff_add(k, shfl_xor_ff(k, o));
    return k;
}

// a + w for a float-float a and a float w.
__device__ __forceinline__ float2 ff_add_f(float2 a, float w) {
    float e;
    const float s = two_sum(a.x, w, e);
    const float lo = __fadd_rn(a.y, e);
    const float hi = __fadd_rn(s, lo);
    return make_float2(hi, __fsub_rn(lo, __fsub_rn(hi, s)));
}

// u * a for a float u and a float-float a (the product's rounding error from
// one fused multiply-add).
__device__ __forceinline__ float2 ff_mul_f(float2 a, float u) {
    const float p = __fmul_rn(u, a.x);
    const float lo = __fadd_rn(__fmaf_rn(u, a.x, -p), __fmul_rn(u, a.y));
    const float hi = __fadd_rn(p, lo);
    return make_float2(hi, __fsub_rn(lo, __fsub_rn(hi, p)));
}

// a > b for normalised float-float values (hi == fl(hi + lo)): compare the
// high parts, then the low parts.
__device__ __forceinline__ bool ff_gt(float2 a, float2 b) {
    return a.x > b.x || (a.x == b.x && a.y > b.y);
}

// ------------------------------------------------------------ acceptance
// Accepted draft count for row r (stochastic mode), computed by one warp.  The
// draft ids are also left in s_ids[1..B-1] for the output step.
__device__ int accepted_len(const Params &P, int r, int lane, bool &bad_id, int *s_ids) {
    const int B = P.B;
    bool bad_any = false;
    int a = -1;
    for (int base = 1; base < B; base += 32) {
        const int i = base + lane;
        bool rej = false;
        bad_id = false;
        if (i < B) {
            const int d = P.block_ids[(long)r * B + i];
            s_ids[i] = d;
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

// Starts pulling elements [seg_begin * kSeg, seg_end * kSeg) of a row into L2
// with one bulk prefetch (a hint: nothing waits on it), so the whole chunk is
// in flight from DRAM while the warps' own loads work through it.  Used when
// the grid has fewer CTAs than the GPU has SMs: one CTA's own loads then
// cannot keep DRAM busy (with two CTAs an SM the prefetch measured slower).
__device__ __forceinline__ void prefetch_chunk_l2(const float *row, int seg_begin, int seg_end,
                                                  int V) {
    if (row == nullptr || seg_begin >= seg_end) return;
    const long e0 = (long)seg_begin * kSeg, e1 = min((long)seg_end * kSeg, (long)V);
    const uintptr_t a = reinterpret_cast<uintptr_t>(row + e0);
    const uint32_t bytes = (uint32_t)(((e1 - e0) * 4) & ~15L);
    if ((a & 15) != 0 || bytes == 0) return;
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(a), "r"(bytes) : "memory");
}

// Segment totals of segments [seg_begin, seg_end) of the chosen distribution,
// written to tot[seg] (shared memory of this or another cluster CTA, or global
// memory).  Each warp loads U segments before reducing them, so its loads
// overlap; each group of four segments is reduced across the warp together.
constexpr int kUnroll = 4;

template <class PT, int U = kUnroll>
__device__ void sweep_chunk(const PT &P, const float *prow, const float *qrow, int seg_begin,
                            int seg_end, int warp, int lane, float2 *tot) {
    if (P.prefetch && threadIdx.x == 0) {
        prefetch_chunk_l2(prow, seg_begin, seg_end, P.V);
        prefetch_chunk_l2(qrow, seg_begin, seg_end, P.V);
    }
    for (int s0 = seg_begin + warp; s0 < seg_end; s0 += U * kWarps) {
        float w[U][8];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int seg = s0 + u * kWarps;
            if (seg < seg_end) load_weights(prow, qrow, (long)seg * kSeg + lane * 8, P.V, w[u]);
            else {
#pragma unroll
                for (int e = 0; e < 8; ++e) w[u][e] = 0.f;
            }
        }
#pragma unroll
        for (int u0 = 0; u0 + 4 <= U; u0 += 4) {
            float2 g[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) g[k] = group_sum_ff(w[u0 + k]);
            const float2 t = warp_sum4_ff(g, lane);
            const int seg = s0 + (u0 + (lane >> 3)) * kWarps;
            if ((lane & 7) == 0 && seg < seg_end) tot[seg] = t;
        }
#pragma unroll
        for (int u = U & ~3; u < U; ++u) {
            const int seg = s0 + u * kWarps;
            if (seg < seg_end) {
                const float2 t = warp_sum_ff(group_sum_ff(w[u]));
                if (lane == 0) tot[seg] = t;
            }
        }
    }
}

// Segment total `i`: plain load from shared memory, or an L2 load of values
// that other CTAs wrote (global path).
template <bool kShared>
__device__ __forceinline__ float2 load_tot(const float2 *tot, int i) {
    if constexpr (kShared)
        return tot[i];
    else
        return __ldcg(tot + i);
}

// Resolve the draw InvCDF(w, u) from the segment totals with the whole CTA:
// a block-wide scan of the totals finds the segment holding the crossing, then
// warp 0 re-reads that one segment and finds the element.  All comparisons are
// made on float-float values (about 48 significant bits), in fp32 arithmetic.
// Every thread returns the token index (-1 when the weights are all zero).
template <bool kShared, class PT>
__device__ int resolve_draw(const PT &P, const float *prow, const float *qrow, float u,
                            const float2 *tot) {
    __shared__ float2 s_wtot[kWarps];
    __shared__ int s_seg;
    __shared__ float2 s_base;
    __shared__ float2 s_T;
    __shared__ int s_last_pos;
    __shared__ int s_tok;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nseg = P.nseg;
    const int per = (nseg + kThreads - 1) / kThreads;
    const int s0 = min(nseg, tid * per), s1 = min(nseg, s0 + per);
    float2 loc = make_float2(0.f, 0.f);
    for (int q = s0; q < s1; ++q) loc = ff_add(loc, load_tot<kShared>(tot, q));
    // block exclusive scan of the per-thread totals
    const float2 inc = warp_scan_ff(loc, lane);
    if (lane == 31) s_wtot[warp] = inc;
    if (tid == 0) {
        s_seg = INT_MAX;
        s_last_pos = -1;
    }
    __syncthreads();
    // the warps' offsets and the grand total: every warp scans the eight
    // warp totals in its lanes 0-7 (three dependent float-float additions
    // where a loop over the warps took sixteen)
    float2 wt = lane < kWarps ? s_wtot[lane] : make_float2(0.f, 0.f);
#pragma unroll
    for (int o = 1; o < kWarps; o <<= 1) {
        const float2 t = shfl_up_ff(wt, o);
        if (lane >= o) wt = ff_add(wt, t);
    }
    const float2 S = shfl_ff(wt, kWarps - 1);
    float2 wexcl = shfl_ff(wt, warp > 0 ? warp - 1 : 0);
    if (warp == 0) wexcl = make_float2(0.f, 0.f);
    float2 excl = shfl_up_ff(inc, 1);
    if (lane == 0) excl = make_float2(0.f, 0.f);
    excl = ff_add(excl, wexcl);
    if (!(S.x > 0.f)) return -1;  // uniform: every thread sees the same S
    const float2 T = ff_mul_f(S, u);
    // first segment whose cumulative total exceeds T
    float2 run = excl;
    int found = -1;
    int last_pos = -1;
    for (int q = s0; q < s1; ++q) {
        const float2 v = load_tot<kShared>(tot, q);
        if (v.x > 0.f) last_pos = q;
        if (found < 0) {
            const float2 next = ff_add(run, v);
            if (ff_gt(next, T)) found = q;
            else run = next;
        }
    }
    if (found >= 0) atomicMin(&s_seg, found);
    if (last_pos >= 0) atomicMax(&s_last_pos, last_pos);
    __syncthreads();
    if (found >= 0 && found == s_seg) {
        s_base = run;
        s_T = T;
    }
    if (tid == 0 && s_seg == INT_MAX) {
        // rounding fallback: the last segment with positive mass, no crossing in it
        s_seg = s_last_pos;
        s_base = make_float2(0.f, 0.f);
        s_T = make_float2(INFINITY, 0.f);
    }
    __syncthreads();
    if (warp == 0 && s_seg < 0) {
        if (lane == 0) s_tok = -1;
    } else if (warp == 0) {
        const int seg_star = s_seg;
        const float2 base_seg = s_base, Tw = s_T;
        // within the segment: one 8-element group per lane
        float w[8];
        const long e0 = (long)seg_star * kSeg + lane * 8;
        load_weights(prow, qrow, e0, P.V, w);
        const float2 gff = group_sum_ff(w);
        const float2 ginc = warp_scan_ff(gff, lane);
        float2 gexcl = shfl_up_ff(ginc, 1);
        if (lane == 0) gexcl = make_float2(0.f, 0.f);
        const float2 gb = ff_add(base_seg, gexcl);
        const unsigned cross = __ballot_sync(0xffffffffu, ff_gt(ff_add(gb, gff), Tw));
        int lane_star;
        bool use_cross;
        if (cross != 0u) {
            lane_star = __ffs(cross) - 1;
            use_cross = true;
        } else {
            const unsigned pos = __ballot_sync(0xffffffffu, gff.x > 0.f);
            lane_star = pos ? 31 - __clz(pos) : 0;
            use_cross = false;
        }
        float2 cum = shfl_ff(gb, lane_star);
        if (lane == lane_star) {
            int k = -1, lp = -1;
            for (int e = 0; e < 8; ++e) {
                if (w[e] > 0.f) lp = e;
                cum = ff_add_f(cum, w[e]);
                if (use_cross && ff_gt(cum, Tw)) {
                    k = e;
                    break;
                }
            }
            if (k < 0) k = lp;
            if (k >= 0) k += (int)e0;
            s_tok = k;
        }
    }
    __syncthreads();
    return s_tok;
}

// ids[i] holds block_ids[r, i] for 1 <= i < B (shared memory).
__device__ void write_outputs(const Params &P, int r, int a, int token, const int *ids,
                              int seq_len) {
    const int B = P.B;
    for (int i = threadIdx.x; i < B; i += blockDim.x) {
        int32_t v = -1;
        if (i < a) v = ids[i + 1];
        else if (i == a) v = token;
        P.out_tokens[(long)r * B + i] = v;
    }
    if (threadIdx.x == 0) {
        P.accept_len[r] = a;
        P.commit_len[r] = a + 1;
        P.bonus_id[r] = token;
        P.new_seq_lens[r] = seq_len + a + 1;
    }
}

// Global path: true in exactly one CTA per row, the last one to finish its
// chunk; that CTA also re-arms the row's counter for the next call.
__device__ bool last_cta_of_row(const Params &P, int r) {
    __shared__ int s_last;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = (atomicAdd(P.counter + r, 1) == P.nchunk - 1);
    __syncthreads();
    if (s_last) {
        __threadfence();
        if (threadIdx.x == 0) P.counter[r] = 0;
    }
    return s_last != 0;
}

// One CTA per (row, chunk); on the cluster path the row's CTAs are one
// cluster (cluster rank == chunk for a 1-D grid of whole clusters).
template <bool kCluster>
__global__ void __launch_bounds__(kThreads) accept_stochastic_kernel(const Params P) {
    grid_dependency_wait();  // the previous kernel's writes (launched with PDL)
    const int r = blockIdx.x / P.nchunk, chunk = blockIdx.x % P.nchunk;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    extern __shared__ float2 s_tot[];  // cluster path: [nseg] totals, used in chunk 0
    __shared__ int s_ids[kMaxB];
    __shared__ int s_a;
    __shared__ float s_u;
    __shared__ int s_sl;
    // First phase of the cluster barrier: once it completes, every CTA of the
    // row has started, so its shared memory may be written.
    if constexpr (kCluster) cluster_arrive_relaxed();
    if (warp == 0) {
        bool bad = false;
        const int a = accepted_len(P, r, lane, bad, s_ids);
        if (lane == 0) {
            s_a = a;
            if (bad && chunk == 0) report_status(P.dev_status, BDSA_DEVICE_OUT_OF_RANGE);
        }
    } else if (warp == 1 && lane == 0) {
        s_u = __ldg(P.u_samp + r);
        s_sl = __ldg(P.seq_lens + r);
    }
    __syncthreads();
    const int a = s_a;
    const float *prow = P.p + r * P.psr + a * P.psi;
    const float *qrow = (a < P.B - 1) ? P.q + r * P.qsr + a * P.qsi : nullptr;
    const int sb = chunk * P.spc, se = min(P.nseg, sb + P.spc);
    float2 *tot;
    if constexpr (kCluster) {
        cluster_wait_acquire();
        tot = map_to_rank(s_tot, 0);
    } else {
        tot = P.seg_tot + (long)r * P.nseg;
    }
    sweep_chunk(P, prow, qrow, sb, se, warp, lane, tot);
    if constexpr (kCluster) {
        cluster_arrive_release();
        cluster_wait_acquire();
        if (chunk != 0) return;
        tot = s_tot;
    } else {
        if (!last_cta_of_row(P, r)) return;
    }
    const float u = s_u;
    int tok = resolve_draw<kCluster>(P, prow, qrow, u, tot);
    if (tok < 0 && qrow != nullptr) {
        // residual has no mass (p <= q everywhere in fp32): draw from p instead
        __syncthreads();
        sweep_chunk(P, prow, nullptr, 0, P.nseg, warp, lane, tot);
        __syncthreads();
        tok = resolve_draw<kCluster>(P, prow, nullptr, u, tot);
    }
    write_outputs(P, r, a, tok, s_ids, s_sl);
}

__device__ __forceinline__ void better(float &bv, int &bi, float v, int i) {
    if (v > bv || (v == bv && i < bi)) {
        bv = v;
        bi = i;
    }
}

// Greedy: every CTA finds, for each block slot i, the argmax of p[r, i] over
// its chunk (warps run through the slots independently, kUnroll segments in
// flight); the resolving CTA combines the chunks and walks the block.
template <bool kCluster>
__global__ void __launch_bounds__(kThreads) accept_greedy_kernel(const Params P) {
    grid_dependency_wait();  // the previous kernel's writes (launched with PDL)
    const int r = blockIdx.x / P.nchunk, chunk = blockIdx.x % P.nchunk;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int B = P.B, C = P.nchunk;
    __shared__ float s_wv[kWarps][kMaxB];
    __shared__ int s_wi[kWarps][kMaxB];
    __shared__ float s_cv[kMaxB * kMaxCluster];  // cluster path: [i][chunk], used in chunk 0
    __shared__ int s_ci[kMaxB * kMaxCluster];
    __shared__ int s_ids[kMaxB];
    __shared__ int s_tp[kMaxB];
    __shared__ int s_sl;
    if constexpr (kCluster) cluster_arrive_relaxed();
    for (int i = threadIdx.x; i < B; i += kThreads) s_ids[i] = P.block_ids[(long)r * B + i];
    if (threadIdx.x == 0) s_sl = __ldg(P.seq_lens + r);
    const int sb = chunk * P.spc, se = min(P.nseg, sb + P.spc);
    for (int i = 0; i < B; ++i) {
        const float *prow = P.p + r * P.psr + (long)i * P.psi;
        float bv = -INFINITY;
        int bi = INT_MAX;
        for (int s0 = sb + warp; s0 < se; s0 += kUnroll * kWarps) {
            float w[kUnroll][8];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int seg = s0 + u * kWarps;
                if (seg < se) load_weights(prow, nullptr, (long)seg * kSeg + lane * 8, P.V, w[u]);
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const long e0 = (long)(s0 + u * kWarps) * kSeg + lane * 8;
                if (s0 + u * kWarps < se) {
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        if (e0 + e < P.V) better(bv, bi, w[u][e], (int)(e0 + e));
                }
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            better(bv, bi, ov, oi);
        }
        if (lane == 0) {
            s_wv[warp][i] = bv;
            s_wi[warp][i] = bi;
        }
    }
    __syncthreads();
    float *cv;
    int *ci;
    if constexpr (kCluster) {
        cluster_wait_acquire();
        cv = map_to_rank(s_cv, 0);
        ci = map_to_rank(s_ci, 0);
    }
    for (int i = threadIdx.x; i < B; i += kThreads) {
        float bv = -INFINITY;
        int bi = INT_MAX;
        for (int w = 0; w < kWarps; ++w) better(bv, bi, s_wv[w][i], s_wi[w][i]);
        if constexpr (kCluster) {
            cv[i * C + chunk] = bv;
            ci[i * C + chunk] = bi;
        } else {
            const long o = ((long)r * B + i) * C + chunk;
            P.am_val[o] = bv;
            P.am_idx[o] = bi;
        }
    }
    if constexpr (kCluster) {
        cluster_arrive_release();
        cluster_wait_acquire();
        if (chunk != 0) return;
    } else {
        if (!last_cta_of_row(P, r)) return;
    }
    for (int i = threadIdx.x; i < B; i += kThreads) {
        float bv = -INFINITY;
        int bi = INT_MAX;
        for (int c = 0; c < C; ++c) {
            if constexpr (kCluster) {
                better(bv, bi, s_cv[i * C + c], s_ci[i * C + c]);
            } else {
                const long o = ((long)r * B + i) * C + c;
                better(bv, bi, __ldcg(P.am_val + o), __ldcg(P.am_idx + o));
            }
        }
        s_tp[i] = (bi == INT_MAX) ? 0 : bi;
    }
    __syncthreads();
    __shared__ int s_a;
    if (threadIdx.x == 0) {
        int a = 0;
        while (a < B - 1 && s_ids[a + 1] == s_tp[a]) ++a;
        s_a = a;
    }
    __syncthreads();
    write_outputs(P, r, s_a, s_tp[s_a], s_ids, s_sl);
}

// ------------------------------------------------------------ I-DLM round
// "From DFlash to dLLM Self-Spec (IV)", sections 4.3 and 4.3.1 (Block-N
// round: the specs carried from the previous round's MASK slots are verified
// left to right against the causal view, a rejection is corrected from the
// residual, a fully verified block draws its bonus and N-1 new specs from the
// MASK slots, a cold start draws one clean token and N-1 specs) and 4.6 (the
// KV rows to keep and the request's advance).  Slot j's distribution p[j]
// predicts slot j + 1.
struct IdlmParams {
    const int32_t *block_ids;  // [bs, 2N-1]
    const int32_t *mode;       // [bs]: 1 verify, 0 cold start
    const float *p;
    const float *q;            // previous round's p rows
    int64_t psr, psi, qsr, qsi;
    const int32_t *q_slot;     // [bs]: q row of spec_0
    const float *u_acc;        // [bs, N-1]
    const float *u_samp;       // [bs, N]: the anchor's, then spec'_j's
    const int32_t *seq_lens;
    int bs, N, V, nchunk, nseg, spc;
    int prefetch;
    int32_t *accept_len, *n_out, *out_tokens, *next_mode, *next_pending, *next_specs,
        *next_q_slot, *new_seq_lens, *kv_keep;
    int32_t *dev_status;
};

// Leading verified specs of row r (one warp, N - 1 <= 31 specs: one lane
// each); spec ids are left in s_ids[1..N-1].  The row's mode, q slot, spec
// ids and uniforms are loaded together, then the p / q pairs: two dependent
// global round trips.  An id outside the vocabulary is a rejection and a data
// error.  Returns -1 for a row that does not verify (cold start).
__device__ int idlm_accepted(const IdlmParams &P, int r, int lane, int &m_out, int &qs_out,
                             bool &bad, int *s_ids) {
    const int N = P.N, blk = 2 * N - 1;
    const bool has = lane < N - 1;
    const int m = __ldg(P.mode + r);
    const int qs = __ldg(P.q_slot + r);
    const int s = has ? __ldg(P.block_ids + (long)r * blk + 1 + lane) : 0;
    const float u = has ? __ldg(P.u_acc + (long)r * (N - 1) + lane) : 0.f;
    m_out = m;
    qs_out = qs;
    bad = false;
    if (!(m == 1 && qs >= 0 && qs <= N)) return -1;
    bool rej = false, bad_id = false;
    if (has) {
        s_ids[1 + lane] = s;
        if (s < 0 || s >= P.V) {
            rej = bad_id = true;
        } else {
            const float pv = __ldg(P.p + r * P.psr + (long)lane * P.psi + s);
            const float qv = __ldg(P.q + r * P.qsr + (long)(qs + lane) * P.qsi + s);
            rej = (qv == 0.f) ? !(pv > 0.f) : !(u < fminf(1.f, __fdiv_rn(pv, qv)));
        }
    }
    bad = __any_sync(0xffffffffu, bad_id);
    const unsigned msk = __ballot_sync(0xffffffffu, rej);
    return msk != 0u ? __ffs(msk) - 1 : N - 1;
}

// One thread-block cluster per (row r, draw j), its CTAs = the vocabulary
// chunks.  Draw 0 is the anchor (correction, bonus or clean token) and writes
// the row's outputs; draw j > 0 is spec'_{j-1}, drawn only when the next round
// verifies.
__global__ void __launch_bounds__(kThreads) idlm_accept_kernel(const IdlmParams P) {
    grid_dependency_wait();  // the previous kernel's writes (launched with PDL)
    // Draw-major: the clusters of draw 0 (every request's anchor draw) have
    // the lowest block indices and are scheduled first; the later draws,
    // which most verifying requests do not need (their CTAs find that out
    // and exit), come after.  Against request-major: 29.9 -> 27.0 us at 32
    // requests, N = 8, V = 151936 (A/B means).
    const int unit = blockIdx.x / P.nchunk, chunk = blockIdx.x % P.nchunk;
    const int r = unit % P.bs, j = unit / P.bs;
    const int N = P.N;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    extern __shared__ float2 s_tot[];  // [nseg] totals, used in chunk 0
    __shared__ int s_ids[kMaxB];
    __shared__ int s_a, s_verify, s_qs, s_sl;
    __shared__ float s_u;
    cluster_arrive_relaxed();
    if (warp == 0) {
        int m, qs;
        bool bad;
        const int av = idlm_accepted(P, r, lane, m, qs, bad, s_ids);
        const bool verify = av >= 0;
        const int a = verify ? av : 0;
        if (lane == 0) {
            s_a = a;
            s_verify = verify;
            s_qs = qs;
            const bool bad_state = (m != 0 && m != 1) || (m == 1 && !verify);
            if (chunk == 0 && j == 0 && (bad || bad_state))
                report_status(P.dev_status, BDSA_DEVICE_OUT_OF_RANGE);
        }
    } else if (warp == 1 && lane == 0) {
        s_u = __ldg(P.u_samp + (long)r * N + j);
        s_sl = __ldg(P.seq_lens + r);
    }
    __syncthreads();
    const int a = s_a;
    const bool verify = s_verify != 0;
    int slot = -1;  // p row this draw samples
    const float *qrow = nullptr;
    if (j == 0) {
        if (!verify) {
            slot = 0;
        } else if (a < N - 1) {
            slot = a;
            qrow = P.q + r * P.qsr + (long)(s_qs + a) * P.qsi;
        } else {
            slot = N - 1;
        }
    } else if (!verify) {
        slot = j;
    } else if (a == N - 1) {
        slot = N + j - 1;
    }
    if (slot < 0) {
        // the next round is a cold start: no spec to draw
        cluster_wait_acquire();
        if (chunk == 0 && threadIdx.x == 0) P.next_specs[(long)r * (N - 1) + j - 1] = -1;
        return;
    }
    const float *prow = P.p + r * P.psr + (long)slot * P.psi;
    const int sb = chunk * P.spc, se = min(P.nseg, sb + P.spc);
    cluster_wait_acquire();
    sweep_chunk(P, prow, qrow, sb, se, warp, lane, map_to_rank(s_tot, 0));
    cluster_arrive_release();
    cluster_wait_acquire();
    if (chunk != 0) return;
    const float u = s_u;
    int tok = resolve_draw<true>(P, prow, qrow, u, s_tot);
    if (tok < 0 && qrow != nullptr) {
        // residual has no mass (p <= q everywhere in fp32): draw from p instead
        __syncthreads();
        sweep_chunk(P, prow, nullptr, 0, P.nseg, warp, lane, s_tot);
        __syncthreads();
        tok = resolve_draw<true>(P, prow, nullptr, u, s_tot);
    }
    if (j > 0) {
        if (threadIdx.x == 0) P.next_specs[(long)r * (N - 1) + j - 1] = tok;
        return;
    }
    for (int i = threadIdx.x; i < N; i += kThreads) {
        int32_t v = -1;
        if (i < a) v = s_ids[i + 1];
        else if (i == a) v = tok;
        P.out_tokens[(long)r * N + i] = v;
    }
    if (threadIdx.x == 0) {
        const bool next_verify = !verify || a == N - 1;
        P.accept_len[r] = a;
        P.n_out[r] = a + 1;
        P.next_pending[r] = tok;
        P.next_mode[r] = next_verify ? 1 : 0;
        P.next_q_slot[r] = !verify ? 1 : (a == N - 1 ? N : -1);
        P.kv_keep[r] = a + 1;
        P.new_seq_lens[r] = s_sl + a + 1;
    }
}

// ------------------------------------------------------------ tree verify
// "Unlocking Lossless Speedups in LLMs via Discrete Diffusion", Psi-Spec Tree
// sampler: the drafted token tree is verified in one forward and rejection
// sampling keeps the verifier's distribution.  The tree's tokens are chosen,
// not sampled, so each draft distribution is one-hot: at node n of depth d the
// verifier draws x from p[n] (InvCDF with u[d], or the argmax when greedy); a
// child of n carrying x is accepted and the walk goes on from it, otherwise x
// is emitted (correction, or bonus at a leaf).
struct TreeParams {
    const int32_t *block_ids, *parent, *seq_lens;
    const float *p;
    int64_t psr, psn;
    const float *u;  // [bs, B] by depth; null = greedy
    int bs, B, V, nchunk, nseg, spc;
    int prefetch;
    int32_t *accept_len, *path, *out_tokens, *bonus_id, *new_seq_lens;
    int32_t *dev_status;
};

// Each step of the walk is one dependent sweep, so a step's latency is what
// counts: four segments in flight a warp, reduced across the warp together
// (two rounds for a chunk of up to 64 segments; five a warp measured 49.2
// against 47.1 us at the Qwen3-8B shape), with registers for two CTAs an SM
// so that every request's cluster is resident at once.
constexpr int kTreeMaxCluster = kMaxCluster;
constexpr int kTreeUnroll = 4;
constexpr int kTreeMaxNodes = BDSA_TREE_MAX_NODES;

// One thread-block cluster per request, its CTAs the vocabulary chunks.  Each
// step of the walk sweeps p[n] (segment totals, or chunk maxima when greedy,
// into the first CTA's shared memory), the first CTA resolves x and finds the
// child, and writes the next node into every CTA of the cluster; two cluster
// barriers a step.  The walk ends within B steps (a child's index exceeds its
// parent's).
__global__ void __launch_bounds__(kThreads, 2) tree_accept_kernel(const TreeParams P) {
    grid_dependency_wait();  // the previous kernel's writes (launched with PDL)
    const int r = blockIdx.x / P.nchunk, chunk = blockIdx.x % P.nchunk;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int B = P.B;
    extern __shared__ float2 s_tot[];  // [nseg], used in chunk 0
    __shared__ int s_ids[kTreeMaxNodes], s_par[kTreeMaxNodes], s_path[kTreeMaxNodes],
        s_tok[kTreeMaxNodes];
    __shared__ float s_cv[kTreeMaxCluster];
    __shared__ int s_ci[kTreeMaxCluster];
    __shared__ float s_wv[kWarps];
    __shared__ int s_wi[kWarps];
    __shared__ int s_next, s_x, s_child;
    if (chunk == 0) {
        for (int i = tid; i < B; i += kThreads) {
            s_ids[i] = __ldg(P.block_ids + (long)r * B + i);
            const int pi = __ldg(P.parent + (long)r * B + i);
            const bool ok = i == 0 ? pi == -1 : (pi >= 0 && pi < i);
            if (!ok) report_status(P.dev_status, BDSA_DEVICE_OUT_OF_RANGE);
            s_par[i] = (i > 0 && ok) ? pi : -1;
            s_path[i] = -1;
            s_tok[i] = -1;
        }
        if (tid == 0) s_path[0] = 0;
    }
    // every CTA of the cluster has started: its shared memory may be written
    cluster_arrive_relaxed();
    cluster_wait_acquire();
    const bool greedy = P.u == nullptr;
    const int sb = chunk * P.spc, se = min(P.nseg, sb + P.spc);
    int n = 0, depth = 0;
    for (int step = 0; step < B; ++step) {
        const float *prow = P.p + r * P.psr + (long)n * P.psn;
        if (!greedy) {
            sweep_chunk<TreeParams, kTreeUnroll>(P, prow, nullptr, sb, se, warp, lane,
                                                 map_to_rank(s_tot, 0));
        } else {
            float bv = -INFINITY;
            int bi = INT_MAX;
            for (int s0 = sb + warp; s0 < se; s0 += kTreeUnroll * kWarps) {
                float w[kTreeUnroll][8];
#pragma unroll
                for (int uu = 0; uu < kTreeUnroll; ++uu) {
                    const int seg = s0 + uu * kWarps;
                    if (seg < se) load_weights(prow, nullptr, (long)seg * kSeg + lane * 8, P.V, w[uu]);
                }
#pragma unroll
                for (int uu = 0; uu < kTreeUnroll; ++uu) {
                    const long e0 = (long)(s0 + uu * kWarps) * kSeg + lane * 8;
                    if (s0 + uu * kWarps < se) {
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            if (e0 + e < P.V) better(bv, bi, w[uu][e], (int)(e0 + e));
                    }
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
                const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
                better(bv, bi, ov, oi);
            }
            if (lane == 0) {
                s_wv[warp] = bv;
                s_wi[warp] = bi;
            }
            __syncthreads();
            if (tid == 0) {
                for (int w = 1; w < kWarps; ++w) better(bv, bi, s_wv[w], s_wi[w]);
                *map_to_rank(&s_cv[chunk], 0) = bv;
                *map_to_rank(&s_ci[chunk], 0) = bi;
            }
        }
        cluster_arrive_release();
        cluster_wait_acquire();
        if (chunk == 0) {
            int x;
            if (!greedy) {
                x = resolve_draw<true>(P, prow, nullptr, __ldg(P.u + (long)r * B + depth), s_tot);
            } else {
                if (tid == 0) {
                    float bv = -INFINITY;
                    int bi = INT_MAX;
                    for (int c = 0; c < P.nchunk; ++c) better(bv, bi, s_cv[c], s_ci[c]);
                    s_x = (bi == INT_MAX) ? 0 : bi;
                }
                __syncthreads();
                x = s_x;
            }
            // the lowest-index child of n carrying x, searched by the whole CTA
            if (tid == 0) s_child = INT_MAX;
            __syncthreads();
            for (int c = n + 1 + tid; c < B; c += kThreads)
                if (s_par[c] == n && s_ids[c] == x) atomicMin(&s_child, c);
            __syncthreads();
            if (tid == 0) {
                const int child = s_child == INT_MAX ? -1 : s_child;
                s_tok[depth] = x;
                if (child >= 0) s_path[depth + 1] = child;
                for (int rk = 0; rk < P.nchunk; ++rk) *map_to_rank(&s_next, (uint32_t)rk) = child;
            }
        }
        cluster_arrive_release();
        cluster_wait_acquire();
        const int next = s_next;
        if (next < 0) break;
        n = next;
        ++depth;
    }
    if (chunk != 0) return;
    for (int i = tid; i < B; i += kThreads) {
        P.path[(long)r * B + i] = s_path[i];
        P.out_tokens[(long)r * B + i] = s_tok[i];
    }
    if (tid == 0) {
        P.accept_len[r] = depth;
        P.bonus_id[r] = s_tok[depth];
        P.new_seq_lens[r] = __ldg(P.seq_lens + r) + depth + 1;
    }
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Clusters above the portable 8 CTAs need an opt-in per kernel (set once).
bool allow_big_clusters(const void *fn, std::atomic<int> &done) {
    if (done.load(std::memory_order_acquire)) return true;
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
        cudaSuccess)
        return false;
    done.store(1, std::memory_order_release);
    return true;
}

}  // namespace

AcceptPlan accept_plan(int bs, int B, int V, int num_sms) {
    AcceptPlan p;
    p.nseg = (V + kSeg - 1) / kSeg;
    p.cluster = p.nseg <= kClusterMaxSeg;
    // about two CTAs per SM over the whole batch, at least 8 segments (2048
    // elements) per CTA, and at most a 16-CTA cluster per row on the
    // cluster path
    long nchunk = bs > 0 ? (2L * num_sms + bs - 1) / bs : 1;
    const long cap = (p.nseg + 7) / 8;
    if (nchunk > cap) nchunk = cap;
    if (p.cluster && nchunk > kMaxCluster) nchunk = kMaxCluster;
    if (nchunk < 1) nchunk = 1;
    const long spc = (p.nseg + nchunk - 1) / nchunk;
    if (!p.cluster) nchunk = (p.nseg + spc - 1) / spc;
    p.nchunk = (int)nchunk;
    p.spc = (int)spc;
    p.prefetch = (long)p.nchunk * bs < num_sms;
    p.workspace = p.cluster ? 0
                            : align256((size_t)bs * sizeof(int32_t)) +
                                  align256((size_t)bs * p.nseg * sizeof(float2)) +
                                  2 * align256((size_t)bs * B * p.nchunk * 4);
    return p;
}

int launch_idlm_accept(const IdlmArgs &a, cudaStream_t stream) {
    if (a.bs == 0) return BDSA_OK;
    // Many (row, draw) clusters of a round find nothing to draw and exit: the
    // chunks are sized for about eight CTAs an SM over all of them (against
    // four: 36.8 -> 30.7 us at 32 requests, N = 8, V = 151936, five chunks a
    // row; eight, ten and sixteen chunks a row measured slower).
    const AcceptPlan plan = accept_plan(a.bs * a.N, 2 * a.N - 1, a.V, 4 * a.num_sms);
    if (!plan.cluster) return BDSA_UNSUPPORTED;
    IdlmParams P;
    P.block_ids = a.block_ids;
    P.mode = a.mode;
    P.p = a.p;
    P.q = a.q;
    P.psr = a.psr;
    P.psi = a.psi;
    P.qsr = a.qsr;
    P.qsi = a.qsi;
    P.q_slot = a.q_slot;
    P.u_acc = a.u_acc;
    P.u_samp = a.u_samp;
    P.seq_lens = a.seq_lens;
    P.bs = a.bs;
    P.N = a.N;
    P.V = a.V;
    P.nchunk = plan.nchunk;
    P.nseg = plan.nseg;
    P.spc = plan.spc;
    P.prefetch = plan.prefetch;
    P.accept_len = a.accept_len;
    P.n_out = a.n_out;
    P.out_tokens = a.out_tokens;
    P.next_mode = a.next_mode;
    P.next_pending = a.next_pending;
    P.next_specs = a.next_specs;
    P.next_q_slot = a.next_q_slot;
    P.new_seq_lens = a.new_seq_lens;
    P.kv_keep = a.kv_keep;
    P.dev_status = a.dev_status;
    const long nblocks = (long)plan.nchunk * a.bs * a.N;
    if (nblocks > 0x7fffffffL) return BDSA_UNSUPPORTED;
    const size_t smem = (size_t)plan.nseg * sizeof(float2);
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(idlm_accept_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
        return BDSA_CUDA_ERROR;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)nblocks);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)plan.nchunk;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // may start while the previous kernel in the stream finishes; the kernel
    // waits for it (griddepcontrol.wait) before its first global read
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    static std::atomic<int> big_ok{0};
    if (plan.nchunk > 8 &&
        !allow_big_clusters(reinterpret_cast<const void *>(&idlm_accept_kernel), big_ok))
        return BDSA_CUDA_ERROR;
    return cudaLaunchKernelEx(&cfg, idlm_accept_kernel, P) == cudaSuccess ? BDSA_OK
                                                                          : BDSA_CUDA_ERROR;
}

int launch_tree_accept(const TreeArgs &a, cudaStream_t stream) {
    if (a.bs == 0) return BDSA_OK;
    const AcceptPlan plan = accept_plan(a.bs, a.B, a.V, a.num_sms);
    if (!plan.cluster) return BDSA_UNSUPPORTED;

    TreeParams P;
    P.block_ids = a.block_ids;
    P.parent = a.parent;
    P.seq_lens = a.seq_lens;
    P.p = a.p;
    P.psr = a.psr;
    P.psn = a.psn;
    P.u = a.u;
    P.bs = a.bs;
    P.B = a.B;
    P.V = a.V;
    P.nchunk = plan.nchunk;
    P.nseg = plan.nseg;
    P.spc = plan.spc;
    P.prefetch = plan.prefetch;
    P.accept_len = a.accept_len;
    P.path = a.path;
    P.out_tokens = a.out_tokens;
    P.bonus_id = a.bonus_id;
    P.new_seq_lens = a.new_seq_lens;
    P.dev_status = a.dev_status;
    const long nblocks = (long)plan.nchunk * a.bs;
    if (nblocks > 0x7fffffffL) return BDSA_UNSUPPORTED;
    const size_t smem = (size_t)plan.nseg * sizeof(float2);
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(tree_accept_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
        return BDSA_CUDA_ERROR;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)nblocks);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)plan.nchunk;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // may start while the previous kernel in the stream finishes; the kernel
    // waits for it (griddepcontrol.wait) before its first global read
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    static std::atomic<int> big_ok{0};
    if (plan.nchunk > 8 &&
        !allow_big_clusters(reinterpret_cast<const void *>(&tree_accept_kernel), big_ok))
        return BDSA_CUDA_ERROR;
    return cudaLaunchKernelEx(&cfg, tree_accept_kernel, P) == cudaSuccess ? BDSA_OK
                                                                          : BDSA_CUDA_ERROR;
}

int launch_spec_accept(const AcceptArgs &a, cudaStream_t stream) {
    if (a.bs == 0) return BDSA_OK;
    AcceptPlan plan = accept_plan(a.bs, a.B, a.V, a.num_sms);
    // Greedy sweeps B rows of p a CTA: on the cluster path (no workspace) it
    // takes twice the chunks (16 against 10 CTAs a row: 80 -> 70 us at the
    // Qwen3-8B shape; the stochastic draw and the tree walk gain nothing or lose).
    if (a.q == nullptr && plan.cluster) plan = accept_plan(a.bs, a.B, a.V, 2 * a.num_sms);
    if (a.workspace_bytes < plan.workspace || (plan.workspace > 0 && a.workspace == nullptr))
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
    P.spc = plan.spc;
    P.prefetch = plan.prefetch;
    P.accept_len = a.accept_len;
    P.commit_len = a.commit_len;
    P.out_tokens = a.out_tokens;
    P.bonus_id = a.bonus_id;
    P.new_seq_lens = a.new_seq_lens;
    P.dev_status = a.dev_status;
    P.seg_tot = nullptr;
    P.counter = nullptr;
    P.am_val = nullptr;
    P.am_idx = nullptr;
    const long nblocks = (long)plan.nchunk * a.bs;
    if (nblocks > 0x7fffffffL) return BDSA_UNSUPPORTED;
    const bool greedy = a.q == nullptr;
    if (plan.cluster) {
        // segment totals of one row live in the first CTA of its cluster
        const size_t smem = greedy ? 0 : (size_t)plan.nseg * sizeof(float2);
        const void *fn = greedy ? reinterpret_cast<const void *>(&accept_greedy_kernel<true>)
                                : reinterpret_cast<const void *>(&accept_stochastic_kernel<true>);
        if (smem > 48 * 1024 &&
            cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
                cudaSuccess)
            return BDSA_CUDA_ERROR;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)nblocks);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = stream;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)plan.nchunk;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        // may start while the previous kernel in the stream finishes; the kernel
        // waits for it (griddepcontrol.wait) before its first global read
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 2;
        static std::atomic<int> big_ok[2] = {{0}, {0}};
        if (plan.nchunk > 8 && !allow_big_clusters(fn, big_ok[greedy ? 1 : 0]))
            return BDSA_CUDA_ERROR;
        const cudaError_t e = greedy ? cudaLaunchKernelEx(&cfg, accept_greedy_kernel<true>, P)
                                     : cudaLaunchKernelEx(&cfg, accept_stochastic_kernel<true>, P);
        return e == cudaSuccess ? BDSA_OK : BDSA_CUDA_ERROR;
    }
    char *ws = static_cast<char *>(a.workspace);
    P.counter = reinterpret_cast<int32_t *>(ws);
    ws += align256((size_t)a.bs * sizeof(int32_t));
    P.seg_tot = reinterpret_cast<float2 *>(ws);
    ws += align256((size_t)a.bs * plan.nseg * sizeof(float2));
    P.am_val = reinterpret_cast<float *>(ws);
    ws += align256((size_t)a.bs * a.B * plan.nchunk * 4);
    P.am_idx = reinterpret_cast<int32_t *>(ws);
    if (cudaMemsetAsync(P.counter, 0, (size_t)a.bs * sizeof(int32_t), stream) != cudaSuccess)
        return BDSA_CUDA_ERROR;
    const unsigned grid = (unsigned)nblocks;
    if (greedy)
        accept_greedy_kernel<false><<<grid, kThreads, 0, stream>>>(P);
    else
        accept_stochastic_kernel<false><<<grid, kThreads, 0, stream>>>(P);
    return cudaGetLastError() == cudaSuccess ? BDSA_OK : BDSA_CUDA_ERROR;
}

}  // namespace bdsa
