// kv_materialize.cu -- the draft KV of the committed prefix, for sm_103a.
//
// "From DFlash to dLLM Self-Spec (II): SGLang Spec V2", section 2.2.6 and the
// DFlash engineering notes: after verify, the target hidden states of every
// request's committed rows are projected into each draft layer's K and V, K
// gets its RMS norm and RoPE, and both are written into the draft KV pool at
// the verify step's cache slots.  Per committed row x, layer l, KV head h:
//   k = W_K[l, h] x,  v = W_V[l, h] x           (bf16 in, fp32 accumulate)
//   kn = k / sqrt(mean(k^2) + eps) * g[l]
//   ko[d] = kn[d] c - kn[d + D/2] s,  ko[d + D/2] = kn[d + D/2] c + kn[d] s
//   with c = cos[pos][d], s = sin[pos][d] (d < D/2), stored as bf16.
//
// Two launches, chained with programmatic dependent launch:
//   gather  four CTAs per request: copy the committed hidden rows into a
//           dense buffer in the workspace and list (slot, position) per row;
//   project one thread-block cluster of three CTAs per (layer, K or V, head):
//           the CTAs take three ranges of the hidden dimension's 64-element
//           slabs.  Each streams its 128-row slice of the weight block once
//           by TMA (128-byte swizzle) while the rows stream from L2, runs
//           D^T = W X^T on the tensor cores (tcgen05, M = 128 head dims, N =
//           up to 128 rows, fp32 accumulator in TMEM), then the three add
//           their partial sums through distributed shared memory: each CTA
//           sends its partners the row chunks they finish and finishes the
//           others (the sum in a fixed order, K norm, RoPE from the tables,
//           bf16 store at the row's slot).
// The stream is bound by the latency of its TMA loads (about 1 us for a
// 16 KB box under load), so its time follows the slabs a CTA streams: three
// CTAs a head stream 21 or 22 slabs each where two streamed 32, and 240 CTAs
// still fit two an SM.  The weights do not depend on the gather, so the
// projection CTAs start their weight stream before waiting for it.  More than
// 256 committed rows run as several passes over the weights.
#include <cuda.h>
#include <cuda_runtime.h>

#include <utility>

#include "bdsa_device.cuh"
#include "bdsa_internal.h"

namespace bdsa {
namespace {

constexpr int kD = 128;              // head dim (the accumulator's 128 lanes)
constexpr int kSplit = 3;            // CTAs (hidden-dimension ranges) a head: a cluster
constexpr int kBox = 128;            // gathered rows per X box (TMA box, MMA N <= 128)
constexpr int kMaxBoxes = 2;         // boxes per weight stream: 256 rows, 256 TMEM columns
constexpr int kStreamRows = kBox * kMaxBoxes;
constexpr int kTmemCols = kStreamRows;
constexpr int kThreads = 192;        // warps 0-3 epilogue, 4 TMA producer, 5 MMA
constexpr int kEpiThreads = 128;
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
// Each weight slab waits on its row boxes (L2 reads) as well as on DRAM:
// one 128-row box a slab instead of up to four 64-row ones measured 45 -> 37
// us for 77 rows and 142 -> 104 us for 512 (32 rows: 33 -> 35 us).
constexpr int kWStages = 3;
constexpr int kXStages = 3;
constexpr int kWSlab = kD * 128;     // 128 weight rows x 64 hidden elements (16 KB)
constexpr int kXSlab = kBox * 128;   // 128 gathered rows x 64 hidden elements (16 KB)
constexpr int kOffW = 0;
constexpr int kOffX = kOffW + kWStages * kWSlab;
constexpr int kOffBar = kOffX + kXStages * kXSlab;
// barriers
constexpr int kWF = 0;                  // weight stage full
constexpr int kWE = kWF + kWStages;     // weight stage free
constexpr int kXF = kWE + kWStages;     // row box full
constexpr int kXE = kXF + kXStages;     // row box free
constexpr int kAF = kXE + kXStages;     // accumulators of the stream complete
constexpr int kTF = kAF + 1;            // epilogue done with TMEM and T
constexpr int kPR = kTF + 1;            // both partners may take this CTA's chunks (remote arrivals)
constexpr int kRX = kPR + 1;            // both partners' chunks have landed here
constexpr int kEB = kRX + 1;            // the four epilogue warps meet
constexpr int kDR = kEB + 1;            // drain of the MMA warp
constexpr int kNumBars = kDR + 1;
constexpr int kOffMisc = kOffBar + 8 * kNumBars;
constexpr int kSmem = kOffMisc + 64 + 1024;  // + slack to align the base to 1 KB
// The epilogue's receive buffers R[p][i] (partner slot p, chunk i: four
// [32 rows][128 dims] fp32 tiles, 64 KB) alias the weight and row rings: they
// are used only between a stream's last MMA and the next stream's first
// loads.  R[0] doubles as the tile of summed rows.  Two CTAs fit one SM
// (shared memory, 256 TMEM columns each).
constexpr int kRTile = 32 * kD * 4;  // one received chunk
static_assert(kWStages * kWSlab + kXStages * kXSlab >= 4 * kRTile && kOffX == kOffW + kWStages * kWSlab,
              "the receive buffers fit the rings");
static_assert(2 * (kSmem + 1024) <= 228 * 1024, "two CTAs an SM");

struct Params {
    const int32_t *count;      // workspace: number of gathered rows
    const int2 *meta;          // workspace: (slot or -1, position) per gathered row
    const uint16_t *k_norm_w;  // [n_layers, D]
    const float *cos_tab;      // [max_pos, D/2]
    const float *sin_tab;
    uint16_t *k_cache;         // [n_layers, num_slots, Hkv, D]
    uint16_t *v_cache;
    long long num_slots;
    int n_layers, Hkv, H, max_pos;
    float eps;
    int32_t *dev_status;
};

// ------------------------------------------------------------ cluster PTX
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t map_shared_rank(uint32_t addr, uint32_t rank) {
    uint32_t out;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(addr), "r"(rank));
    return out;
}
__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ void mbar_arrive_remote_release(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(
                     cluster_addr)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded like mbar_wait, with cluster-scope acquire (the arrivals come from
// the partner CTA and order its distributed-shared-memory stores).
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity,
                                                  volatile int *abort, int32_t *dev_status) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if (*abort) return false;
        if (global_timer_ns() - t0 > kWaitLimitNs) {
            *abort = 1;
            report_status(dev_status, BDSA_DEVICE_TIMEOUT);
            return false;
        }
    }
}
// Every thread of both CTAs (not required to be converged).
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release;\n\t"
                 "barrier.cluster.wait.acquire;" ::
                     : "memory");
}

__device__ __forceinline__ float bf16_to_f32(uint16_t b) {
    return __uint_as_float(((uint32_t)b) << 16);
}
__device__ __forceinline__ uint32_t pack2_bf16(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// ------------------------------------------------------------------ gather
// Request r's committed rows r*B .. r*B + cl - 1 (cl = commit_len clamped to
// [0, B]) go to dense rows pre .. pre + cl - 1, pre = the committed rows of
// the requests before r.  A row whose slot or position is out of range is
// listed with slot -1 (not written) and reported.  Grid (bs, kGatherParts):
// part p of request r copies the p-th share of its rows' 16-byte pieces, four
// loads in flight a thread.
constexpr int kGatherParts = 4;
constexpr int kGatherThreads = 256;

__global__ void __launch_bounds__(kGatherThreads)
    kvmat_gather_kernel(const uint4 *__restrict__ hidden, const int32_t *__restrict__ commit_len,
                        const int32_t *__restrict__ positions,
                        const int32_t *__restrict__ cache_loc, int bs, int B, int H, int max_pos,
                        long long num_slots, int32_t *count, int2 *meta, uint4 *xc,
                        int32_t *dev_status) {
    // the projection kernel may start streaming weights now
    grid_launch_dependents();
    __shared__ int s_part[kGatherThreads / 32];
    const int r = blockIdx.x, part = blockIdx.y, tid = threadIdx.x;
    int pre = 0;
    for (int q = tid; q < r; q += kGatherThreads) pre += min(max(__ldg(commit_len + q), 0), B);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) pre += __shfl_xor_sync(0xffffffffu, pre, o);
    if ((tid & 31) == 0) s_part[tid >> 5] = pre;
    __syncthreads();
    pre = 0;
#pragma unroll
    for (int w = 0; w < kGatherThreads / 32; ++w) pre += s_part[w];
    const int cl = min(max(__ldg(commit_len + r), 0), B);
    if (part == 0) {
        for (int i = tid; i < cl; i += kGatherThreads) {
            const long row = (long)r * B + i;
            int slot = __ldg(cache_loc + row);
            const int pos = __ldg(positions + row);
            if (slot < 0 || (long long)slot >= num_slots || pos < 0 || pos >= max_pos) {
                report_status(dev_status, BDSA_DEVICE_OUT_OF_RANGE);
                slot = -1;
            }
            meta[pre + i] = make_int2(slot, pos);
        }
        if (r == bs - 1 && tid == 0) *count = pre + cl;
    }
    const long n = (long)cl * (H / 8);  // 16-byte pieces of the request's committed rows
    const long e0 = n * part / kGatherParts, e1 = n * (part + 1) / kGatherParts;
    const uint4 *src = hidden + (long)r * B * (H / 8);
    uint4 *dst = xc + (long)pre * (H / 8);
    constexpr int kU = 4;
    for (long e = e0 + tid; e < e1; e += (long)kU * kGatherThreads) {
        uint4 v[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const long k = e + (long)u * kGatherThreads;
            if (k < e1) v[u] = __ldg(src + k);
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const long k = e + (long)u * kGatherThreads;
            if (k < e1) dst[k] = v[u];
        }
    }
}

// ------------------------------------------------------------------ project
// CTA (cluster rank `rank`) of head `head` = (l * 2 + kv) * Hkv + h handles
// the hidden dimension's 64-element slabs [rank * n / 3, (rank + 1) * n / 3),
// n = H / 64.  Weight stream g covers gathered rows [g * 256, g * 256 + 256)
// as up to two 128-row boxes, box b accumulating into TMEM columns [128 b,
// 128 b + 128).  Its 32-row chunk c is finished by the CTA of rank c % 3; the
// epilogue works in rounds of six chunks (two a CTA), chunk 6 rho + 3 i +
// rank summed into R[0][i].
__global__ void __launch_bounds__(kThreads, 2)
    kvmat_project_kernel(const __grid_constant__ CUtensorMap tm_w,
                         const __grid_constant__ CUtensorMap tm_x, const Params P) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (sbase - raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    auto bar = [&](int i) -> uint32_t { return sbase + kOffBar + 8u * (uint32_t)i; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kOffMisc + 4);

    const uint32_t rank = cluster_rank();
    const int head = (int)(blockIdx.x / kSplit);
    const int Hkv = P.Hkv;
    const int l = head / (2 * Hkv), kv = (head / Hkv) & 1, h = head % Hkv;
    const int nslab_all = P.H / 64;
    const int s_begin = (int)rank * nslab_all / kSplit;
    const int nslab = ((int)rank + 1) * nslab_all / kSplit - s_begin;
    const int k0 = s_begin * 64;
    const int w_row = head * kD;

    if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int s = 0; s < kWStages; ++s) {
            mbar_init(bar(kWF + s), 1);
            mbar_init(bar(kWE + s), 1);
        }
        for (int s = 0; s < kXStages; ++s) {
            mbar_init(bar(kXF + s), 1);
            mbar_init(bar(kXE + s), 1);
        }
        mbar_init(bar(kAF), 1);
        mbar_init(bar(kTF), kEpiThreads / 32);
        mbar_init(bar(kPR), kSplit - 1);
        mbar_init(bar(kRX), (kSplit - 1) * kEpiThreads);
        mbar_init(bar(kEB), kEpiThreads / 32);
        mbar_init(bar(kDR), 1);
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    if (warp == kProducerWarp && lane == 0) {
        tma_prefetch_desc(&tm_w);
        tma_prefetch_desc(&tm_x);
    }
    tc_fence_before();
    // every CTA's barriers exist before any arrives on another's
    cluster_sync_all();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kProducerWarp) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            // the weights do not depend on the gather: start them at once
            const int pre = min(nslab, kWStages);
            for (int s = 0; s < pre; ++s) {
                mbar_arrive_expect_tx(bar(kWF + s), (uint32_t)kWSlab);
                tma_load_2d(sbase + kOffW + s * kWSlab, &tm_w, k0 + s * 64, w_row, bar(kWF + s));
            }
            grid_dependency_wait();
            const int M = __ldcg(P.count);
            const int nstream = (M + kStreamRows - 1) / kStreamRows;
            long issued_w = pre, xb = 0;  // weight slabs / row boxes issued so far
            bool ok = true;
            for (int g = 0; ok && g < nstream; ++g) {
                const int nrows = min(kStreamRows, M - g * kStreamRows);
                const int nbox = (nrows + kBox - 1) / kBox;
                for (int s = 0; ok && s < nslab; ++s) {
                    const long gs = (long)g * nslab + s;
                    if (g > 0 && s == 0) {
                        // the rings double as the epilogue's receive buffers
                        ok = mbar_wait(bar(kTF), (uint32_t)((g - 1) & 1), abort_flag,
                                       P.dev_status);
                        if (!ok) break;
                    }
                    if (gs >= issued_w) {
                        const int st = (int)(gs % kWStages);
                        ok = mbar_wait(bar(kWE + st), (uint32_t)(((gs / kWStages) & 1) ^ 1),
                                       abort_flag, P.dev_status);
                        if (!ok) break;
                        mbar_arrive_expect_tx(bar(kWF + st), (uint32_t)kWSlab);
                        tma_load_2d(sbase + kOffW + st * kWSlab, &tm_w, k0 + s * 64, w_row,
                                    bar(kWF + st));
                        issued_w = gs + 1;
                    }
                    for (int b = 0; b < nbox; ++b, ++xb) {
                        const int xs = (int)(xb % kXStages);
                        ok = mbar_wait(bar(kXE + xs), (uint32_t)(((xb / kXStages) & 1) ^ 1),
                                       abort_flag, P.dev_status);
                        if (!ok) break;
                        mbar_arrive_expect_tx(bar(kXF + xs), (uint32_t)kXSlab);
                        tma_load_2d(sbase + kOffX + xs * kXSlab, &tm_x, k0 + s * 64,
                                    g * kStreamRows + b * kBox, bar(kXF + xs));
                    }
                }
            }
            // drain: the last load into each stage has landed before exit
            for (long i = max(0L, issued_w - kWStages); i < issued_w; ++i)
                mbar_wait_drain(bar(kWF + (int)(i % kWStages)), (uint32_t)((i / kWStages) & 1));
            for (long i = max(0L, xb - kXStages); i < xb; ++i)
                mbar_wait_drain(bar(kXF + (int)(i % kXStages)), (uint32_t)((i / kXStages) & 1));
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            grid_dependency_wait();
            const int M = __ldcg(P.count);
            const int nstream = (M + kStreamRows - 1) / kStreamRows;
            long xb = 0;
            bool ok = true;
            for (int g = 0; ok && g < nstream; ++g) {
                const int nrows = min(kStreamRows, M - g * kStreamRows);
                const int nbox = (nrows + kBox - 1) / kBox;
                if (g > 0) {
                    // the epilogue has read the previous stream out of TMEM
                    ok = mbar_wait(bar(kTF), (uint32_t)((g - 1) & 1), abort_flag, P.dev_status);
                    if (!ok) break;
                }
                for (int s = 0; ok && s < nslab; ++s) {
                    const long gs = (long)g * nslab + s;
                    const int ws = (int)(gs % kWStages);
                    ok = mbar_wait(bar(kWF + ws), (uint32_t)((gs / kWStages) & 1), abort_flag,
                                   P.dev_status);
                    for (int b = 0; ok && b < nbox; ++b, ++xb) {
                        const int xs = (int)(xb % kXStages);
                        ok = mbar_wait(bar(kXF + xs), (uint32_t)((xb / kXStages) & 1), abort_flag,
                                       P.dev_status);
                        if (!ok) break;
                        tc_fence_after();
                        const int rows_b = min(kBox, nrows - b * kBox);
                        const uint32_t idesc =
                            idesc_bf16_f32(128, (uint32_t)((rows_b + 15) & ~15), 0, 0);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint64_t a =
                                smem_desc_sw128(sbase + kOffW + ws * kWSlab + kk * 32, 16, 1024);
                            const uint64_t bd =
                                smem_desc_sw128(sbase + kOffX + xs * kXSlab + kk * 32, 16, 1024);
                            umma_bf16(tmem + (uint32_t)(b * kBox), a, bd, idesc,
                                      (s > 0 || kk > 0) ? 1u : 0u);
                        }
                        umma_commit(bar(kXE + xs));
                    }
                    if (ok) umma_commit(bar(kWE + ws));
                }
                if (ok) umma_commit(bar(kAF));
            }
            // every MMA issued above has completed before TMEM is released
            umma_commit(bar(kDR));
            mbar_wait_drain(bar(kDR), 0);
        }
    } else {
        // ------------------------------------------------ epilogue (warps 0-3)
        // Thread tid holds TMEM lane tid = head dim d of the accumulators.
        grid_dependency_wait();
        const int M = __ldcg(P.count);
        const int nstream = (M + kStreamRows - 1) / kStreamRows;
        const int d = tid;
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        // R[p][i] at kOffW + (2 p + i) * kRTile; R[0] ([64 rows][kD]) takes the sums
        float *R = reinterpret_cast<float *>(smem + kOffW);
        float *T = R;
        // partner slot j (0, 1) is the CTA of rank (rank + 1 + j) % 3; in that
        // CTA this one is partner slot 1 - j
        uint32_t r_peer[2], pr_peer[2], rx_peer[2];
        for (int j = 0; j < 2; ++j) {
            const uint32_t y = (rank + 1u + (uint32_t)j) % (uint32_t)kSplit;
            r_peer[j] = map_shared_rank(sbase + kOffW + (uint32_t)((1 - j) * 2 * kRTile), y);
            pr_peer[j] = map_shared_rank(bar(kPR), y);
            rx_peer[j] = map_shared_rank(bar(kRX), y);
        }
        const int q = tid & 3;  // dims [16q, 16q + 16) and [64 + 16q, 64 + 16q + 16)
        uint16_t *cache = kv == 0 ? P.k_cache : P.v_cache;
        float gain[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) gain[e] = 1.f;
        if (kv == 0) {
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                gain[e] = bf16_to_f32(__ldg(P.k_norm_w + (long)l * kD + 16 * q + e));
                gain[16 + e] = bf16_to_f32(__ldg(P.k_norm_w + (long)l * kD + 64 + 16 * q + e));
            }
        }
        int eb = 0;     // phases of kEB so far
        int round = 0;  // exchange rounds so far (phases of kPR and kRX)
        auto epi_sync = [&]() -> bool {
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kEB));
            const bool r = __all_sync(
                0xffffffffu, mbar_wait(bar(kEB), (uint32_t)(eb & 1), abort_flag, P.dev_status));
            ++eb;
            return r;
        };
        bool ok = true;
        for (int g = 0; ok && g < nstream; ++g) {
            const int nrows = min(kStreamRows, M - g * kStreamRows);
            const int nchunk = (nrows + 31) / 32;
            ok = __all_sync(0xffffffffu,
                            mbar_wait(bar(kAF), (uint32_t)(g & 1), abort_flag, P.dev_status));
            if (!ok) break;
            tc_fence_after();
            for (int c0 = 0; ok && c0 < nchunk; c0 += 2 * kSplit, ++round) {
                // This CTA's receive buffers may take the partners' chunks: its
                // MMAs are done and (after the first round) its warps have
                // finished reading them.
                if (c0 > 0) {
                    ok = epi_sync();
                    if (!ok) break;
                }
                if (tid == 0) {
                    mbar_arrive_remote_release(pr_peer[0]);
                    mbar_arrive_remote_release(pr_peer[1]);
                }
                ok = __all_sync(0xffffffffu, mbar_wait_cluster(bar(kPR), (uint32_t)(round & 1),
                                                               abort_flag, P.dev_status));
                if (!ok) break;
                // each partner's chunks of the round, this thread's dim d of 32 rows
                for (int jp = 0; jp < 2; ++jp) {
                    const int y = (int)((rank + 1u + (uint32_t)jp) % (uint32_t)kSplit);
                    for (int i = 0; i < 2; ++i) {
                        const int c = c0 + kSplit * i + y;
                        if (c >= nchunk) break;
                        float v[32];
                        tmem_ld32(tmem + lane_base + (uint32_t)(c * 32), v);
                        tmem_wait_ld();
                        if (nslab == 0) {  // no slab of the hidden dimension here (H = 128)
#pragma unroll
                            for (int jj = 0; jj < 32; ++jj) v[jj] = 0.f;
                        }
                        const uint32_t base = r_peer[jp] + (uint32_t)((i * 32 * kD + d) * 4);
#pragma unroll
                        for (int jj = 0; jj < 32; ++jj)
                            st_cluster_f32(base + (uint32_t)(jj * kD * 4), v[jj]);
                    }
                }
                mbar_arrive_remote_release(rx_peer[0]);
                mbar_arrive_remote_release(rx_peer[1]);
                ok = __all_sync(0xffffffffu, mbar_wait_cluster(bar(kRX), (uint32_t)(round & 1),
                                                               abort_flag, P.dev_status));
                if (!ok) break;
                // this CTA's chunks: own partial + slot 0's + slot 1's, into R[0]
                for (int i = 0; i < 2; ++i) {
                    const int c = c0 + kSplit * i + (int)rank;
                    if (c >= nchunk) break;
                    float v[32];
                    tmem_ld32(tmem + lane_base + (uint32_t)(c * 32), v);
                    tmem_wait_ld();
                    if (nslab == 0) {
#pragma unroll
                        for (int jj = 0; jj < 32; ++jj) v[jj] = 0.f;
                    }
                    float *col0 = R + i * 32 * kD + d;
                    const float *col1 = R + (2 + i) * 32 * kD + d;
#pragma unroll
                    for (int jj = 0; jj < 32; ++jj)
                        col0[jj * kD] = (v[jj] + col0[jj * kD]) + col1[jj * kD];
                }
                tc_fence_before();
                ok = epi_sync();  // the sums are complete: every epilogue warp has added its dims
                if (!ok) break;
                // finish this CTA's rows of the round, four threads a row
                for (int i = 0; i < 2; ++i) {
                    const int tl = i * 32 + (tid >> 2);             // row of T
                    const int c = c0 + kSplit * i + (int)rank;      // its chunk
                    const int t = c * 32 + (tl & 31);               // its row in the stream
                    const bool live = t < nrows;
                    float v[32];
                    const float *row = T + tl * kD;
#pragma unroll
                    for (int e = 0; e < 16; e += 4) {
                        const float4 lo = *reinterpret_cast<const float4 *>(row + 16 * q + e);
                        const float4 hi =
                            *reinterpret_cast<const float4 *>(row + 64 + 16 * q + e);
                        v[e] = lo.x; v[e + 1] = lo.y; v[e + 2] = lo.z; v[e + 3] = lo.w;
                        v[16 + e] = hi.x; v[17 + e] = hi.y; v[18 + e] = hi.z; v[19 + e] = hi.w;
                    }
                    const int2 m = live ? __ldcg(P.meta + (long)g * kStreamRows + t)
                                        : make_int2(-1, 0);
                    if (kv == 0) {
                        float ss = 0.f;
#pragma unroll
                        for (int e = 0; e < 32; ++e) ss = fmaf(v[e], v[e], ss);
                        ss += __shfl_xor_sync(0xffffffffu, ss, 1);
                        ss += __shfl_xor_sync(0xffffffffu, ss, 2);
                        const float inv = rsqrtf(ss * (1.f / kD) + P.eps);
#pragma unroll
                        for (int e = 0; e < 32; ++e) v[e] = v[e] * inv * gain[e];
                        if (live && m.x >= 0) {
                            const float *cs = P.cos_tab + (long)m.y * (kD / 2) + 16 * q;
                            const float *sn = P.sin_tab + (long)m.y * (kD / 2) + 16 * q;
#pragma unroll
                            for (int e = 0; e < 16; ++e) {
                                const float cv = __ldg(cs + e), sv = __ldg(sn + e);
                                const float a0 = v[e], a1 = v[16 + e];
                                v[e] = a0 * cv - a1 * sv;
                                v[16 + e] = a1 * cv + a0 * sv;
                            }
                        }
                    }
                    if (live && m.x >= 0) {
                        uint16_t *dst = cache + (((long)l * P.num_slots + m.x) * Hkv + h) * kD;
                        uint4 w[4];
                        uint32_t *wp = reinterpret_cast<uint32_t *>(w);
#pragma unroll
                        for (int e = 0; e < 16; ++e) wp[e] = pack2_bf16(v[2 * e], v[2 * e + 1]);
                        *reinterpret_cast<uint4 *>(dst + 16 * q) = w[0];
                        *reinterpret_cast<uint4 *>(dst + 16 * q + 8) = w[1];
                        *reinterpret_cast<uint4 *>(dst + 64 + 16 * q) = w[2];
                        *reinterpret_cast<uint4 *>(dst + 64 + 16 * q + 8) = w[3];
                    }
                }
            }
            if (!ok) break;
            // this warp is done with TMEM and with T for this stream
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kTF));
        }
    }

    // Every thread of the cluster's CTAs gets here (all waits are bounded):
    // after this barrier no CTA touches another's shared memory again.
    __syncwarp();
    tc_fence_before();
    cluster_sync_all();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ------------------------------------------------------------------ host side
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn tensor_map_encoder() {
    static EncodeTiledFn fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<EncodeTiledFn>(p);
        return static_cast<EncodeTiledFn>(nullptr);
    }();
    return fn;
}

// 2-D bf16 tensor [rows, cols] (cols contiguous) in 64-column, 128-byte
// swizzled boxes of box_rows rows.
bool encode_rows(EncodeTiledFn enc, CUtensorMap *tm, const void *base, uint64_t rows,
                 uint64_t cols, uint32_t box_rows) {
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t es[2] = {1, 1};
    return enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides,
               box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

struct WsLayout {
    size_t off_meta, off_x, total;
};

WsLayout ws_layout(int bs, int B, int H) {
    const size_t rows = (size_t)bs * B;
    WsLayout w;
    w.off_meta = 256;  // the row count lives at offset 0
    w.off_x = w.off_meta + align256(rows * sizeof(int2));
    w.total = w.off_x + align256(rows * (size_t)H * 2);
    return w;
}

}  // namespace

size_t kvmat_workspace_bytes(int bs, int B, int H) { return ws_layout(bs, B, H).total; }

int launch_kv_materialize(const KvMatArgs &a, cudaStream_t stream) {
    if (a.bs == 0) return BDSA_OK;
    EncodeTiledFn enc = tensor_map_encoder();
    if (enc == nullptr) return BDSA_CUDA_ERROR;
    const WsLayout wl = ws_layout(a.bs, a.B, a.H);
    char *ws = static_cast<char *>(a.workspace);
    int32_t *count = reinterpret_cast<int32_t *>(ws);
    int2 *meta = reinterpret_cast<int2 *>(ws + wl.off_meta);
    uint16_t *xc = reinterpret_cast<uint16_t *>(ws + wl.off_x);
    const long heads = (long)a.n_layers * 2 * a.Hkv;
    CUtensorMap tm_w, tm_x;
    if (!encode_rows(enc, &tm_w, a.w_kv, (uint64_t)heads * kD, (uint64_t)a.H, kD) ||
        !encode_rows(enc, &tm_x, xc, (uint64_t)a.bs * a.B, (uint64_t)a.H, kBox))
        return BDSA_CUDA_ERROR;
    static bool attr_set = false;
    if (!attr_set) {
        // two CTAs an SM need the largest shared-memory carve-out
        if (cudaFuncSetAttribute(kvmat_project_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kSmem) != cudaSuccess ||
            // the gather runs with the same carve-out, so that projection
            // CTAs can start on SMs still running gather CTAs
            cudaFuncSetAttribute(kvmat_gather_kernel,
                                 cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared) != cudaSuccess ||
            cudaFuncSetAttribute(kvmat_project_kernel,
                                 cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared) != cudaSuccess)
            return BDSA_CUDA_ERROR;
        attr_set = true;
    }
    kvmat_gather_kernel<<<dim3((unsigned)a.bs, kGatherParts), kGatherThreads, 0, stream>>>(
        reinterpret_cast<const uint4 *>(a.hidden), a.commit_len, a.positions, a.cache_loc, a.bs,
        a.B, a.H, a.max_pos, a.num_slots, count, meta, reinterpret_cast<uint4 *>(xc),
        a.dev_status);
    if (cudaGetLastError() != cudaSuccess) return BDSA_CUDA_ERROR;
    Params P;
    P.count = count;
    P.meta = meta;
    P.k_norm_w = a.k_norm_w;
    P.cos_tab = a.cos_tab;
    P.sin_tab = a.sin_tab;
    P.k_cache = a.k_cache;
    P.v_cache = a.v_cache;
    P.num_slots = a.num_slots;
    P.n_layers = a.n_layers;
    P.Hkv = a.Hkv;
    P.H = a.H;
    P.max_pos = a.max_pos;
    P.eps = a.eps;
    P.dev_status = a.dev_status;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(heads * kSplit));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kSplit;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kvmat_project_kernel, tm_w, tm_x, P) == cudaSuccess
               ? BDSA_OK
               : BDSA_CUDA_ERROR;
}

}  // namespace bdsa
