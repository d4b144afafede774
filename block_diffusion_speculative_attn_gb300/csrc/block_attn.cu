// block_attn.cu -- block attention over a paged KV cache for sm_103a.
//
// Computes, per request r, KV head h and block row i (query heads j = h*G + g):
//   o = softmax(scale * q k^T) v over keys t < limit(i), where
//   limit(i) = L_r + B (DRAFT: rectangular intra-block mask) or L_r + i + 1
//   (VERIFY: token-causal), as defined on "SGLang dLLM / LLaDA 2.0", section
//   "Attention Mask", and used by the draft/verify passes of "From DFlash to
//   dLLM Self-Spec (II)", sections 2.2.3-2.2.4 and "(IV)", section 4.4.1.
//
// One call = three launches chained with programmatic dependent launch:
//   plan    one CTA: per-request tile counts -> prefix; validates every page id
//           a request references and flags the request if one is out of range;
//   attend  persistent, one CTA per SM.  Every (request, KV head) unit is a run
//           of 128-key tiles; the runs are concatenated and each CTA takes an
//           equal contiguous range (stream-K style), so the work is balanced to
//           one tile.  A unit wholly inside one CTA is written directly; a unit
//           cut between CTAs leaves an fp32 partial (o / l and log2-sum-exp) in
//           one of each CTA's two slots;
//   merge   one CTA per range boundary that cuts a unit: merges the unit's
//           partials in tile order.
//
// Inside a CTA (warp roles: 0-3 softmax + epilogue, 4 Q/K producer, 5 MMA
// issuer + TMEM owner, 6 V producer):
//   * the G*B query rows (row m = i*G + g) form the A operand of a tcgen05 MMA
//     tile: M = 64 when G*B <= 64, else M = 128 (zero rows pad it).  An M = 64
//     accumulator spreads its rows over lanes 0-15 of all four TMEM lane
//     quadrants, so all four SM sub-partitions run the softmax with two
//     threads per row (16x32bx2 TMEM accesses); M = 128 has one thread per row;
//   * K and V tiles arrive by TMA, one box per page (or per 128 keys of a
//     larger page), into 128-byte-swizzled shared memory, through a K ring and
//     a deeper V ring fed by separate producer warps, with an L2 evict-first
//     policy since every K/V byte is read exactly once;
//   * S = Q K^T and O += P V run on the tensor cores with fp32 accumulators in
//     TMEM: two S buffers and two O buffers (512 columns), so consecutive units
//     overlap;
//   * softmax in the log2 domain: one FFMA + ex2 per score, running max with a
//     lazy rescale of O in TMEM only when the max grows by more than 2^8, P
//     rounded to bf16 and written swizzled for the PV MMA.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>
#include <utility>

#include "bdsa_device.cuh"
#include "bdsa_internal.h"

namespace bdsa {
namespace {

constexpr int kBN = 128;                  // keys per tile
constexpr int kThreads = 224;
constexpr int kKProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kVProducerWarp = 6;
constexpr int kSoftmaxWarps = 4;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 256;          // S at columns 0 / 128, O at 256 / 384
constexpr float kRescaleLog2 = 8.0f;      // rescale O only when the max grows by > 2^8
constexpr float kLn2 = 0.6931471805599453f;

template <int D, int M>
struct Cfg {
    static constexpr int DH = D / 64;               // 64-element (128-byte) slabs per row
    static constexpr int kSlab = M * 128;           // one M-row slab of 128-byte rows
    static constexpr int kKVSlab = kBN * 128;       // one 128-key slab
    static constexpr int NQ = (M == 64) ? 2 : 1;    // Q buffers
    static constexpr int NP = (M == 64) ? 2 : 1;    // P buffers
    // V is held from its load until PV, K only until S: the deeper V ring lets
    // each V load start about three tiles before its PV.
    static constexpr int NK = (D == 128) ? 2 : 4;
    static constexpr int NV = (D == 128) ? 3 : 4;
    static constexpr int TPR = (M == 64) ? 2 : 1;   // softmax threads per row
    static constexpr int NC = kBN / TPR;            // score columns per thread
    static constexpr int OC = D / TPR;              // output columns per thread
    static constexpr int kQBuf = DH * kSlab;
    static constexpr int kStage = DH * kKVSlab;
    static constexpr int kPBuf = 2 * kSlab;         // 128 keys = two 64-key slabs
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kOffQ + NQ * kQBuf;
    static constexpr int kOffV = kOffK + NK * kStage;
    static constexpr int kOffP = kOffV + NV * kStage;
    static constexpr int kOffBar = kOffP + NP * kPBuf;
    // barrier indices
    static constexpr int QF = 0;          // NQ: Q loaded
    static constexpr int QE = QF + NQ;    // NQ: Q buffer free (last S MMA of its unit done)
    static constexpr int KF = QE + NQ;
    static constexpr int KE = KF + NK;
    static constexpr int VF = KE + NK;
    static constexpr int VE = VF + NV;
    static constexpr int SF = VE + NV;    // 2: S buffer full
    static constexpr int SR = SF + 2;     // 2: S buffer read by the softmax
    // P written, one barrier per P buffer: with two buffers a softmax warp may
    // run one tile ahead of the others, and a single shared barrier would mix
    // arrivals of consecutive tiles into one phase.
    static constexpr int PF = SR + 2;     // NP
    static constexpr int PV = PF + NP;    // NP: PV done, per P buffer
    static constexpr int OE = PV + NP;    // 2: O buffer read by the epilogue
    static constexpr int DR = OE + 2;     // drain
    static constexpr int kNumBars = DR + 1;
    static constexpr int kOffMisc = kOffBar + 8 * kNumBars;
    static constexpr int kSmem = kOffMisc + 16 + 1024;  // + slack to align the base to 1 KB
};

struct Params {
    const int32_t *block_table;
    const int32_t *seq_lens;
    const int32_t *prefix;   // [bs + 1] exclusive prefix of per-request tile counts
    const int32_t *bad;      // [bs] request references a page id outside the pool
    uint16_t *out;
    float *lse;
    float *part_o;           // [2 * grid, rows, D]
    float *part_lse;         // [2 * grid, rows]
    int32_t *dev_status;
    int max_pages, num_pages, bs, B, Hq, Hkv, G, rows, page_size, log2_ps, box_rows, mode;
    float scale_log2;
};

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// One 32-column chunk of this thread's share of a TMEM accumulator block.
template <int M, int OFF>
__device__ __forceinline__ void tmem_load_chunk(uint32_t taddr, float (&v)[32]) {
    if constexpr (M == 64) tmem_ld16x2_32<OFF>(taddr, v);
    else tmem_ld32(taddr, v);
}
template <int M, int OFF>
__device__ __forceinline__ void tmem_store_chunk(uint32_t taddr, const float (&v)[32]) {
    if constexpr (M == 64) tmem_st16x2_32<OFF>(taddr, v);
    else tmem_st32(taddr, v);
}

// A maximal run of one unit's tiles inside a CTA's range.
struct Piece {
    int r, h, a, e, nt, L;
    long u_off;  // global index of the unit's first tile
};

__device__ __forceinline__ void locate(const int32_t *pre, int bs, int Hkv,
                                       const int32_t *seq_lens, long x, long x1, Piece &pc) {
    int lo = 0, hi = bs - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((long)Hkv * __ldg(pre + mid) <= x) lo = mid;
        else hi = mid - 1;
    }
    const long base = (long)Hkv * __ldg(pre + lo);
    pc.r = lo;
    pc.nt = __ldg(pre + lo + 1) - __ldg(pre + lo);
    const long y = x - base;
    pc.h = (int)(y / pc.nt);
    pc.a = (int)(y % pc.nt);
    pc.e = (int)min((long)pc.nt, (long)pc.a + (x1 - x));
    pc.L = __ldg(seq_lens + lo);
    pc.u_off = base + (long)pc.h * pc.nt;
}

// Start of CTA b's range and the CTA whose range holds global tile x.
__device__ __forceinline__ long range_start(int b, long W, int S) { return (long)b * W / S; }
__device__ __forceinline__ int cta_of(long x, long W, int S) {
    return (int)(((x + 1) * (long)S - 1) / W);
}

// Number of TMA boxes of tile t0 that hold keys of the request (never past its
// block-table row).
__device__ __forceinline__ int boxes_of(long n_keys, long t0, int rows_box, int log2_ps,
                                        int max_pages) {
    const long valid = max(0L, min((long)kBN, n_keys - t0));
    int nbox = (int)((valid + rows_box - 1) / rows_box);
    while (nbox > 0 && ((t0 + (long)(nbox - 1) * rows_box) >> log2_ps) >= max_pages) --nbox;
    return nbox;
}

template <int D, int M>
__global__ void __launch_bounds__(kThreads, 1)
    block_attn_kernel(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const Params prm) {
    using C = Cfg<D, M>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (sbase - raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int B = prm.B, G = prm.G;
    const long ps = prm.page_size;

    auto bar = [&](int i) -> uint32_t { return sbase + C::kOffBar + 8u * (uint32_t)i; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kOffMisc + 4);

    // ---- prologue (overlaps the plan kernel under programmatic dependent launch)
    grid_launch_dependents();
    if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int k = 0; k < C::NQ; ++k) {
            mbar_init(bar(C::QF + k), 1);
            mbar_init(bar(C::QE + k), 1);
        }
        for (int k = 0; k < C::NK; ++k) {
            mbar_init(bar(C::KF + k), 1);
            mbar_init(bar(C::KE + k), 1);
        }
        for (int k = 0; k < C::NV; ++k) {
            mbar_init(bar(C::VF + k), 1);
            mbar_init(bar(C::VE + k), 1);
        }
        for (int k = 0; k < 2; ++k) {
            mbar_init(bar(C::SF + k), 1);
            mbar_init(bar(C::SR + k), kSoftmaxWarps);
            mbar_init(bar(C::OE + k), kSoftmaxWarps);
        }
        for (int k = 0; k < C::NP; ++k) {
            mbar_init(bar(C::PF + k), kSoftmaxWarps);
            mbar_init(bar(C::PV + k), 1);
        }
        mbar_init(bar(C::DR), 1);
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    if (warp == kKProducerWarp && lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
    }
    if (warp == kVProducerWarp && lane == 0) tma_prefetch_desc(&tm_v);
    // Zero the padding rows of every Q buffer so padded S rows stay finite.
    if (prm.rows < M) {
        const int pad = M - prm.rows;
        for (int idx = tid; idx < C::NQ * C::DH * pad * 8; idx += kThreads) {
            const int u = idx & 7;
            const int m = prm.rows + (idx >> 3) % pad;
            const int slab = (idx >> 3) / pad;  // qbuf * DH + c
            st_shared_v4(sbase + C::kOffQ + slab * C::kSlab + m * 128 + u * 16, 0, 0, 0, 0);
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // ---- the plan kernel's outputs are needed from here on
    grid_dependency_wait();
    // Warm L1 with the tile prefix: every role's first binary search reads it.
    for (int i = tid * 32; i <= prm.bs; i += kThreads * 32)
        asm volatile("prefetch.global.L1 [%0];" ::"l"(prm.prefix + i));
    const int S = gridDim.x;
    const int b = blockIdx.x;
    const long W = (long)prm.Hkv * __ldg(prm.prefix + prm.bs);
    const long x0 = range_start(b, W, S), x1 = range_start(b + 1, W, S);

    if (warp == kKProducerWarp || warp == kVProducerWarp) {
        // ------------------------------------------------ TMA producers
        const bool is_k = warp == kKProducerWarp;
        if (lane == 0) {
            const uint64_t policy = l2_policy_evict_first();
            const int rows_box = prm.box_rows;
            const int NR = is_k ? C::NK : C::NV;
            const int FULL = is_k ? C::KF : C::VF;
            const int EMPTY = is_k ? C::KE : C::VE;
            const uint32_t dst0 = sbase + (is_k ? C::kOffK : C::kOffV);
            const void *tmap = is_k ? (const void *)&tm_k : (const void *)&tm_v;
            long g = 0, issued = 0, q_issued = 0;
            int k = 0;
            bool ok = true;
            for (long x = x0; ok && x < x1; ++k) {
                Piece pc;
                locate(prm.prefix, prm.bs, prm.Hkv, prm.seq_lens, x, x1, pc);
                if (is_k) {
                    const int qb = k % C::NQ;
                    if (k >= C::NQ) {
                        ok = mbar_wait(bar(C::QE + qb), ((k / C::NQ) - 1) & 1, abort_flag,
                                       prm.dev_status);
                        if (!ok) break;
                    }
                    mbar_arrive_expect_tx(bar(C::QF + qb), (uint32_t)(prm.rows * D * 2));
                    for (int c = 0; c < C::DH; ++c)
                        tma_load_4d(sbase + C::kOffQ + qb * C::kQBuf + c * C::kSlab, &tm_q,
                                    c * 64, 0, pc.h, pc.r * B, bar(C::QF + qb));
                    q_issued = k + 1;
                }
                const long n_keys = (long)pc.L + B;
                const int32_t *bt = prm.block_table + (long)pc.r * prm.max_pages;
                for (int j = pc.a; j < pc.e; ++j, ++g) {
                    const long t0 = (long)j * kBN;
                    const int nbox = boxes_of(n_keys, t0, rows_box, prm.log2_ps, prm.max_pages);
                    const int st = (int)(g % NR);
                    ok = mbar_wait(bar(EMPTY + st), (uint32_t)(((g / NR) & 1) ^ 1), abort_flag,
                                   prm.dev_status);
                    if (!ok) break;
                    mbar_arrive_expect_tx(bar(FULL + st),
                                          (uint32_t)(nbox * rows_box * 128 * C::DH));
                    for (int bx = 0; bx < nbox; ++bx) {
                        const long t = t0 + (long)bx * rows_box;
                        const int32_t slot =
                            bt[t >> prm.log2_ps] * prm.page_size + (int32_t)(t & (ps - 1));
                        for (int c = 0; c < C::DH; ++c)
                            tma_load_2d_hint(dst0 + st * C::kStage + c * C::kKVSlab +
                                                 bx * rows_box * 128,
                                             tmap, pc.h * D + c * 64, slot, bar(FULL + st),
                                             policy);
                    }
                    issued = g + 1;
                }
                x += pc.e - pc.a;
            }
            // Drain: the last load issued into each buffer must have landed before exit.
            for (long i = max(0L, q_issued - C::NQ); i < q_issued; ++i)
                mbar_wait_drain(bar(C::QF + (int)(i % C::NQ)), (uint32_t)((i / C::NQ) & 1));
            for (long i = max(0L, issued - NR); i < issued; ++i)
                mbar_wait_drain(bar(FULL + (int)(i % NR)), (uint32_t)((i / NR) & 1));
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_qk = idesc_bf16_f32(M, kBN, 0, 0);
            constexpr uint32_t idesc_pv = idesc_bf16_f32(M, D, 0, 1);
            // PV of tile g is issued after S of tile g + 1 within a unit; the last
            // PV of a unit is issued before the next unit's first S.
            struct Pending {
                long g;
                int k;
                bool first;
            } pend{0, 0, false};
            bool have = false;
            auto issue_pv = [&](const Pending &pv) -> bool {
                const int ob = pv.k & 1;
                if (pv.first && pv.k >= 2) {
                    if (!mbar_wait(bar(C::OE + ob), ((pv.k >> 1) - 1) & 1, abort_flag,
                                   prm.dev_status))
                        return false;
                }
                const int pb = (int)(pv.g % C::NP);
                if (!mbar_wait(bar(C::PF + pb), (uint32_t)((pv.g / C::NP) & 1), abort_flag,
                               prm.dev_status))
                    return false;
                const int vs = (int)(pv.g % C::NV);
                if (!mbar_wait(bar(C::VF + vs), (uint32_t)((pv.g / C::NV) & 1), abort_flag,
                               prm.dev_status))
                    return false;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk) {
                    const uint64_t a = smem_desc_sw128(
                        sbase + C::kOffP + pb * C::kPBuf + (kk >> 2) * C::kSlab + (kk & 3) * 32,
                        16, 1024);
                    const uint64_t bdesc = smem_desc_sw128(
                        sbase + C::kOffV + vs * C::kStage + kk * 16 * 128, C::kKVSlab, 1024);
                    umma_bf16(tmem + kTmemO + ob * 128, a, bdesc, idesc_pv,
                              (pv.first && kk == 0) ? 0u : 1u);
                }
                umma_commit(bar(C::PV + pb));
                umma_commit(bar(C::VE + vs));
                return true;
            };
            long g = 0;
            int k = 0;
            bool ok = true;
            for (long x = x0; ok && x < x1; ++k) {
                Piece pc;
                locate(prm.prefix, prm.bs, prm.Hkv, prm.seq_lens, x, x1, pc);
                if (have) {
                    ok = issue_pv(pend);
                    have = false;
                    if (!ok) break;
                }
                const int qb = k % C::NQ;
                ok = mbar_wait(bar(C::QF + qb), (k / C::NQ) & 1, abort_flag, prm.dev_status);
                const int n = pc.e - pc.a;
                for (int j = 0; ok && j < n; ++j, ++g) {
                    const int ks = (int)(g % C::NK);
                    ok = mbar_wait(bar(C::KF + ks), (uint32_t)((g / C::NK) & 1), abort_flag,
                                   prm.dev_status);
                    if (!ok) break;
                    const int sb = (int)(g & 1);
                    if (g >= 2) {
                        ok = mbar_wait(bar(C::SR + sb), (uint32_t)(((g >> 1) - 1) & 1),
                                       abort_flag, prm.dev_status);
                        if (!ok) break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint64_t a = smem_desc_sw128(sbase + C::kOffQ + qb * C::kQBuf +
                                                               (kk >> 2) * C::kSlab + (kk & 3) * 32,
                                                           16, 1024);
                        const uint64_t bdesc =
                            smem_desc_sw128(sbase + C::kOffK + ks * C::kStage +
                                                (kk >> 2) * C::kKVSlab + (kk & 3) * 32,
                                            16, 1024);
                        umma_bf16(tmem + sb * 128, a, bdesc, idesc_qk, kk > 0 ? 1u : 0u);
                    }
                    umma_commit(bar(C::SF + sb));
                    umma_commit(bar(C::KE + ks));
                    if (j == n - 1) umma_commit(bar(C::QE + qb));
                    if (have) ok = issue_pv(pend);
                    pend = Pending{g, k, j == 0};
                    have = true;
                }
                x += n;
            }
            if (ok && have) ok = issue_pv(pend);
            // Drain: every MMA issued above has completed before TMEM is released.
            umma_commit(bar(C::DR));
            mbar_wait_drain(bar(C::DR), 0);
        }
    } else if (warp < kSoftmaxWarps) {
        // ------------------------------------------------ softmax + epilogue
        // Thread -> (row, column half).  M = 128: row = tid, all 128 columns.
        // M = 64: row = 16 * warp + lane % 16, half = lane / 16 owns columns
        // [64 * half, 64 * half + 64) of every 128-column block.
        constexpr int NC = C::NC;
        constexpr int OC = C::OC;
        const int half = (M == 64) ? (lane >> 4) : 0;
        const int row = (M == 64) ? warp * 16 + (lane & 15) : tid;
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        const float sl2 = prm.scale_log2;
        const bool valid_row = row < prm.rows;
        const int i_blk = row / G;
        long g = 0;
        int k = 0;
        bool ok = true;
        for (long x = x0; ok && x < x1; ++k) {
            Piece pc;
            locate(prm.prefix, prm.bs, prm.Hkv, prm.seq_lens, x, x1, pc);
            const int bad = __ldg(prm.bad + pc.r);  // used only in the epilogue
            const long n_keys = (long)pc.L + B;
            const long limit =
                (prm.mode == BDSA_MODE_DRAFT) ? n_keys : min(n_keys, (long)pc.L + i_blk + 1);
            const int ob = k & 1;
            float m_used = -INFINITY;
            float l4[4] = {0.f, 0.f, 0.f, 0.f};
            for (int j = pc.a; j < pc.e; ++j, ++g) {
                const long t0 = (long)j * kBN;
                const int sb = (int)(g & 1);
                ok = mbar_wait(bar(C::SF + sb), (uint32_t)((g >> 1) & 1), abort_flag,
                               prm.dev_status);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc_fence_after();
                float sv[NC];
#pragma unroll
                for (int c = 0; c < NC / 32; ++c)
                    tmem_load_chunk<M, NC>(tmem + lane_base + sb * 128 + c * 32,
                                           *reinterpret_cast<float(*)[32]>(&sv[c * 32]));
                tmem_wait_ld();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(C::SR + sb));

                // mask past this row's limit (raw scores; scale > 0 keeps the max)
                const long nvalid = limit - t0 - half * NC;
                if (nvalid < NC) {
#pragma unroll
                    for (int c = 0; c < NC; ++c)
                        if (c >= nvalid) sv[c] = -INFINITY;
                }
                float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int c = 0; c < NC; ++c) mx[c & 3] = fmaxf(mx[c & 3], sv[c]);
                float mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
                if constexpr (M == 64) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 16));
                const float m_new = mt * sl2;
                float alpha = 1.f;
                bool resc = false;
                if (m_new > m_used + kRescaleLog2) {
                    alpha = ex2_approx(m_used - m_new);
                    m_used = m_new;
                    resc = true;
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) l4[q] *= alpha;
                uint32_t pk[NC / 2];
                if (m_used == -INFINITY) {
#pragma unroll
                    for (int c = 0; c < NC / 2; ++c) pk[c] = 0u;
                } else {
                    const float neg_m = -m_used;
#pragma unroll
                    for (int c = 0; c < NC / 2; ++c) {
                        const float p0 = ex2_approx(fmaf(sv[2 * c], sl2, neg_m));
                        const float p1 = ex2_approx(fmaf(sv[2 * c + 1], sl2, neg_m));
                        l4[c & 3] += p0 + p1;
                        pk[c] = pack_bf16x2(p0, p1);
                    }
                }
                const int pb = (int)(g % C::NP);
                // The P buffer must be free: PV of tile g - NP has read it.
                if (g >= C::NP) {
                    const long prev = g - C::NP;
                    ok = mbar_wait(bar(C::PV + pb), (uint32_t)((prev / C::NP) & 1), abort_flag,
                                   prm.dev_status);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                }
                // A grown max rescales O, which needs PV of the previous tile of this unit.
                if (j > pc.a && __any_sync(0xffffffffu, resc)) {
                    const long prev = g - 1;
                    ok = mbar_wait(bar(C::PV + (int)(prev % C::NP)),
                                   (uint32_t)((prev / C::NP) & 1), abort_flag, prm.dev_status);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll
                    for (int c = 0; c < OC / 32; ++c) {
                        float ov[32];
                        const uint32_t ta = tmem + lane_base + kTmemO + ob * 128 + c * 32;
                        tmem_load_chunk<M, D / 2>(ta, ov);
                        tmem_wait_ld();
#pragma unroll
                        for (int q = 0; q < 32; ++q) ov[q] *= alpha;
                        tmem_store_chunk<M, D / 2>(ta, ov);
                    }
                    tmem_wait_st();
                }
                // P row -> shared memory, K-major with the 128-byte swizzle.
                {
                    const uint32_t pbase = sbase + C::kOffP + pb * C::kPBuf;
#pragma unroll
                    for (int u = 0; u < NC / 8; ++u) {
                        const int slab = (M == 64) ? half : (u >> 3);
                        const int cu = u & 7;
                        const uint32_t addr = pbase + slab * C::kSlab + row * 128 +
                                              ((uint32_t)(cu ^ (row & 7)) << 4);
                        st_shared_v4(addr, pk[4 * u], pk[4 * u + 1], pk[4 * u + 2],
                                     pk[4 * u + 3]);
                    }
                }
                // Ragged tile: V rows past the request's keys hold stale or never-written
                // cache slots (possibly NaN); P is 0 there, but 0 * NaN is not.
                const long tile_keys = n_keys - t0;
                if (tile_keys < kBN) {
                    const int vs = (int)(g % C::NV);
                    ok = mbar_wait(bar(C::VF + vs), (uint32_t)((g / C::NV) & 1), abort_flag,
                                   prm.dev_status);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                    if (tid >= tile_keys) {
#pragma unroll
                        for (int c = 0; c < C::DH; ++c)
#pragma unroll
                            for (int u = 0; u < 8; ++u)
                                st_shared_v4(sbase + C::kOffV + vs * C::kStage + c * C::kKVSlab +
                                                 tid * 128 + u * 16,
                                             0, 0, 0, 0);
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(C::PF + pb));
            }
            if (!ok) break;

            // ---- epilogue of the piece
            {
                const long lastg = g - 1;
                ok = mbar_wait(bar(C::PV + (int)(lastg % C::NP)), (uint32_t)((lastg / C::NP) & 1),
                               abort_flag, prm.dev_status);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
            }
            tc_fence_after();
            float l = (l4[0] + l4[1]) + (l4[2] + l4[3]);
            if constexpr (M == 64) l += __shfl_xor_sync(0xffffffffu, l, 16);
            const float inv_l = l > 0.f ? 1.f / l : 0.f;
            const float lse2 = l > 0.f ? m_used + log2f(l) : -INFINITY;
            const bool complete = (pc.a == 0 && pc.e == pc.nt);
            const long token = (long)pc.r * B + i_blk;
            const long orow = token * prm.Hq + (long)pc.h * G + row % G;
            const int slot = 2 * b + (k == 0 ? 0 : 1);
#pragma unroll
            for (int c = 0; c < OC / 32; ++c) {
                float ov[32];
                tmem_load_chunk<M, D / 2>(tmem + lane_base + kTmemO + ob * 128 + c * 32, ov);
                tmem_wait_ld();
                if (!valid_row) continue;
                const int col0 = half * OC + c * 32;
                if (bad) {
                    uint4 *dst = reinterpret_cast<uint4 *>(prm.out + orow * D + col0);
#pragma unroll
                    for (int v = 0; v < 4; ++v) dst[v] = make_uint4(0, 0, 0, 0);
                } else if (complete) {
                    uint4 *dst = reinterpret_cast<uint4 *>(prm.out + orow * D + col0);
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        uint4 w;
                        w.x = pack_bf16x2(ov[8 * v + 0] * inv_l, ov[8 * v + 1] * inv_l);
                        w.y = pack_bf16x2(ov[8 * v + 2] * inv_l, ov[8 * v + 3] * inv_l);
                        w.z = pack_bf16x2(ov[8 * v + 4] * inv_l, ov[8 * v + 5] * inv_l);
                        w.w = pack_bf16x2(ov[8 * v + 6] * inv_l, ov[8 * v + 7] * inv_l);
                        dst[v] = w;
                    }
                } else {
                    float4 *dst = reinterpret_cast<float4 *>(
                        prm.part_o + ((long)slot * prm.rows + row) * D + col0);
#pragma unroll
                    for (int v = 0; v < 8; ++v)
                        dst[v] = make_float4(ov[4 * v] * inv_l, ov[4 * v + 1] * inv_l,
                                             ov[4 * v + 2] * inv_l, ov[4 * v + 3] * inv_l);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::OE + ob));
            if (valid_row && half == 0) {
                if (bad) {
                    if (prm.lse) prm.lse[orow] = -INFINITY;
                } else if (complete) {
                    if (prm.lse) prm.lse[orow] = lse2 * kLn2;
                } else {
                    prm.part_lse[(long)slot * prm.rows + row] = lse2;
                }
            }
            x += pc.e - pc.a;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// Merge the partials of every unit cut between CTAs.  Blocks (b, sub): b picks
// the unit whose first interior cut is the start of CTA b's range; the unit's
// (row, 4-column) items are spread over kMergeSub blocks of 256 threads, one
// item per thread, with the pieces' loads issued kMB at a time.
constexpr int kMergeSub = 8;
constexpr int kMergeThreads = 256;

template <int D>
__global__ void __launch_bounds__(kMergeThreads) attn_merge_kernel(const Params prm, int S) {
    grid_dependency_wait();
    const int b = blockIdx.x;
    const long W = (long)prm.Hkv * __ldg(prm.prefix + prm.bs);
    if (b == 0 || W == 0) return;
    const long x = range_start(b, W, S);
    if (x >= W) return;
    Piece pc;
    locate(prm.prefix, prm.bs, prm.Hkv, prm.seq_lens, x, W, pc);
    // split at this cut, and no earlier cut lies inside the unit
    if (!(pc.u_off < x && range_start(b - 1, W, S) <= pc.u_off)) return;
    if (__ldg(prm.bad + pc.r)) return;
    const int b_first = cta_of(pc.u_off, W, S);
    const int b_last = cta_of(pc.u_off + pc.nt - 1, W, S);
    constexpr int C4 = D / 4;
    const int items = prm.rows * C4;
    constexpr int kMB = 8;  // pieces whose loads are in flight together
    for (int it = blockIdx.y * kMergeThreads + threadIdx.x; it < items;
         it += kMergeSub * kMergeThreads) {
        const int row = it / C4, c4 = it % C4;
        // running max / sum of the pieces' log2-sum-exp for this row
        float mmax = -INFINITY, den = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int b0 = b_first; b0 <= b_last; b0 += kMB) {
            float ls[kMB];
            float4 po[kMB];
#pragma unroll
            for (int q = 0; q < kMB; ++q) {
                const int bb = b0 + q;
                const long fb = range_start(bb, W, S);
                const bool live = bb <= b_last && fb < range_start(bb + 1, W, S);
                const int sl = 2 * bb + (fb >= pc.u_off ? 0 : 1);
                ls[q] = live ? __ldcg(prm.part_lse + (long)sl * prm.rows + row) : -INFINITY;
                po[q] = live ? __ldcg(reinterpret_cast<const float4 *>(
                                   prm.part_o + ((long)sl * prm.rows + row) * D) + c4)
                             : make_float4(0.f, 0.f, 0.f, 0.f);
            }
            float bm = mmax;
#pragma unroll
            for (int q = 0; q < kMB; ++q) bm = fmaxf(bm, ls[q]);
            if (bm == -INFINITY) continue;
            const float sc = (mmax == -INFINITY) ? 0.f : exp2f(mmax - bm);
            den *= sc;
            acc.x *= sc;
            acc.y *= sc;
            acc.z *= sc;
            acc.w *= sc;
#pragma unroll
            for (int q = 0; q < kMB; ++q) {
                if (ls[q] == -INFINITY) continue;
                const float w = exp2f(ls[q] - bm);
                den += w;
                acc.x += w * po[q].x;
                acc.y += w * po[q].y;
                acc.z += w * po[q].z;
                acc.w += w * po[q].w;
            }
            mmax = bm;
        }
        const float inv = den > 0.f ? 1.f / den : 0.f;
        const long orow =
            ((long)pc.r * prm.B + row / prm.G) * prm.Hq + (long)pc.h * prm.G + row % prm.G;
        uint2 w;
        w.x = pack_bf16x2(acc.x * inv, acc.y * inv);
        w.y = pack_bf16x2(acc.z * inv, acc.w * inv);
        *reinterpret_cast<uint2 *>(prm.out + orow * D + c4 * 4) = w;
        if (c4 == 0 && prm.lse) prm.lse[orow] = den > 0.f ? (mmax + log2f(den)) * kLn2 : -INFINITY;
    }
}

// Per-request tile counts -> exclusive prefix; per-request page-id validation.
// One CTA of 1024 threads.
constexpr int kPlanChunk = 2048;  // requests validated per pass (page prefix in shared memory)

__global__ void __launch_bounds__(1024)
    attn_plan_kernel(const int32_t *__restrict__ seq_lens, const int32_t *__restrict__ block_table,
                     int bs, int B, int max_pages, int num_pages, int page_size,
                     int32_t *__restrict__ prefix, int32_t *__restrict__ bad,
                     int32_t *dev_status) {
    grid_launch_dependents();
    __shared__ int warp_tot[32];
    __shared__ int carry;
    __shared__ int page_pre[kPlanChunk + 1];
    __shared__ int any_bad;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    if (tid == 0) {
        carry = 0;
        any_bad = 0;
    }
    __syncthreads();
    for (int base = 0; base < bs; base += 1024) {
        const int i = base + tid;
        int nt = 0;
        if (i < bs) {
            const long nk = (long)seq_lens[i] + B;
            nt = nk > 0 ? (int)min((nk + kBN - 1) / kBN, 1L << 24) : 1;
        }
        int inc = nt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += t;
        }
        if (lane == 31) warp_tot[wid] = inc;
        __syncthreads();
        if (wid == 0) {
            const int v = warp_tot[lane];
            int vi = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int t = __shfl_up_sync(0xffffffffu, vi, o);
                if (lane >= o) vi += t;
            }
            warp_tot[lane] = vi - v;  // exclusive prefix of warp totals
        }
        __syncthreads();
        const int excl = carry + warp_tot[wid] + inc - nt;
        if (i < bs) prefix[i] = excl;
        __syncthreads();
        if (tid == 1023) carry = excl + nt;
        __syncthreads();
    }
    if (tid == 0) prefix[bs] = carry;

    // Validation: the pages each request references, flattened over a chunk of
    // requests and split evenly over the threads so the loads are in flight
    // together.
    for (int base = 0; base < bs; base += kPlanChunk) {
        const int n = min(kPlanChunk, bs - base);
        __syncthreads();
        if (tid == 0) {
            int acc = 0;
            for (int q = 0; q < n; ++q) {
                const int r = base + q;
                const long L = seq_lens[r];
                const long need = (L + B + page_size - 1) / page_size;
                const bool shape_bad = L < 0 || need > max_pages;
                page_pre[q] = acc;
                bad[r] = shape_bad ? 1 : 0;
                if (shape_bad) any_bad = 1;
                else acc += (int)need;
            }
            page_pre[n] = acc;
        }
        __syncthreads();
        const int total = page_pre[n];
        const int per = (total + 1023) / 1024;
        const int p0 = min(total, tid * per), p1 = min(total, p0 + per);
        int q = 0;
        {
            int lo = 0, hi = n - 1;  // request holding flattened page p0
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (page_pre[mid] <= p0) lo = mid;
                else hi = mid - 1;
            }
            q = lo;
        }
        for (int p = p0; p < p1; ++p) {
            while (q < n - 1 && page_pre[q + 1] <= p) ++q;
            const int r = base + q;
            const int32_t pg = __ldg(block_table + (long)r * max_pages + (p - page_pre[q]));
            if (pg < 0 || pg >= num_pages) {
                bad[r] = 1;
                any_bad = 1;
            }
        }
    }
    __syncthreads();
    if (tid == 0 && any_bad) report_status(dev_status, BDSA_DEVICE_OUT_OF_RANGE);
}

// ------------------------------------------------------------------ host side
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// Launch with the programmatic-stream-serialization attribute, so the kernel
// may start its prologue while the previous kernel on the stream finishes.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

template <int D, int M>
int launch_impl(const AttnArgs &a, const AttnPlan &plan, cudaStream_t stream) {
    using C = Cfg<D, M>;
    EncodeTiledFn enc = encode_fn();
    if (enc == nullptr) return BDSA_CUDA_ERROR;
    const int G = a.Hq / a.Hkv;
    CUtensorMap tq, tk, tv;
    {
        // q[(token*Hq + h*G + g)*D + d] as a 4-D tensor (d, g, h, token).
        cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)G, (cuuint64_t)a.Hkv,
                              (cuuint64_t)a.bs * a.B};
        cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)G * D * 2,
                                 (cuuint64_t)a.Hq * D * 2};
        cuuint32_t box[4] = {64, (cuuint32_t)G, 1, (cuuint32_t)a.B};
        cuuint32_t es[4] = {1, 1, 1, 1};
        if (enc(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<uint16_t *>(a.q), dims,
                strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
            CUDA_SUCCESS)
            return BDSA_CUDA_ERROR;
    }
    const int box_rows = a.page_size < kBN ? a.page_size : kBN;
    for (int which = 0; which < 2; ++which) {
        // cache[slot][h][d] as a 2-D tensor (h*D + d, slot).
        cuuint64_t dims[2] = {(cuuint64_t)a.Hkv * D, (cuuint64_t)a.num_pages * a.page_size};
        cuuint64_t strides[1] = {(cuuint64_t)a.Hkv * D * 2};
        cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
        cuuint32_t es[2] = {1, 1};
        if (enc(which == 0 ? &tk : &tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                const_cast<uint16_t *>(which == 0 ? a.k_cache : a.v_cache), dims, strides, box,
                es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
            CUDA_SUCCESS)
            return BDSA_CUDA_ERROR;
    }
    char *ws = static_cast<char *>(a.workspace);
    Params prm;
    prm.block_table = a.block_table;
    prm.seq_lens = a.seq_lens;
    prm.prefix = reinterpret_cast<const int32_t *>(ws + plan.off_prefix);
    prm.bad = reinterpret_cast<const int32_t *>(ws + plan.off_bad);
    prm.out = a.out;
    prm.lse = a.lse;
    prm.part_o = reinterpret_cast<float *>(ws + plan.off_part_o);
    prm.part_lse = reinterpret_cast<float *>(ws + plan.off_part_lse);
    prm.dev_status = a.dev_status;
    prm.max_pages = a.max_pages;
    prm.num_pages = a.num_pages;
    prm.bs = a.bs;
    prm.B = a.B;
    prm.Hq = a.Hq;
    prm.Hkv = a.Hkv;
    prm.G = G;
    prm.rows = G * a.B;
    prm.page_size = a.page_size;
    int lg = 0;
    while ((1 << lg) < a.page_size) ++lg;
    prm.log2_ps = lg;
    prm.box_rows = box_rows;
    prm.mode = a.mode;
    prm.scale_log2 = a.scale * 1.4426950408889634f;
    static bool attr_set = false;  // per (D, M) instantiation
    if (!attr_set) {
        if (cudaFuncSetAttribute(block_attn_kernel<D, M>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 C::kSmem) != cudaSuccess)
            return BDSA_CUDA_ERROR;
        attr_set = true;
    }
    attn_plan_kernel<<<1, 1024, 0, stream>>>(
        a.seq_lens, a.block_table, a.bs, a.B, a.max_pages, a.num_pages, a.page_size,
        reinterpret_cast<int32_t *>(ws + plan.off_prefix),
        reinterpret_cast<int32_t *>(ws + plan.off_bad), a.dev_status);
    if (cudaGetLastError() != cudaSuccess) return BDSA_CUDA_ERROR;
    if (launch_pdl(block_attn_kernel<D, M>, dim3(plan.grid), dim3(kThreads), C::kSmem, stream,
                   tq, tk, tv, prm) != cudaSuccess)
        return BDSA_CUDA_ERROR;
    if (launch_pdl(attn_merge_kernel<D>, dim3(plan.grid, kMergeSub), dim3(kMergeThreads), 0,
                   stream, prm, plan.grid) != cudaSuccess)
        return BDSA_CUDA_ERROR;
    return BDSA_OK;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

AttnPlan attn_plan(int bs, int B, int Hq, int Hkv, int D, int max_ctx_len, int num_sms) {
    (void)max_ctx_len;
    AttnPlan p;
    p.grid = num_sms > 0 ? num_sms : 1;
    p.rows = (Hq / Hkv) * B;
    size_t off = 0;
    p.off_prefix = off;
    off += align256((size_t)(bs + 1) * sizeof(int32_t));
    p.off_bad = off;
    off += align256((size_t)bs * sizeof(int32_t));
    p.off_part_lse = off;
    off += align256((size_t)2 * p.grid * p.rows * sizeof(float));
    p.off_part_o = off;
    off += align256((size_t)2 * p.grid * p.rows * D * sizeof(float));
    p.workspace = off;
    return p;
}

int launch_block_attn(const AttnArgs &a, cudaStream_t stream) {
    const AttnPlan plan = attn_plan(a.bs, a.B, a.Hq, a.Hkv, a.D, a.max_ctx_len, a.num_sms);
    if (a.workspace == nullptr || a.workspace_bytes < plan.workspace)
        return BDSA_WORKSPACE_TOO_SMALL;
    const bool m64 = (a.Hq / a.Hkv) * a.B <= 64;
    if (a.D == 128)
        return m64 ? launch_impl<128, 64>(a, plan, stream) : launch_impl<128, 128>(a, plan, stream);
    if (a.D == 64)
        return m64 ? launch_impl<64, 64>(a, plan, stream) : launch_impl<64, 128>(a, plan, stream);
    return BDSA_UNSUPPORTED;
}

}  // namespace bdsa
