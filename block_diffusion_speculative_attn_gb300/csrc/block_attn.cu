// block_attn.cu -- block attention over a paged KV cache for sm_103a.
//
// Computes, per request r, KV head h and block row i (query heads j = h*G + g):
//   o = softmax(scale * q k^T) v over keys t < limit(i), where
//   limit(i) = L_r + B (DRAFT: rectangular intra-block mask) or L_r + i + 1
//   (VERIFY: token-causal), as defined on "SGLang dLLM / LLaDA 2.0", section
//   "Attention Mask", and used by the draft/verify passes of "From DFlash to
//   dLLM Self-Spec (II)", sections 2.2.3-2.2.4 and "(IV)", section 4.4.1.
//
// One CTA owns one (request, KV head, KV split) unit:
//   * the G*B query rows of the unit (GQA heads x block rows, row m = i*G + g)
//     form the A operand of one tcgen05 MMA tile: M = 64 when G*B <= 64, else
//     M = 128 (zero rows pad it).  An M = 64 accumulator spreads its rows over
//     lanes 0-15 of all four TMEM lane quadrants, so all four SM sub-partitions
//     take part in the softmax with two threads per row (16x32bx2 TMEM
//     accesses); an M = 128 accumulator has one thread per row;
//   * K/V are streamed in 128-key tiles, one TMA box per page (or per 128 keys
//     of a large page) into 128-byte-swizzled shared memory, through a 3-deep
//     K ring and a 2-deep V ring;
//   * S = Q K^T (K = D) and O += P V (K = 128 keys) run on the tensor cores
//     with fp32 accumulators in TMEM (S double-buffered);
//   * softmax in the log2 domain: one FFMA + ex2 per score, running max with a
//     lazy rescale of O in TMEM only when the max grows by more than 2^8, P
//     rounded to bf16 and written swizzled for the PV MMA (double-buffered in
//     M = 64 mode so the next tile's P never waits for the previous PV);
//   * with several splits the CTA writes an fp32 partial (o / l, log2 lse) and
//     a second kernel merges them, so no CTA ever waits for another.
// Warp roles: 0-3 softmax/epilogue, 4 TMA producer, 5 MMA issuer + TMEM owner.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "bdsa_device.cuh"
#include "bdsa_internal.h"

namespace bdsa {
namespace {

constexpr int kBN = 128;                  // keys per tile
constexpr int kThreads = 192;
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kSoftmaxWarps = 4;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 256;          // S buffers at columns 0 and 128, O at 256
constexpr float kRescaleLog2 = 8.0f;      // rescale O only when the max grows by > 2^8
constexpr float kLn2 = 0.6931471805599453f;

template <int D, int M>
struct Cfg {
    static constexpr int DH = D / 64;               // 64-element (128-byte) slabs per row
    static constexpr int kSlab = M * 128;           // one M-row slab of 128-byte rows
    static constexpr int kKVSlab = kBN * 128;       // one 128-key slab
    static constexpr int NP = (M == 64) ? 2 : 1;    // P buffers
    static constexpr int NK = (D == 128) ? 3 : 4;
    static constexpr int NV = (D == 128) ? 2 : 4;
    static constexpr int TPR = (M == 64) ? 2 : 1;   // softmax threads per row
    static constexpr int NC = kBN / TPR;            // score columns per thread
    static constexpr int kStage = DH * kKVSlab;
    static constexpr int kPBuf = 2 * kSlab;         // 128 keys = two 64-key slabs
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kOffQ + DH * kSlab;
    static constexpr int kOffV = kOffK + NK * kStage;
    static constexpr int kOffP = kOffV + NV * kStage;
    static constexpr int kOffBar = kOffP + NP * kPBuf;
    // barrier indices
    static constexpr int QF = 0;
    static constexpr int KF = 1;
    static constexpr int KE = KF + NK;
    static constexpr int VF = KE + NK;
    static constexpr int VE = VF + NV;
    static constexpr int SF = VE + NV;    // 2: S buffer full
    static constexpr int SR = SF + 2;     // 2: S buffer released
    static constexpr int PF = SR + 2;     // P written (one per tile)
    static constexpr int PV = PF + 1;     // NP: PV done, per P buffer
    static constexpr int DR = PV + NP;    // drain
    static constexpr int kNumBars = DR + 1;
    static constexpr int kOffMisc = kOffBar + 8 * kNumBars;
    static constexpr int kSmem = kOffMisc + 16 + 1024;  // + slack to align the base to 1 KB
};

struct Params {
    const int32_t *block_table;
    const int32_t *seq_lens;
    uint16_t *out;
    float *lse;
    float *part_o;
    float *part_lse;
    int32_t *dev_status;
    int max_pages, num_pages, bs, B, Hq, Hkv, G, rows, page_size, log2_ps, box_rows, mode;
    int nsplit, tps;
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

// Loads this thread's share of a 128-column fp32 accumulator block from TMEM:
// all 128 columns of its lane (M = 128) or its half of the row (M = 64).
template <int M, int NC>
__device__ __forceinline__ void load_cols(uint32_t taddr, float (&v)[NC]) {
    if constexpr (M == 64) {
#pragma unroll
        for (int c = 0; c < NC / 32; ++c)
            tmem_ld16x2_32<NC>(taddr + c * 32, *reinterpret_cast<float(*)[32]>(&v[c * 32]));
    } else {
#pragma unroll
        for (int c = 0; c < NC / 32; ++c)
            tmem_ld32(taddr + c * 32, *reinterpret_cast<float(*)[32]>(&v[c * 32]));
    }
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
    const int s = blockIdx.x % prm.nsplit;
    const int h = (blockIdx.x / prm.nsplit) % prm.Hkv;
    const int r = blockIdx.x / (prm.nsplit * prm.Hkv);
    const int B = prm.B, G = prm.G;
    const int L = prm.seq_lens[r];
    const long n_keys = (long)L + B;
    const long ps = prm.page_size;
    const long ntiles = (n_keys + kBN - 1) / kBN;
    const long tb = (long)s * prm.tps;
    const long te = (s == prm.nsplit - 1) ? ntiles : min(ntiles, tb + prm.tps);
    const int nt = (int)max(0L, te - tb);

    // ---- validate every page id of the request (not only this split's), so a bad
    // entry skips all splits of the unit alike
    bool bad = (L < 0) || (n_keys > (long)prm.max_pages * ps);
    if (!bad) {
        const long last = (n_keys - 1) >> prm.log2_ps;
        const int32_t *bt = prm.block_table + (long)r * prm.max_pages;
        for (long pi = tid; pi <= last; pi += kThreads) {
            const int32_t pg = bt[pi];
            if (pg < 0 || pg >= prm.num_pages) bad = true;
        }
    }
    bad = __syncthreads_or(bad);
    if (bad || nt == 0) {
        if (bad && tid == 0) report_status(prm.dev_status, BDSA_DEVICE_OUT_OF_RANGE);
        for (int m = tid; m < prm.rows; m += kThreads) {
            const long token = (long)r * B + m / G;
            const long row = token * prm.Hq + (long)h * G + m % G;
            if (prm.nsplit == 1) {
                uint4 z = make_uint4(0, 0, 0, 0);
                uint4 *o = reinterpret_cast<uint4 *>(prm.out + row * D);
                for (int k = 0; k < D / 8; ++k) o[k] = z;
                if (prm.lse) prm.lse[row] = -INFINITY;
            } else {
                prm.part_lse[(long)s * prm.bs * B * prm.Hq + row] = -INFINITY;
            }
        }
        return;
    }

    auto bar = [&](int i) -> uint32_t { return sbase + C::kOffBar + 8u * (uint32_t)i; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kOffMisc + 4);

    if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(bar(C::QF), 1);
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
        }
        mbar_init(bar(C::PF), kSoftmaxWarps);
        for (int k = 0; k < C::NP; ++k) mbar_init(bar(C::PV + k), 1);
        mbar_init(bar(C::DR), 1);
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    // Zero the padding rows of the Q tile so padded S rows stay finite.
    if (prm.rows < M) {
        const int pad = M - prm.rows;
        for (int idx = tid; idx < pad * C::DH * 8; idx += kThreads) {
            const int u = idx & 7, c = (idx >> 3) % C::DH, m = prm.rows + (idx >> 3) / C::DH;
            st_shared_v4(sbase + C::kOffQ + c * C::kSlab + m * 128 + u * 16, 0, 0, 0, 0);
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kProducerWarp) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            mbar_arrive_expect_tx(bar(C::QF), (uint32_t)(prm.rows * D * 2));
            for (int c = 0; c < C::DH; ++c)
                tma_load_4d(sbase + C::kOffQ + c * C::kSlab, &tm_q, c * 64, 0, h, r * B,
                            bar(C::QF));
            const int32_t *bt = prm.block_table + (long)r * prm.max_pages;
            const int rows_box = prm.box_rows;
            int issued = 0;
            for (int jj = 0; jj < nt; ++jj) {
                const long t0 = (tb + jj) * kBN;
                const int valid = (int)min((long)kBN, n_keys - t0);
                const int nbox = (valid + rows_box - 1) / rows_box;
                const uint32_t bytes = (uint32_t)(nbox * rows_box * 128 * C::DH);
                const int ks = jj % C::NK;
                if (!mbar_wait(bar(C::KE + ks), ((jj / C::NK) & 1) ^ 1, abort_flag,
                               prm.dev_status))
                    break;
                mbar_arrive_expect_tx(bar(C::KF + ks), bytes);
                for (int b = 0; b < nbox; ++b) {
                    const long t = t0 + (long)b * rows_box;
                    const int32_t slot =
                        bt[t >> prm.log2_ps] * prm.page_size + (int32_t)(t & (ps - 1));
                    for (int c = 0; c < C::DH; ++c)
                        tma_load_2d(sbase + C::kOffK + ks * C::kStage + c * C::kKVSlab +
                                        b * rows_box * 128,
                                    &tm_k, h * D + c * 64, slot, bar(C::KF + ks));
                }
                const int vs = jj % C::NV;
                if (!mbar_wait(bar(C::VE + vs), ((jj / C::NV) & 1) ^ 1, abort_flag,
                               prm.dev_status)) {
                    issued = -(jj + 1);  // K of tile jj issued, V not
                    break;
                }
                mbar_arrive_expect_tx(bar(C::VF + vs), bytes);
                for (int b = 0; b < nbox; ++b) {
                    const long t = t0 + (long)b * rows_box;
                    const int32_t slot =
                        bt[t >> prm.log2_ps] * prm.page_size + (int32_t)(t & (ps - 1));
                    for (int c = 0; c < C::DH; ++c)
                        tma_load_2d(sbase + C::kOffV + vs * C::kStage + c * C::kKVSlab +
                                        b * rows_box * 128,
                                    &tm_v, h * D + c * 64, slot, bar(C::VF + vs));
                }
                issued = jj + 1;
            }
            // Drain: the last load issued into each stage must have landed before exit.
            const int nk_issued = issued >= 0 ? issued : -issued;
            const int nv_issued = issued >= 0 ? issued : -issued - 1;
            mbar_wait_drain(bar(C::QF), 0);
            for (int jj = max(0, nk_issued - C::NK); jj < nk_issued; ++jj)
                mbar_wait_drain(bar(C::KF + jj % C::NK), (jj / C::NK) & 1);
            for (int jj = max(0, nv_issued - C::NV); jj < nv_issued; ++jj)
                mbar_wait_drain(bar(C::VF + jj % C::NV), (jj / C::NV) & 1);
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_qk = idesc_bf16_f32(M, kBN, 0, 0);
            constexpr uint32_t idesc_pv = idesc_bf16_f32(M, D, 0, 1);
            auto issue_pv = [&](int j) -> bool {
                if (!mbar_wait(bar(C::PF), j & 1, abort_flag, prm.dev_status)) return false;
                const int vs = j % C::NV;
                if (!mbar_wait(bar(C::VF + vs), (j / C::NV) & 1, abort_flag, prm.dev_status))
                    return false;
                tc_fence_after();
                const int pb = j % C::NP;
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk) {
                    const uint64_t a = smem_desc_sw128(
                        sbase + C::kOffP + pb * C::kPBuf + (kk >> 2) * C::kSlab + (kk & 3) * 32,
                        16, 1024);
                    const uint64_t b = smem_desc_sw128(
                        sbase + C::kOffV + vs * C::kStage + kk * 16 * 128, C::kKVSlab, 1024);
                    umma_bf16(tmem + kTmemO, a, b, idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
                }
                umma_commit(bar(C::PV + pb));
                umma_commit(bar(C::VE + vs));
                return true;
            };
            bool ok = mbar_wait(bar(C::QF), 0, abort_flag, prm.dev_status);
            for (int jj = 0; ok && jj < nt; ++jj) {
                const int ks = jj % C::NK;
                ok = mbar_wait(bar(C::KF + ks), (jj / C::NK) & 1, abort_flag, prm.dev_status);
                if (!ok) break;
                const int sb = jj & 1;
                if (jj >= 2) {
                    ok = mbar_wait(bar(C::SR + sb), ((jj >> 1) - 1) & 1, abort_flag,
                                   prm.dev_status);
                    if (!ok) break;
                }
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t a = smem_desc_sw128(
                        sbase + C::kOffQ + (kk >> 2) * C::kSlab + (kk & 3) * 32, 16, 1024);
                    const uint64_t b = smem_desc_sw128(
                        sbase + C::kOffK + ks * C::kStage + (kk >> 2) * C::kKVSlab + (kk & 3) * 32,
                        16, 1024);
                    umma_bf16(tmem + sb * 128, a, b, idesc_qk, kk > 0 ? 1u : 0u);
                }
                umma_commit(bar(C::SF + sb));
                umma_commit(bar(C::KE + ks));
                if (jj >= 1) ok = issue_pv(jj - 1);
            }
            if (ok) ok = issue_pv(nt - 1);
            // Drain: every MMA issued above has completed before TMEM is released.
            umma_commit(bar(C::DR));
            mbar_wait_drain(bar(C::DR), 0);
        }
    } else {
        // ------------------------------------------------ softmax + epilogue
        // Thread -> (row, column half).  M = 128: row = tid, all 128 columns.
        // M = 64: row = 16 * warp + lane % 16, half = lane / 16 owns columns
        // [64 * half, 64 * half + 64) of every 128-column block.
        constexpr int NC = C::NC;
        const int half = (M == 64) ? (lane >> 4) : 0;
        const int row = (M == 64) ? warp * 16 + (lane & 15) : tid;
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        const int i_blk = row / G;
        const long limit =
            (prm.mode == BDSA_MODE_DRAFT) ? n_keys : min(n_keys, (long)L + i_blk + 1);
        const float sl2 = prm.scale_log2;
        float m_used = -INFINITY;
        float l4[4] = {0.f, 0.f, 0.f, 0.f};
        bool ok = true;
        for (int jj = 0; jj < nt; ++jj) {
            const long t0 = (tb + jj) * kBN;
            const int sb = jj & 1;
            ok = mbar_wait(bar(C::SF + sb), (jj >> 1) & 1, abort_flag, prm.dev_status);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            float sv[NC];
            load_cols<M, NC>(tmem + lane_base + sb * 128, sv);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::SR + sb));

            // mask the scores past this row's limit (raw scores; scale > 0 keeps the max)
            const long nvalid = limit - t0 - half * NC;
            if (nvalid < NC) {
#pragma unroll
                for (int k = 0; k < NC; ++k)
                    if (k >= nvalid) sv[k] = -INFINITY;
            }
            float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int k = 0; k < NC; ++k) mx[k & 3] = fmaxf(mx[k & 3], sv[k]);
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
                for (int k = 0; k < NC / 2; ++k) pk[k] = 0u;
            } else {
                const float neg_m = -m_used;
#pragma unroll
                for (int k = 0; k < NC / 2; ++k) {
                    const float p0 = ex2_approx(fmaf(sv[2 * k], sl2, neg_m));
                    const float p1 = ex2_approx(fmaf(sv[2 * k + 1], sl2, neg_m));
                    l4[k & 3] += p0 + p1;
                    pk[k] = pack_bf16x2(p0, p1);
                }
            }
            const int pb = jj % C::NP;
            // The P buffer must be free: PV of tile jj - NP has read it.
            if (jj >= C::NP) {
                const int prev = jj - C::NP;
                ok = mbar_wait(bar(C::PV + pb), (prev / C::NP) & 1, abort_flag, prm.dev_status);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
            }
            // A grown max rescales O, which needs PV of the previous tile to be done.
            if (jj >= 1 && __any_sync(0xffffffffu, resc)) {
                const int prev = jj - 1;
                ok = mbar_wait(bar(C::PV + prev % C::NP), (prev / C::NP) & 1, abort_flag,
                               prm.dev_status);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < D / (32 * C::TPR); ++c) {
                    float ov[32];
                    if constexpr (M == 64) {
                        tmem_ld16x2_32<D / 2>(tmem + lane_base + kTmemO + c * 32, ov);
                    } else {
                        tmem_ld32(tmem + lane_base + kTmemO + c * 32, ov);
                    }
                    tmem_wait_ld();
#pragma unroll
                    for (int k = 0; k < 32; ++k) ov[k] *= alpha;
                    if constexpr (M == 64) {
                        tmem_st16x2_32<D / 2>(tmem + lane_base + kTmemO + c * 32, ov);
                    } else {
                        tmem_st32(tmem + lane_base + kTmemO + c * 32, ov);
                    }
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
                    st_shared_v4(addr, pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
                }
            }
            // Ragged last tile: V rows past the request's keys hold stale or unloaded data.
            const long tile_keys = n_keys - t0;
            if (tile_keys < kBN) {
                const int vs = jj % C::NV;
                ok = mbar_wait(bar(C::VF + vs), (jj / C::NV) & 1, abort_flag, prm.dev_status);
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
            if (lane == 0) mbar_arrive(bar(C::PF));
        }
        if (ok) {
            const int last = nt - 1;
            ok = mbar_wait(bar(C::PV + last % C::NP), (last / C::NP) & 1, abort_flag,
                           prm.dev_status);
            ok = __all_sync(0xffffffffu, ok);
        }
        if (ok) {
            tc_fence_after();
            float l = (l4[0] + l4[1]) + (l4[2] + l4[3]);
            if constexpr (M == 64) l += __shfl_xor_sync(0xffffffffu, l, 16);
            const bool valid = row < prm.rows;
            const long token = (long)r * B + i_blk;
            const long orow = token * prm.Hq + (long)h * G + row % G;
            const float inv_l = l > 0.f ? 1.f / l : 0.f;
            constexpr int OC = D / C::TPR;  // output columns per thread
#pragma unroll
            for (int c = 0; c < OC / 32; ++c) {
                float ov[32];
                if constexpr (M == 64) {
                    tmem_ld16x2_32<D / 2>(tmem + lane_base + kTmemO + c * 32, ov);
                } else {
                    tmem_ld32(tmem + lane_base + kTmemO + c * 32, ov);
                }
                tmem_wait_ld();
                if (!valid) continue;
                const int col0 = half * OC + c * 32;
                if (prm.nsplit == 1) {
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
                        prm.part_o + ((long)s * prm.bs * B * prm.Hq + orow) * D + col0);
#pragma unroll
                    for (int v = 0; v < 8; ++v)
                        dst[v] = make_float4(ov[4 * v] * inv_l, ov[4 * v + 1] * inv_l,
                                             ov[4 * v + 2] * inv_l, ov[4 * v + 3] * inv_l);
                }
            }
            if (valid && half == 0) {
                const float lse2 = l > 0.f ? m_used + log2f(l) : -INFINITY;
                if (prm.nsplit == 1) {
                    if (prm.lse) prm.lse[orow] = lse2 * kLn2;
                } else {
                    prm.part_lse[(long)s * prm.bs * B * prm.Hq + orow] = lse2;
                }
            }
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

// Merge split-KV partials: one warp per (token, query head) row.
template <int D>
__global__ void __launch_bounds__(256)
    attn_combine_kernel(const float *__restrict__ part_o, const float *__restrict__ part_lse,
                        uint16_t *__restrict__ out, float *__restrict__ lse, int nsplit,
                        long rows_total) {
    const long row = ((long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (row >= rows_total) return;
    float m = -INFINITY;
    for (int s = lane; s < nsplit; s += 32) m = fmaxf(m, part_lse[s * rows_total + row]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    constexpr int E = D / 32;  // elements per lane
    float acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
    float den = 0.f;
    if (m != -INFINITY) {
        for (int s = 0; s < nsplit; ++s) {
            const float ls = part_lse[s * rows_total + row];
            if (ls == -INFINITY) continue;
            const float w = exp2f(ls - m);
            den += w;
            const float *src = part_o + (s * rows_total + row) * D + lane * E;
            if constexpr (E == 4) {
                const float4 v = *reinterpret_cast<const float4 *>(src);
                acc[0] += w * v.x;
                acc[1] += w * v.y;
                acc[2] += w * v.z;
                acc[3] += w * v.w;
            } else {
                const float2 v = *reinterpret_cast<const float2 *>(src);
                acc[0] += w * v.x;
                acc[1] += w * v.y;
            }
        }
    }
    const float inv = den > 0.f ? 1.f / den : 0.f;
    uint16_t *dst = out + row * D + lane * E;
    if constexpr (E == 4) {
        uint2 w;
        w.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
        w.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
        *reinterpret_cast<uint2 *>(dst) = w;
    } else {
        *reinterpret_cast<uint32_t *>(dst) = pack_bf16x2(acc[0] * inv, acc[1] * inv);
    }
    if (lse && lane == 0) lse[row] = den > 0.f ? (m + log2f(den)) * kLn2 : -INFINITY;
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
    Params prm;
    prm.block_table = a.block_table;
    prm.seq_lens = a.seq_lens;
    prm.out = a.out;
    prm.lse = a.lse;
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
    prm.nsplit = plan.nsplit;
    prm.tps = plan.tiles_per_split;
    prm.scale_log2 = a.scale * 1.4426950408889634f;
    const long rows_total = (long)a.bs * a.B * a.Hq;
    if (plan.nsplit > 1) {
        prm.part_o = static_cast<float *>(a.workspace);
        prm.part_lse = prm.part_o + (size_t)plan.nsplit * rows_total * D;
    } else {
        prm.part_o = nullptr;
        prm.part_lse = nullptr;
    }
    static bool attr_set = false;  // per (D, M) instantiation
    if (!attr_set) {
        if (cudaFuncSetAttribute(block_attn_kernel<D, M>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 C::kSmem) != cudaSuccess)
            return BDSA_CUDA_ERROR;
        attr_set = true;
    }
    const long grid_l = (long)a.bs * a.Hkv * plan.nsplit;
    if (grid_l > 0x7fffffffL) return BDSA_UNSUPPORTED;
    const unsigned grid = (unsigned)grid_l;
    block_attn_kernel<D, M><<<grid, kThreads, C::kSmem, stream>>>(tq, tk, tv, prm);
    if (cudaGetLastError() != cudaSuccess) return BDSA_CUDA_ERROR;
    if (plan.nsplit > 1) {
        const long threads = rows_total * 32;
        const unsigned cgrid = (unsigned)((threads + 255) / 256);
        attn_combine_kernel<D><<<cgrid, 256, 0, stream>>>(prm.part_o, prm.part_lse, a.out, a.lse,
                                                         plan.nsplit, rows_total);
        if (cudaGetLastError() != cudaSuccess) return BDSA_CUDA_ERROR;
    }
    return BDSA_OK;
}

}  // namespace

AttnPlan attn_plan(int bs, int B, int Hq, int Hkv, int D, int max_ctx_len, int num_sms) {
    AttnPlan p;
    const long units = (long)bs * Hkv;
    const long max_tiles = ((long)max_ctx_len + B + kBN - 1) / kBN;
    const long target = 2L * num_sms;  // one resident CTA per SM: aim for two waves
    long nsplit = 1;
    if (units < target) nsplit = (target + units - 1) / units;
    if (nsplit > max_tiles) nsplit = max_tiles;
    if (nsplit < 1) nsplit = 1;
    long tps = (max_tiles + nsplit - 1) / nsplit;
    if (tps < 1) tps = 1;
    nsplit = (max_tiles + tps - 1) / tps;
    if (nsplit < 1) nsplit = 1;
    p.nsplit = (int)nsplit;
    p.tiles_per_split = (int)tps;
    const size_t rows_total = (size_t)bs * B * Hq;
    p.workspace = nsplit > 1 ? (size_t)nsplit * rows_total * ((size_t)D + 1) * sizeof(float) : 0;
    return p;
}

int launch_block_attn(const AttnArgs &a, cudaStream_t stream) {
    const AttnPlan plan = attn_plan(a.bs, a.B, a.Hq, a.Hkv, a.D, a.max_ctx_len, a.num_sms);
    if (plan.workspace > 0 && (a.workspace == nullptr || a.workspace_bytes < plan.workspace))
        return BDSA_WORKSPACE_TOO_SMALL;
    const bool m64 = (a.Hq / a.Hkv) * a.B <= 64;
    if (a.D == 128)
        return m64 ? launch_impl<128, 64>(a, plan, stream) : launch_impl<128, 128>(a, plan, stream);
    if (a.D == 64)
        return m64 ? launch_impl<64, 64>(a, plan, stream) : launch_impl<64, 128>(a, plan, stream);
    return BDSA_UNSUPPORTED;
}

}  // namespace bdsa
