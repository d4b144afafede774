// block_attn.cu -- block attention over a paged KV cache for sm_103a.
//
// Computes, per request r, KV head h and block row i (query heads j = h*G + g):
//   o = softmax(scale * q k^T) v over keys t < limit(i), where
//   limit(i) = L_r + B (DRAFT: rectangular intra-block mask) or L_r + i + 1
//   (VERIFY: token-causal), as defined on "SGLang dLLM / LLaDA 2.0", section
//   "Attention Mask", and used by the draft/verify passes of "From DFlash to
//   dLLM Self-Spec (II)", sections 2.2.3-2.2.4 and "(IV)", section 4.4.1; or
//   (TREE) block key j visible to block row i iff bit j of tree_mask[r, i] is
//   set (the node and its ancestors: the tree attention of the Psi-Spec Tree
//   sampler, "Unlocking Lossless Speedups in LLMs via Discrete Diffusion").
//
// One call = one or two launches chained with programmatic dependent launch:
//   attend  persistent, one CTA per SM.  Every (request, KV head) unit is a run
//           of 128-key tiles; the runs are concatenated and each CTA takes an
//           equal contiguous range (stream-K style), so the work is balanced to
//           one tile.  Each CTA derives the schedule itself: its threads read
//           the context lengths, scan the per-request tile counts and locate
//           the CTA's first unit, then every role walks the units in order.  A
//           unit wholly inside one CTA is written directly; a unit cut between
//           CTAs leaves an fp32 partial (o / l and log2-sum-exp) in one of each
//           CTA's two slots.  The softmax warps check every page id a piece
//           references; a unit that references one outside the pool is written
//           as zeros (lse -inf) and reported.  With a grid no larger than the
//           device (and not a TREE call with the 128-row tile), a cut unit's
//           pieces other than its first are each the first piece of a later
//           CTA and are published early (a ready word carrying the call's
//           ticket); the CTA holding the first piece -- its last piece --
//           merges them into its own before writing the unit's output, so no
//           second launch;
//   merge   otherwise (TREE calls with the 128-row tile, or a grid larger than
//           the device): one CTA per range boundary that is a unit's first cut
//           merges the unit's partials in tile order, as soon as each is
//           published (128-row tile) or once the attention grid has finished.
//
// Inside a CTA (warp roles: the softmax + epilogue warps -- four with the
// 64-row tile, eight with the 128-row tile -- then the Q/K producer, the MMA
// issuer + TMEM owner, the V producer and, with the fused append, the append
// warp):
//   * the G*B query rows (row m = i*G + g) form the A operand of a tcgen05 MMA
//     tile: M = 64 when G*B <= 64, else M = 128 (zero rows pad it).  An M = 64
//     accumulator spreads its rows over lanes 0-15 of all four TMEM lane
//     quadrants, so all four SM sub-partitions run the softmax with two
//     threads per row (16x32bx2 TMEM accesses); with M = 128 warps w and w + 4
//     share lane quadrant w % 4 and take the two 64-column halves of a row,
//     exchanging row maxima and sums through shared memory;
//   * K and V tiles arrive by TMA, one box per page (or per 128 keys of a
//     larger page), into 128-byte-swizzled shared memory, through a K ring and
//     a deeper V ring fed by separate producer warps, with an L2 evict-first
//     policy since every K/V byte is read exactly once;
//   * S = Q K^T and O += P V run on the tensor cores with fp32 accumulators in
//     TMEM: two S buffers and two O buffers (512 columns), so consecutive units
//     overlap;
//   * softmax in the log2 domain: one ex2 per score, the scale, the row max
//     (three-input max) and the row sum on packed fp32 pairs, running max with
//     a lazy rescale of O in TMEM only when the max grows by more than 2^8, P
//     rounded to bf16 and written swizzled for the PV MMA.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdlib>
#include <chrono>
#include <mutex>
#include <utility>

#include "bdsa_device.cuh"
#include "bdsa_internal.h"

namespace bdsa {
namespace {

constexpr int kBN = 128;                  // keys per tile
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 256;          // S at columns 0 / 128, O at 256 / 384
constexpr float kRescaleLog2 = 8.0f;      // rescale O only when the max grows by > 2^8
constexpr float kLn2 = 0.6931471805599453f;

// W8: the 128-row tile with eight softmax warps, two threads a row: its
// 128-column softmax is bound by instruction latency, which one warp per SM
// sub-partition cannot hide (a large tree's row tiles, which read keys mostly
// from L2, most of all); the 64-row tile keeps four softmax warps.
template <int D, int M, bool W8 = false>
struct Cfg {
    static_assert(!W8 || M == 128, "eight softmax warps only with the 128-row tile");
    static constexpr int DH = D / 64;               // 64-element (128-byte) slabs per row
    static constexpr int kSlab = M * 128;           // one M-row slab of 128-byte rows
    static constexpr int kKVSlab = kBN * 128;       // one 128-key slab
    static constexpr int NQ = (M == 64) ? 2 : 1;    // Q buffers
    static constexpr int NP = (M == 64) ? 2 : 1;    // P buffers
    // V is held from its load until PV, K only until S: the deeper V ring lets
    // each V load start about three tiles before its PV (two with eight
    // softmax warps, whose keys come mostly from L2, to make room for the
    // row-statistics exchange).
    static constexpr int NK = (D == 128) ? 2 : 4;
    static constexpr int NV = (D == 128) ? (W8 ? 2 : 3) : 4;
    static constexpr int TPR = (M == 64 || W8) ? 2 : 1;  // softmax threads per row
    // warp roles: softmax warps first, then the Q/K producer, the MMA issuer,
    // the V producer and (with the fused append) the append warp
    static constexpr int SW = W8 ? 8 : 4;
    static constexpr int KPW = SW, MMAW = SW + 1, VPW = SW + 2, APW = SW + 3;
    static constexpr int kThreads = (SW + 3) * 32;
    static constexpr int kThreadsAppend = kThreads + 32;
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
    // M = 64 epilogue staging in the P buffers: every softmax warp wrote its
    // rows (EW), the tile store has read them (ER); one phase per piece.
    static constexpr int EW = OE + 2;
    static constexpr int ER = EW + 1;
    static constexpr int DR = ER + 1;     // drain
    // every softmax warp has fenced its stores of a partial piece; one phase
    // per partial piece, waited by thread 0 alone before it publishes the slot
    static constexpr int PB = DR + 1;
    // owner merge: every softmax warp has read the other pieces'
    // ready words; waited by thread 0 alone before it resets them
    static constexpr int MR = PB + 1;
    // W8: the two warps sharing a TMEM lane quadrant have written their halves
    // of an exchange (one barrier per pair of warps, a phase per exchange)
    static constexpr int XB = MR + 1;
    static constexpr int kNumBars = XB + (W8 ? 4 : 0);
    // W8: the two threads of a row exchange their row maxima (per tile) and
    // row sums (per piece) through shared memory, two buffers by exchange
    // parity
    static constexpr int kOffXch = kOffBar + 8 * kNumBars;
    static constexpr int kXchBytes = W8 ? 2 * 2 * 128 * 4 : 0;
    static constexpr int kOffMisc = kOffXch + kXchBytes;
    static constexpr int kOffMiscEnd = kOffMisc + 176;  // the schedule state (Sched)
    // + slack to align the base to 1 KB.  With D = 128 this is within a few
    // hundred bytes of the SM's shared memory less one merge CTA's, so that a
    // merge CTA can wait beside each attention CTA: keep both small.
    static constexpr int kSmem = kOffMiscEnd + 1024;
};

struct Params {
    const int32_t *block_table;
    const int32_t *seq_lens;
    int32_t *part_bad;       // [2 * grid] partial slot saw a page id outside the pool
    uint64_t *part_ready;    // [2 * grid] the call's ticket once the slot is written
    uint64_t ticket;         // this call's ticket (unique a call, never 0)
    uint64_t owner_ticket;   // the ticket the owner merge waits for (= ticket; see
                             // expire_owner_waits)
    int early_merge;         // M = 128: partials are published, the merge starts on them
    int owner_merge;         // the CTA holding a cut unit's first tile merges it
    uint16_t *out;
    float *lse;
    const uint64_t *tree_mask;  // TREE mode: [bs * B, mask_words] block keys visible to each row
    float *part_o;           // [2 * grid, rows, D]
    float *part_lse;         // [2 * grid, rows]
    int32_t *dev_status;
    uint64_t magic_S;        // floor((2^64 - 1) / grid), see range_start
    int max_pages, num_pages, bs, B, Hq, Hkv, G, rows, page_size, log2_ps, box_rows, mode;
    // Row tiles: a block of more rows than one tile (TREE with G * B > 128)
    // is cut into n_rt tiles of npt nodes, and the KV heads are folded into
    // the virtual requests: rv = (r * Hkv + h) * n_rt + t is request r's KV
    // head h, row tile t, one unit each (hu = 1), so that the row tiles that
    // read the same keys and values run back to back.  Otherwise n_rt = 1,
    // npt = B, rv = r and a virtual request has hu = Hkv units, one a head.
    int bs_v, n_rt, npt, hu;
    int mask_words;          // TREE: 64-bit words of a node's ancestor-or-self set
    int out_v8;              // out is 32-byte aligned: the M = 128 epilogue stores 32 bytes
    int unit_cost;           // virtual tiles a unit switch is charged in the schedule
    float scale_log2;
};

// The fused append's buffers, a kernel argument of their own (left out of
// Params, which the merge kernel shares).
struct AppendParams {
    const uint16_t *k_new;   // the block's own keys / values, [bs * B, Hkv, D]
    const uint16_t *v_new;
    uint16_t *k_cache;       // the caches they are written into
    uint16_t *v_cache;
};

__device__ __forceinline__ void st_release_gpu_u64(uint64_t *p, uint64_t v) {
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ uint64_t ld_acquire_gpu_u64(const uint64_t *p) {
    uint64_t v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// 32-byte global load bypassing L1 (one whole sector per lane); p 32-byte aligned.
__device__ __forceinline__ void ld_cg_v8(const float *p, float *v) {
    asm volatile("ld.global.cg.v8.f32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]),
                   "=f"(v[6]), "=f"(v[7])
                 : "l"(p)
                 : "memory");
}

// 32-byte global store (one whole sector per lane).
__device__ __forceinline__ void st_global_v8(void *p, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d, uint32_t e, uint32_t f, uint32_t g,
                                             uint32_t h) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(a),
                 "r"(b), "r"(c), "r"(d), "r"(e), "r"(f), "r"(g), "r"(h)
                 : "memory");
}

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

// Pairs of fp32 values in one 64-bit register, for the f32x2 arithmetic of
// the sm_100 family (two results per instruction), and the three-input max:
// the softmax at 128 columns a thread is bound by instruction issue, and
// these halve its max, scale and sum instructions.
__device__ __forceinline__ uint64_t f2_pack(float a, float b) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ float2 f2_unpack(uint64_t r) {
    float2 v;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(v.x), "=f"(v.y) : "l"(r));
    return v;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ float max3f(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
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


// 128-key tiles of a unit with nk keys (at least one, so that every unit has
// an epilogue).
__device__ __forceinline__ int tiles_of_keys(long nk) {
    return nk > 0 ? (int)min((nk + kBN - 1) / kBN, 1L << 24) : 1;
}

// Virtual request rv: its request, its first KV head (the head of unit u of
// rv is vreq_h0 + u), its first node (the row tile's), the context length
// and its key count -- the context and the block's first min(B, (t + 1) *
// npt) slots: a node sees only itself and its ancestors, all at lower block
// slots, so a row tile's keys end at its last node.  kRT: row tiles are
// possible (the TREE instantiations); otherwise a virtual request is a
// request, compiled as such.
template <bool kRT>
__device__ __forceinline__ int vreq_r(const Params &prm, int rv) {
    return (!kRT || prm.n_rt == 1) ? rv : rv / (prm.Hkv * prm.n_rt);
}
template <bool kRT>
__device__ __forceinline__ int vreq_h0(const Params &prm, int rv) {
    return (!kRT || prm.n_rt == 1) ? 0 : (rv / prm.n_rt) % prm.Hkv;
}
template <bool kRT>
__device__ __forceinline__ int vreq_node0(const Params &prm, int rv) {
    return (!kRT || prm.n_rt == 1) ? 0 : (rv % prm.n_rt) * prm.npt;
}
template <bool kRT>
__device__ __forceinline__ int vreq_L(const Params &prm, int rv) {
    return __ldg(prm.seq_lens + vreq_r<kRT>(prm, rv));
}
template <bool kRT>
__device__ __forceinline__ long vreq_keys(const Params &prm, int rv, long L) {
    if constexpr (!kRT) return L + prm.B;
    return L + min(prm.B, vreq_node0<kRT>(prm, rv) + prm.npt);
}
template <bool kRT>
__device__ __forceinline__ int vreq_count(const Params &prm) { return kRT ? prm.bs_v : prm.bs; }
template <bool kRT>
__device__ __forceinline__ int vreq_units(const Params &prm) { return kRT ? prm.hu : prm.Hkv; }

// Schedule.  Units (request, KV head) are concatenated in order; each unit is
// prm.unit_cost "virtual" tiles followed by its real tiles, and CTA b takes
// the cost range [b * Wc / S, (b + 1) * Wc / S).  The virtual tiles carry no
// work: they charge every unit switch (a Q load, an epilogue, a ragged last
// tile) about the time of unit_cost tiles, so a CTA that touches more units
// gets fewer tiles.  The real tiles inside a CTA's cost range form its range
// [x0, x1) of global tile indices.  The host picks the cost per call (see
// unit_cost_for).

// Schedule state (shared memory).
struct Sched {
    uint32_t tmem;           // attention: TMEM base address (written by tcgen05.alloc)
    int abort;               // attention: a bounded wait gave up
    int r0, u0, nt0, L0;     // the unit holding the CTA's cost start (if below Wc)
    long long u_off0;        // its first real tile
    long long cu0;           // its cost offset
    long long x0, x1, W, Wc;
    long long wsum[12];      // per-warp partial sums of the scan (<= 384 threads)
    int appended;            // attention with the fused append: 32 x pieces whose rows are written
};
static_assert(sizeof(Sched) <= 176, "the attention kernel keeps Sched in 176 bytes");

// The unit a role is working through, walked in (virtual request, unit)
// order; u is the unit's index within its virtual request.
struct Cursor {
    int r, u, nt, L;
    long u_off;  // global index of the unit's first tile
};

// A maximal run of one unit's tiles inside a CTA's range: r the virtual
// request, u the unit within it, h its KV head.
struct Piece {
    int r, u, h, a, e, nt, L;
    long u_off;
};

template <bool kRT>
__device__ __forceinline__ Piece piece_at(const Params &prm, const Cursor &c, long x, long x1) {
    Piece pc;
    pc.r = c.r;
    pc.u = c.u;
    pc.h = vreq_h0<kRT>(prm, c.r) + c.u;
    pc.nt = c.nt;
    pc.L = c.L;
    pc.u_off = c.u_off;
    pc.a = (int)(x - c.u_off);
    pc.e = (int)min((long)c.nt, (long)pc.a + (x1 - x));
    return pc;
}

// Start of CTA b's range and the CTA whose range holds global tile x.
// b * W / S without a 64-bit division (which the GPU emulates in software):
// magic = floor((2^64 - 1) / S) comes from the host, and the multiply-high
// quotient is at most one short for b * W < 2^63, which one step corrects.
__device__ __forceinline__ long range_start(int b, long W, int S, uint64_t magic) {
    if (b <= 0) return 0;
    const uint64_t n = (uint64_t)b * (uint64_t)W;
    uint64_t q = __umul64hi(n, magic);
    if (n - q * (uint64_t)S >= (uint64_t)S) ++q;
    return (long)q;
}

// Block-wide schedule of CTA b of S (NT threads): every thread sums the tile
// counts of a contiguous block of requests, a scan gives each block's first
// tile, and the threads whose blocks hold the CTA's cost bounds map them to
// real tiles.  Two __syncthreads; results in *sch.
template <int NT, bool kRT>
__device__ void schedule(const Params &prm, int b, int S, Sched *sch) {
    static_assert(NT % 32 == 0 && NT <= 384, "scan partials hold 12 warps");
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int bs = vreq_count<kRT>(prm);  // virtual requests
    const int per = (bs + NT - 1) / NT;
    const int i0 = min(bs, tid * per), i1 = min(bs, i0 + per);
    long long sum = 0;
    for (int i = i0; i < i1; ++i)
        sum += tiles_of_keys(vreq_keys<kRT>(prm, i, vreq_L<kRT>(prm, i)));
    long long inc = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const long long t = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += t;
    }
    if (lane == 31) sch->wsum[warp] = inc;
    __syncthreads();
    long long wex = 0, T = 0;
#pragma unroll
    for (int w = 0; w < NT / 32; ++w) {
        const long long v = sch->wsum[w];
        if (w < warp) wex += v;
        T += v;
    }
    const long long Hkv = vreq_units<kRT>(prm);  // units a virtual request
    const long long uc = prm.unit_cost;
    const long long W = Hkv * T, Wc = Hkv * (T + uc * bs);
    const long long c0 = range_start(b, Wc, S, prm.magic_S);
    const long long c1 = range_start(b + 1, Wc, S, prm.magic_S);
    const long long pre = wex + inc - sum;  // tiles before request i0
    // cost offset of request i: Hkv * (tiles before it + unit_cost * i)
    const long long clo = Hkv * (pre + uc * i0);
    const long long chi = Hkv * (pre + sum + uc * i1);
    for (int which = 0; which < 2; ++which) {
        const long long c = which == 0 ? c0 : c1;
        if (!(c < Wc && clo <= c && c < chi)) continue;
        long long tp = pre;  // tiles before request i
        for (int i = i0; i < i1; ++i) {
            const int L = vreq_L<kRT>(prm, i);
            const int nt = tiles_of_keys(vreq_keys<kRT>(prm, i, L));
            const long long ci = Hkv * (tp + uc * i);
            const long long span = nt + uc;  // cost of one unit of request i
            if (c < ci + Hkv * span) {
                const int h = (int)((c - ci) / span);
                const long long pos = (c - ci) - h * span;
                const long long u_off = Hkv * tp + (long long)h * nt;
                const long long x = u_off + max(0LL, pos - uc);
                if (which == 0) {
                    sch->r0 = i;
                    sch->u0 = h;
                    sch->nt0 = nt;
                    sch->L0 = L;
                    sch->u_off0 = u_off;
                    sch->cu0 = ci + (long long)h * span;
                    sch->x0 = x;
                } else {
                    sch->x1 = x;
                }
                break;
            }
            tp += nt;
        }
    }
    if (tid == 0) {
        if (c0 >= Wc) sch->x0 = W;
        if (c1 >= Wc) sch->x1 = W;
        sch->W = W;
        sch->Wc = Wc;
    }
    __syncthreads();
}

// Move the cursor past a finished unit.
template <bool kRT>
__device__ __forceinline__ void next_unit(Cursor &c, const Params &prm) {
    c.u_off += c.nt;
    if (++c.u == vreq_units<kRT>(prm)) {
        c.u = 0;
        if (++c.r < vreq_count<kRT>(prm)) {
            c.L = vreq_L<kRT>(prm, c.r);
            c.nt = tiles_of_keys(vreq_keys<kRT>(prm, c.r, c.L));
        }
    }
}
__device__ __forceinline__ int cta_of(long x, long W, int S) {
    return (int)(((x + 1) * (long)S - 1) / W);
}

constexpr int kMaxBoxes = kBN / 8;  // page_size >= 8

// Number of TMA boxes of tile t0 that hold keys of the request (never past its
// block-table row).
__device__ __forceinline__ int boxes_of(long n_keys, long t0, int rows_box, int log2_ps,
                                        int max_pages) {
    const long valid = max(0L, min((long)kBN, n_keys - t0));
    int nbox = (int)((valid + rows_box - 1) / rows_box);
    while (nbox > 0 && ((t0 + (long)(nbox - 1) * rows_box) >> log2_ps) >= max_pages) --nbox;
    return nbox;
}

// Fused append, one warp: the block's own keys and values of request r, KV
// head h at positions [p_lo, p_hi) -- the part of L..L+B-1 inside one piece of
// the schedule -- go to their cache slots (slot = page * ps + position % ps
// from the request's block-table row).  Rows on a page id outside the pool, or
// past the block-table row, are not written.  Each lane keeps kU 16-byte
// pieces of K and of V in flight.
template <int D>
__device__ void append_piece_rows(const Params &prm, const AppendParams &app, const int32_t *bt,
                                  int r, int h, long L, long t_lo, long t_hi, int lane) {
    const long p_lo = max(t_lo, L), p_hi = min(t_hi, L + prm.B);
    if (L < 0 || p_lo >= p_hi) return;
    constexpr int kChunks = D / 8;  // 16-byte pieces of one row
    constexpr int kU = 4;
    const int total = (int)(p_hi - p_lo) * kChunks;
    for (int base = 0; base < total; base += 32 * kU) {
        uint4 kv[kU], vv[kU];
        long off[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            off[u] = -1;
            const int idx = base + u * 32 + lane;
            if (idx >= total) continue;
            const long p = p_lo + idx / kChunks;
            const int c = idx % kChunks;
            const long src = (((long)r * prm.B + (p - L)) * prm.Hkv + h) * D + c * 8;
            kv[u] = __ldg(reinterpret_cast<const uint4 *>(app.k_new + src));
            vv[u] = __ldg(reinterpret_cast<const uint4 *>(app.v_new + src));
            const long page = p >> prm.log2_ps;
            if (page >= prm.max_pages) continue;
            const int32_t pg = __ldg(bt + page);
            if (pg < 0 || pg >= prm.num_pages) continue;
            const long slot = (long)pg * prm.page_size + (p & (prm.page_size - 1));
            off[u] = (slot * prm.Hkv + h) * D + c * 8;
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            if (off[u] < 0) continue;
            *reinterpret_cast<uint4 *>(app.k_cache + off[u]) = kv[u];
            *reinterpret_cast<uint4 *>(app.v_cache + off[u]) = vv[u];
        }
    }
}

// kTree: the TREE mask (block keys by tree_mask bits), in an instantiation of
// its own so that the DRAFT / VERIFY tile loop carries none of its code.
template <int D, int M, bool kAppend, bool kTree>
__global__ void __launch_bounds__(kAppend ? Cfg<D, M, M == 128>::kThreadsAppend
                                          : Cfg<D, M, M == 128>::kThreads,
                                  1)
    block_attn_kernel(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ CUtensorMap tm_out,
                      const __grid_constant__ CUtensorMap tm_part, const Params prm,
                      const AppendParams app) {
    constexpr bool W8 = M == 128;
    using C = Cfg<D, M, W8>;
    // the owner merge is compiled into every instantiation but the 128-row
    // TREE one, whose latency-bound softmax measured 5 % slower with it in
    constexpr bool kOwner = M == 64 || !kTree;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (sbase - raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int B = prm.B, G = prm.G;
    const long ps = prm.page_size;
    constexpr int NT = kAppend ? C::kThreadsAppend : C::kThreads;
    constexpr int kKProducerWarp = C::KPW, kMmaWarp = C::MMAW, kVProducerWarp = C::VPW;
    constexpr int kAppendWarp = C::APW, kSoftmaxWarps = C::SW;

    auto bar = [&](int i) -> uint32_t { return sbase + C::kOffBar + 8u * (uint32_t)i; };
    Sched *sch = reinterpret_cast<Sched *>(smem + C::kOffMisc);
    uint32_t *tmem_slot = &sch->tmem;
    volatile int *abort_flag = &sch->abort;

    // ---- prologue (overlaps the previous kernel under programmatic dependent launch)
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
        mbar_init(bar(C::EW), kSoftmaxWarps);
        mbar_init(bar(C::ER), 1);
        mbar_init(bar(C::DR), 1);
        mbar_init(bar(C::PB), kSoftmaxWarps);
        mbar_init(bar(C::MR), kSoftmaxWarps);
        if constexpr (W8) {
            for (int k = 0; k < 4; ++k) mbar_init(bar(C::XB + k), 2);
        }
        *abort_flag = 0;
        sch->appended = 0;
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
        for (int idx = tid; idx < C::NQ * C::DH * pad * 8; idx += NT) {
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

    // ---- inputs written by earlier kernels on the stream are read from here on
    grid_dependency_wait();
    // The merge kernel may start now: its schedule reads only this call's
    // inputs.  With the owner merge there is no merge kernel, and the next
    // kernel on the stream is left to start when this grid ends: launched
    // early, it made a Qwen3-8B-shaped step (prepare, attention, acceptance)
    // 8.5 us slower (89.4 against 80.9 us, A/B medians).
    if (!prm.owner_merge) grid_launch_dependents();
    const int S = gridDim.x;
    const int b = blockIdx.x;
    schedule<NT, kTree>(prm, b, S, sch);
    if (warp == kKProducerWarp && sch->x0 < sch->x1) {
        // Warm L2 with the block-table entries of this CTA's range: its first
        // request's row from the first tile's page (lanes 0-15, 512 entries)
        // and the next request's row (lanes 16-31), so that later page
        // lookups, at unit switches, hit L2.  Issued only now: the whole table
        // prefetched by every CTA at the start delayed the schedule's
        // context-length reads (Qwen3-8B-shaped verify call 64.3 -> 62.3 us
        // mean, A/B over 200 steps).
        const long r = (long)vreq_r<kTree>(prm, sch->r0) + (lane >> 4);
        const long p0 = (long)(((sch->x0 - sch->u_off0) * kBN) >> prm.log2_ps) & ~31L;
        const long e = (lane < 16 ? p0 : 0L) + (long)(lane & 15) * 32;  // 32 entries a line
        if (r < prm.bs && e < prm.max_pages)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(prm.block_table + r * prm.max_pages + e));
    }
    const long x0 = sch->x0, x1 = sch->x1;
    Cursor cur0;
    if (x0 < x1) {
        cur0.r = sch->r0;
        cur0.u = sch->u0;
        cur0.nt = sch->nt0;
        cur0.L = sch->L0;
        cur0.u_off = sch->u_off0;
    }

    if (warp == kKProducerWarp || warp == kVProducerWarp) {
        // ------------------------------------------------ TMA producers
        const bool is_k = warp == kKProducerWarp;
        if (lane == 0) {
            // Every K / V byte is read once, except by the row tiles of a large
            // tree, which read their (request, KV head)'s keys one after another.
            const uint64_t policy =
                prm.n_rt == 1 ? l2_policy_evict_first() : l2_policy_evict_normal();
            const int rows_box = prm.box_rows;
            const int NR = is_k ? C::NK : C::NV;
            const int FULL = is_k ? C::KF : C::VF;
            const int EMPTY = is_k ? C::KE : C::VE;
            const uint32_t dst0 = sbase + (is_k ? C::kOffK : C::kOffV);
            const void *tmap = is_k ? (const void *)&tm_k : (const void *)&tm_v;
            long g = 0, issued = 0, q_issued = 0;
            int k = 0;
            bool ok = true;
            Cursor cur = cur0;
            for (long x = x0; ok && x < x1; ++k) {
                const Piece pc = piece_at<kTree>(prm, cur, x, x1);
                if (is_k) {
                    const int qb = k % C::NQ;
                    if (k >= C::NQ) {
                        ok = mbar_wait(bar(C::QE + qb), ((k / C::NQ) - 1) & 1, abort_flag,
                                       prm.dev_status);
                        if (!ok) break;
                    }
                    mbar_arrive_expect_tx(bar(C::QF + qb), (uint32_t)(prm.rows * D * 2));
                    const int qtok = vreq_r<kTree>(prm, pc.r) * B + vreq_node0<kTree>(prm, pc.r);
                    for (int c = 0; c < C::DH; ++c)
                        tma_load_4d(sbase + C::kOffQ + qb * C::kQBuf + c * C::kSlab, &tm_q,
                                    c * 64, 0, pc.h, qtok, bar(C::QF + qb));
                    q_issued = k + 1;
                }
                const long n_keys = vreq_keys<kTree>(prm, pc.r, pc.L);
                const int32_t *bt =
                    prm.block_table + (long)vreq_r<kTree>(prm, pc.r) * prm.max_pages;
                // With the fused append, the first tile holding the block's
                // own rows waits until the append warp has written this piece.
                const int j_app = (kAppend && pc.L >= 0) ? max(pc.a, pc.L / kBN) : pc.e;
                for (int j = pc.a; j < pc.e; ++j, ++g) {
                    const long t0 = (long)j * kBN;
                    if (kAppend && j == j_app) {
                        ok = wait_counter_geq(&sch->appended, 32 * (k + 1), abort_flag,
                                              prm.dev_status);
                        if (!ok) break;
                    }
                    const int nbox = boxes_of(n_keys, t0, rows_box, prm.log2_ps, prm.max_pages);
                    // look the pages up before waiting for the stage
                    int32_t slot[kMaxBoxes];
#pragma unroll
                    for (int bx = 0; bx < kMaxBoxes; ++bx) {
                        const long t = t0 + (long)bx * rows_box;
                        if (bx < nbox)
                            slot[bx] =
                                bt[t >> prm.log2_ps] * prm.page_size + (int32_t)(t & (ps - 1));
                    }
                    const int st = (int)(g % NR);
                    ok = mbar_wait(bar(EMPTY + st), (uint32_t)(((g / NR) & 1) ^ 1), abort_flag,
                                   prm.dev_status);
                    if (!ok) break;
                    mbar_arrive_expect_tx(bar(FULL + st),
                                          (uint32_t)(nbox * rows_box * 128 * C::DH));
#pragma unroll
                    for (int bx = 0; bx < kMaxBoxes; ++bx) {
                        if (bx >= nbox) break;
                        for (int c = 0; c < C::DH; ++c)
                            tma_load_2d_hint(dst0 + st * C::kStage + c * C::kKVSlab +
                                                 bx * rows_box * 128,
                                             tmap, pc.h * D + c * 64, slot[bx], bar(FULL + st),
                                             policy);
                    }
                    issued = g + 1;
                }
                x += pc.e - pc.a;
                if (pc.e == pc.nt) next_unit<kTree>(cur, prm);
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
            Cursor cur = cur0;
            for (long x = x0; ok && x < x1; ++k) {
                const Piece pc = piece_at<kTree>(prm, cur, x, x1);
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
                if (pc.e == pc.nt) next_unit<kTree>(cur, prm);
            }
            if (ok && have) ok = issue_pv(pend);
            // Drain: every MMA issued above has completed before TMEM is released.
            umma_commit(bar(C::DR));
            mbar_wait_drain(bar(C::DR), 0);
        }
    } else if (kAppend && warp == kAppendWarp) {
        // ------------------------------------------------ fused append
        // Walks the CTA's pieces ahead of the producers: writes each piece's
        // block rows, fences them against the async proxy and counts the piece
        // (a release per lane) for the producers' TMA loads.
        Cursor cur = cur0;
        for (long x = x0; x < x1;) {
            const Piece pc = piece_at<kTree>(prm, cur, x, x1);
            append_piece_rows<D>(prm, app, prm.block_table + (long)pc.r * prm.max_pages, pc.r,
                                 pc.h, pc.L, (long)pc.a * kBN, (long)pc.e * kBN, lane);
            fence_proxy_async_global();
            red_release_add_shared(&sch->appended, 1);
            x += pc.e - pc.a;
            if (pc.e == pc.nt) next_unit<kTree>(cur, prm);
        }
    } else if (warp < kSoftmaxWarps) {
        // ------------------------------------------------ softmax + epilogue
        // Thread -> (row, column half).  M = 128: row = tid, all 128 columns.
        // M = 64: row = 16 * warp + lane % 16, half = lane / 16 owns columns
        // [64 * half, 64 * half + 64) of every 128-column block.
        constexpr int NC = C::NC;
        constexpr int OC = C::OC;
        // W8: warps w and w + 4 share TMEM lane quadrant w % 4 (rows
        // 32 (w % 4) + lane), warp w / 4 = half taking columns [64 half, 64
        // half + 64) of S and [half * OC, half * OC + OC) of O; the row's two
        // threads exchange row maxima and sums through xch (named barrier
        // 1 + w % 4 for the pair of warps).
        const int half = (M == 64) ? (lane >> 4) : (W8 ? (warp >> 2) : 0);
        const int row = (M == 64) ? warp * 16 + (lane & 15) : (W8 ? (warp & 3) * 32 + lane : tid);
        const uint32_t lane_base = (uint32_t)((W8 ? (warp & 3) : warp) * 32) << 16;
        const uint32_t s_col = W8 ? (uint32_t)(half * NC) : 0u;  // this thread's S columns
        const uint32_t o_col = W8 ? (uint32_t)(half * OC) : 0u;  // and O columns
        float *xch = reinterpret_cast<float *>(smem + C::kOffXch);
        // W8: exchange v with the row's other thread (exchange n of the pair
        // of warps uses buffer n % 2 and phase n of barrier XB + w % 4; a
        // bounded wait, so a pair whose other warp gave up ends too)
        int n_xch = 0;
        auto pair_exchange = [&](float v, float &other) -> bool {
            const int bufi = n_xch & 1;
            xch[(bufi * 2 + half) * 128 + row] = v;
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::XB + (warp & 3)));
            bool okx = mbar_wait(bar(C::XB + (warp & 3)), (uint32_t)(n_xch & 1), abort_flag,
                                 prm.dev_status);
            okx = __all_sync(0xffffffffu, okx);
            other = xch[(bufi * 2 + (half ^ 1)) * 128 + row];
            ++n_xch;
            return okx;
        };
        const float sl2 = prm.scale_log2;
        // (set per piece: a row tile's rows past the request's last node are
        // not real rows)
        bool valid_row = row < prm.rows;
        const int i_blk = row / G;  // node within the row tile
        // A piece's output: O from TMEM scaled by 1/l, to `out` (bf16) when the
        // piece is the whole unit (or the owner of a cut unit, which first
        // merges the unit's other pieces into madd), else to the CTA's
        // partial slot (fp32).
        struct Epi {
            long lastg, orow;
            float inv_l, lse2;
            int ob, slot, r, h, k;
            bool complete, owner, bad;
        };
        // Owner merge: the other pieces' share of this thread's output
        // columns, added to O * inv_l by the epilogue (zero for other pieces).
        float madd[OC];
        // M = 64: a piece's tile store reads the P buffers after the epilogue
        // returns; they are released before the next write to them.
        bool stage_busy = false;
        int n_stage = 0;  // pieces staged in the P buffers so far (phases of EW / ER)
        int n_pub = 0;    // partial pieces published so far (phases of PB)
        auto release_stage = [&]() -> bool {
            if (tid == 0) {
                bulk_wait_group_read0();
                mbar_arrive(bar(C::ER));
            }
            bool okr = mbar_wait(bar(C::ER), (uint32_t)((n_stage - 1) & 1), abort_flag,
                                 prm.dev_status);
            okr = __all_sync(0xffffffffu, okr);
            stage_busy = false;
            return okr;
        };
        auto epilogue = [&](const Epi &e) -> bool {
            bool okw = mbar_wait(bar(C::PV + (int)(e.lastg % C::NP)),
                                 (uint32_t)((e.lastg / C::NP) & 1), abort_flag, prm.dev_status);
            okw = __all_sync(0xffffffffu, okw);
            if (!okw) return false;
            tc_fence_after();
            const float sc = e.inv_l;
            const bool fin = e.complete || e.owner;  // this piece writes the unit's output
            const bool zero = fin && e.bad;  // zeros, whatever O holds (it may be NaN)
            // This thread's output columns [half * OC, half * OC + OC), read from
            // TMEM 32 at a time.
            auto load_chunk = [&](int c, float (&v32)[32]) {
                tmem_load_chunk<M, D / 2>(tmem + lane_base + kTmemO + e.ob * 128 + o_col + c * 32,
                                          v32);
                tmem_wait_ld();
                if (zero) {
#pragma unroll
                    for (int q = 0; q < 32; ++q) v32[q] = 0.f;
                }
            };
            // fp32 partial rows stored directly, 32 bytes a lane per instruction
            // (whole sectors; the partial slots are 256-byte aligned).
            auto store_partial_direct = [&]() {
#pragma unroll
                for (int c = 0; c < OC / 32; ++c) {
                    float v32[32];
                    load_chunk(c, v32);
                    if (!valid_row) continue;
                    const int col0 = half * OC + c * 32;
                    float *dst = prm.part_o + ((long)e.slot * prm.rows + row) * D + col0;
#pragma unroll
                    for (int v = 0; v < 4; ++v)
                        st_global_v8(dst + 8 * v, __float_as_uint(v32[8 * v] * sc),
                                     __float_as_uint(v32[8 * v + 1] * sc),
                                     __float_as_uint(v32[8 * v + 2] * sc),
                                     __float_as_uint(v32[8 * v + 3] * sc),
                                     __float_as_uint(v32[8 * v + 4] * sc),
                                     __float_as_uint(v32[8 * v + 5] * sc),
                                     __float_as_uint(v32[8 * v + 6] * sc),
                                     __float_as_uint(v32[8 * v + 7] * sc));
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(C::OE + e.ob));
            };
            if constexpr (M == 64) {
                if (fin || !prm.owner_merge) {
                    // Stage the rows in the two P buffers (free: the piece's last
                    // two PVs are done and the next tile's P is not written before
                    // this returns), 128-byte rows swizzled like the tensor maps,
                    // then one thread stores them with TMA: bf16 to `out` for a
                    // unit's output, fp32 to the partial slot otherwise.
                    const uint32_t stage = sbase + C::kOffP;
#pragma unroll
                    for (int c = 0; c < OC / 32; ++c) {
                        float v32[32];
                        load_chunk(c, v32);
                        if (!valid_row) continue;
                        const int col0 = half * OC + c * 32;
                        if (fin) {
                            // 32 bf16 = four 16-byte chunks of the 64-column slab
                            const uint32_t rbase = stage + (col0 >> 6) * C::kSlab + row * 128;
                            const int u0 = (col0 & 63) >> 3;
                            const float *ad = madd + c * 32;
#pragma unroll
                            for (int v = 0; v < 4; ++v)
                                st_shared_v4(
                                    rbase + (((u0 + v) ^ (row & 7)) << 4),
                                    pack_bf16x2(fmaf(v32[8 * v + 0], sc, ad[8 * v + 0]),
                                                fmaf(v32[8 * v + 1], sc, ad[8 * v + 1])),
                                    pack_bf16x2(fmaf(v32[8 * v + 2], sc, ad[8 * v + 2]),
                                                fmaf(v32[8 * v + 3], sc, ad[8 * v + 3])),
                                    pack_bf16x2(fmaf(v32[8 * v + 4], sc, ad[8 * v + 4]),
                                                fmaf(v32[8 * v + 5], sc, ad[8 * v + 5])),
                                    pack_bf16x2(fmaf(v32[8 * v + 6], sc, ad[8 * v + 6]),
                                                fmaf(v32[8 * v + 7], sc, ad[8 * v + 7])));
                        } else {
                            // 32 fp32 = one 128-byte row of a 32-column box
                            const uint32_t rbase = stage + (col0 >> 5) * C::kSlab + row * 128;
#pragma unroll
                            for (int v = 0; v < 8; ++v)
                                st_shared_v4(rbase + ((v ^ (row & 7)) << 4),
                                             __float_as_uint(v32[4 * v + 0] * sc),
                                             __float_as_uint(v32[4 * v + 1] * sc),
                                             __float_as_uint(v32[4 * v + 2] * sc),
                                             __float_as_uint(v32[4 * v + 3] * sc));
                        }
                    }
                    // the O buffer may take the next unit but one as soon as it is read
                    tc_fence_before();
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(bar(C::OE + e.ob));
                        mbar_arrive(bar(C::EW));
                    }
                    if (tid == 0) {
                        const bool okw2 = mbar_wait(bar(C::EW), (uint32_t)(n_stage & 1),
                                                    abort_flag, prm.dev_status);
                        if (okw2) {
                            if (fin) {
                                for (int sl = 0; sl < D / 64; ++sl)
                                    tma_store_4d(&tm_out, stage + sl * C::kSlab, sl * 64, 0, e.h,
                                                 e.r * B);
                            } else {
                                for (int bx = 0; bx < D / 32; ++bx)
                                    tma_store_2d(&tm_part, stage + bx * C::kSlab, bx * 32,
                                                 e.slot * prm.rows);
                            }
                            bulk_commit_group();
                        }
                    }
                    // The staging area is released (ER) before the next P write,
                    // by when the store has long read it.
                    stage_busy = true;
                    ++n_stage;
                } else {
                    // a piece the owner merges: published with direct stores below
                    store_partial_direct();
                }
            } else if (fin) {
                // M = 128: each thread stores its share of its row directly, 32
                // bytes a lane per instruction (whole sectors; out when it is
                // 32-byte aligned), the owner's the whole cut unit's
#pragma unroll
                for (int c = 0; c < OC / 32; ++c) {
                    float v32[32];
                    load_chunk(c, v32);
                    if (!valid_row) continue;
                    const int col0 = half * OC + c * 32;
                    uint32_t w[16];
                    if constexpr (kOwner) {
                        const float *ad = madd + c * 32;
#pragma unroll
                        for (int v = 0; v < 16; ++v)
                            w[v] = pack_bf16x2(fmaf(v32[2 * v], sc, ad[2 * v]),
                                               fmaf(v32[2 * v + 1], sc, ad[2 * v + 1]));
                    } else {
#pragma unroll
                        for (int v = 0; v < 16; ++v)
                            w[v] = pack_bf16x2(v32[2 * v] * sc, v32[2 * v + 1] * sc);
                    }
                    uint16_t *dst = prm.out + e.orow * D + col0;
                    if (prm.out_v8) {
                        st_global_v8(dst, w[0], w[1], w[2], w[3], w[4], w[5], w[6], w[7]);
                        st_global_v8(dst + 16, w[8], w[9], w[10], w[11], w[12], w[13], w[14],
                                     w[15]);
                    } else {
                        uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
                        for (int v = 0; v < 4; ++v)
                            d4[v] = make_uint4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(C::OE + e.ob));
            } else {
                store_partial_direct();
            }
            if (valid_row && half == 0) {
                if (fin && e.bad) {
                    if (prm.lse) prm.lse[e.orow] = -INFINITY;
                } else if (fin) {
                    if (prm.lse) prm.lse[e.orow] = e.lse2 * kLn2;
                } else {
                    prm.part_lse[(long)e.slot * prm.rows + row] = e.lse2;
                }
            }
            if (!fin && tid == 0) prm.part_bad[e.slot] = e.bad ? 1 : 0;
            if (!fin && (M == 128 || prm.owner_merge)) {
                // Publish the partial: once every softmax warp has arrived after
                // its stores of it (the arrival releases them at CTA scope),
                // thread 0 writes this call's ticket into the slot's ready word
                // with a GPU-scope release, which carries those stores with it;
                // the owner CTA, or the merge kernel (M = 128 without the owner
                // merge), may read the slot once it acquires the word.  Only
                // thread 0 waits, and boundedly.  (Without the owner merge,
                // M = 64 stores its partials with TMA tile stores, and its
                // merge kernel waits for the whole attention grid.)
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(C::PB));
                if (tid == 0) {
                    if (mbar_wait(bar(C::PB), (uint32_t)(n_pub & 1), abort_flag, prm.dev_status))
                        st_release_gpu_u64(prm.part_ready + e.slot, prm.ticket);
                }
                ++n_pub;
            }
            return true;
        };
        // Owner merge: before the epilogue of the piece holding a cut
        // unit's first tile -- always the last piece of this CTA -- fold in
        // the unit's other pieces.  Each is the first piece of a later CTA
        // (slot 2 * bb), published with a ready word carrying this call's
        // ticket; they are read in tile order as each word shows the ticket
        // (a bounded wait), combined in the log2 domain with this piece's
        // (m_used, l), and leave madd = the other pieces' share of the output
        // and e.inv_l, e.lse2, e.bad for the whole unit.  The words read are
        // then reset to 0, so a CUDA graph replaying this call's ticket never
        // finds one already set.
        int n_own = 0;  // units merged by this CTA as owner (phases of MR)
        auto owner_gather = [&](Epi &e, const Piece &pc, float lr) -> bool {
            const long long cu =
                (long long)pc.u_off +
                (long long)prm.unit_cost * ((long long)pc.r * vreq_units<kTree>(prm) + pc.u);
            const long long last = cu + prm.unit_cost + pc.nt - 1;  // cost of the unit's last tile
            const long long Wc = sch->Wc;
            float m_run = e.lse2;
            float s_own = m_run == -INFINITY ? 0.f : 1.f;
            float den = s_own;
            bool bad = e.bad, okg = true;
#pragma unroll
            for (int c = 0; c < OC; ++c) madd[c] = 0.f;
            int bb = b + 1;
            for (; okg && bb < S; ++bb) {
                const long long cb = range_start(bb, Wc, S, prm.magic_S);
                if (cb > last) break;
                if (cb >= range_start(bb + 1, Wc, S, prm.magic_S)) continue;  // empty range
                const int sl = 2 * bb;
                if (!valid_row) continue;
                const uint64_t *w = prm.part_ready + sl;
                if (ld_acquire_gpu_u64(w) != prm.owner_ticket) {
                    const uint64_t t0 = global_timer_ns();
                    while (ld_acquire_gpu_u64(w) != prm.owner_ticket) {
                        if (*abort_flag) {
                            okg = false;
                            break;
                        }
                        if (global_timer_ns() - t0 > kWaitLimitNs) {
                            *abort_flag = 1;
                            report_status(prm.dev_status, BDSA_DEVICE_TIMEOUT);
                            okg = false;
                            break;
                        }
                        __nanosleep(64);
                    }
                    if (!okg) break;
                }
                // this thread's OC columns of the row: 32-byte loads (whole
                // sectors), all in flight before the first is used
                const float *src = prm.part_o + ((long)sl * prm.rows + row) * D + half * OC;
                float po[OC];
#pragma unroll
                for (int v = 0; v < OC / 8; ++v) ld_cg_v8(src + 8 * v, &po[8 * v]);
                const float ls = __ldcg(prm.part_lse + (long)sl * prm.rows + row);
                bad = bad || __ldcg(prm.part_bad + sl) != 0;
                if (ls == -INFINITY) continue;  // no key of that piece is visible to the row
                const float m_new = fmaxf(m_run, ls);
                const float a = m_run == -INFINITY ? 0.f : exp2f(m_run - m_new);
                const float wj = exp2f(ls - m_new);
                s_own *= a;
                den = den * a + wj;
#pragma unroll
                for (int c = 0; c < OC; ++c) madd[c] = fmaf(madd[c], a, wj * po[c]);
                m_run = m_new;
            }
            // every softmax warp has read the words (a bounded wait on MR, one
            // phase per owned unit) before thread 0 resets them
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::MR));
            if (tid == 0 &&
                mbar_wait(bar(C::MR), (uint32_t)(n_own & 1), abort_flag, prm.dev_status)) {
                for (int q = b + 1; q < bb && q < S; ++q) {
                    const long long cb = range_start(q, Wc, S, prm.magic_S);
                    if (cb < range_start(q + 1, Wc, S, prm.magic_S))
                        prm.part_ready[2 * q] = 0ull;
                }
            }
            ++n_own;
            okg = __all_sync(0xffffffffu, okg);
            bad = __any_sync(0xffffffffu, bad);
            const bool good = !bad && den > 0.f;
            const float inv_den = good ? 1.f / den : 0.f;
            // (a bad piece's partial may hold anything, NaN included)
#pragma unroll
            for (int c = 0; c < OC; ++c) madd[c] = good ? madd[c] * inv_den : 0.f;
            e.inv_l = (good && lr > 0.f) ? s_own * inv_den / lr : 0.f;
            e.lse2 = good ? m_run + log2f(den) : -INFINITY;
            e.bad = bad;
            return okg;
        };
        long g = 0;
        int k = 0;
        bool ok = true;
        Cursor cur = cur0;
        for (long x = x0; ok && x < x1; ++k) {
            const Piece pc = piece_at<kTree>(prm, cur, x, x1);
            const long n_keys = vreq_keys<kTree>(prm, pc.r, pc.L);
            const int rr = vreq_r<kTree>(prm, pc.r);              // the request
            const int node = vreq_node0<kTree>(prm, pc.r) + i_blk;  // this row's block slot
            valid_row = row < prm.rows && node < B;
            // Page ids this piece references: a context that needs more pages
            // than the block-table row holds (for the whole block, so every row
            // tile of a request agrees), or an id outside the pool, makes the
            // unit's output zeros.  Each tile's ids are loaded during the tile
            // and checked during the next one (or the epilogue).
            const bool shape_bad =
                pc.L < 0 || ((long)pc.L + B + ps - 1) / ps > (long)prm.max_pages;
            const int32_t *bt_row = prm.block_table + (long)rr * prm.max_pages;
            bool page_bad = false, pend = false;
            int32_t pend_pg = 0;
            const long limit = (kTree || prm.mode == BDSA_MODE_DRAFT)
                                   ? n_keys
                                   : min(n_keys, (long)pc.L + i_blk + 1);
            // TREE: the block keys this row's node sees (itself and its
            // ancestors), mask_words words from mrow
            const uint64_t *mrow = nullptr;
            if constexpr (kTree) {
                if (valid_row) mrow = prm.tree_mask + ((long)rr * B + node) * prm.mask_words;
            }
            const int ob = k & 1;
            float m_used = -INFINITY;
            // Partial sums of the scores' exponentials, two packed pairs.
            // TREE: lacc[0] holds them (the lse) and lacc[1] the same values
            // rounded to bf16 as the PV product sees them (the normalisation,
            // so that o is a convex combination of V rows: a row that sees few
            // keys, as in a short tree, is then within rounding of its
            // dominant V row).
            uint64_t lacc[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
            for (int j = pc.a; j < pc.e; ++j, ++g) {
                const long t0 = (long)j * kBN;
                const int sb = (int)(g & 1);
                // TREE: the mask words this tile's block keys need (at most
                // three from word wb), loaded before the wait for S
                long moff = 0;
                int wb = 0;
                uint64_t mw0 = 0ull, mw1 = 0ull, mw2 = 0ull;
                if constexpr (kTree) {
                    moff = t0 + half * NC - pc.L;  // block slot of this thread's column 0
                    if (moff + NC > 0 && mrow != nullptr) {
                        wb = (int)(max(moff, 0L) >> 6);
                        const int W = prm.mask_words;
                        if (wb < W) mw0 = __ldg(mrow + wb);
                        if (wb + 1 < W) mw1 = __ldg(mrow + wb + 1);
                        if (wb + 2 < W) mw2 = __ldg(mrow + wb + 2);
                    }
                }
                if (pend) page_bad |= pend_pg < 0 || pend_pg >= prm.num_pages;
                {
                    const long kend = min(t0 + kBN, n_keys);
                    const long p0 = t0 >> prm.log2_ps;
                    pend = !shape_bad && kend > t0 && p0 + lane <= ((kend - 1) >> prm.log2_ps);
                    if (pend) pend_pg = __ldg(bt_row + p0 + lane);
                }
                ok = mbar_wait(bar(C::SF + sb), (uint32_t)((g >> 1) & 1), abort_flag,
                               prm.dev_status);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc_fence_after();
                float sv[NC];
#pragma unroll
                for (int c = 0; c < NC / 32; ++c)
                    tmem_load_chunk<M, NC>(tmem + lane_base + sb * 128 + s_col + c * 32,
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
                if constexpr (kTree) {
                    if (moff + NC > 0) {
                        // visibility of this thread's columns, 64 to a word: context
                        // keys (slot < 0) visible, block keys by the row's mask
                        // (bits past the tree are 0; keys past the row tile's
                        // last node are already masked by the limit)
#pragma unroll
                        for (int wd = 0; wd < NC / 64; ++wd) {
                            const long o = moff + 64 * wd;
                            uint64_t vis = ~0ull;
                            if (o < 0) {
                                if (o > -64) vis = (mw0 << (-o)) | ((1ull << (-o)) - 1ull);
                            } else {
                                const int w = (int)(o >> 6) - wb, sh = (int)(o & 63);
                                const uint64_t lo = w == 0 ? mw0 : (w == 1 ? mw1 : mw2);
                                const uint64_t hi = w == 0 ? mw1 : (w == 1 ? mw2 : 0ull);
                                vis = sh ? (lo >> sh) | (hi << (64 - sh)) : lo;
                            }
                            const uint32_t vlo = (uint32_t)vis, vhi = (uint32_t)(vis >> 32);
#pragma unroll
                            for (int c = 0; c < 32; ++c) {
                                if (!((vlo >> c) & 1u)) sv[64 * wd + c] = -INFINITY;
                                if (!((vhi >> c) & 1u)) sv[64 * wd + 32 + c] = -INFINITY;
                            }
                        }
                    }
                }
                float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int c = 0; c < NC; c += 2)
                    mx[(c >> 1) & 3] = max3f(mx[(c >> 1) & 3], sv[c], sv[c + 1]);
                float mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
                if constexpr (M == 64) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 16));
                if constexpr (W8) {
                    float mo;
                    ok = pair_exchange(mt, mo);
                    if (!ok) break;
                    mt = fmaxf(mt, mo);
                }
                const float m_new = mt * sl2;
                float alpha = 1.f;
                bool resc = false;
                if (m_new > m_used + kRescaleLog2) {
                    alpha = ex2_approx(m_used - m_new);
                    m_used = m_new;
                    resc = true;
                }
                {
                    const uint64_t a2 = f2_pack(alpha, alpha);
                    lacc[0] = f2_mul(lacc[0], a2);
                    lacc[1] = f2_mul(lacc[1], a2);
                }
                uint32_t pk[NC / 2];
                if (m_used == -INFINITY) {
#pragma unroll
                    for (int c = 0; c < NC / 2; ++c) pk[c] = 0u;
                } else {
                    const float neg_m = -m_used;
                    const uint64_t sc2 = f2_pack(sl2, sl2), nm2 = f2_pack(neg_m, neg_m);
#pragma unroll
                    for (int c = 0; c < NC / 2; ++c) {
                        const float2 xv =
                            f2_unpack(f2_fma(f2_pack(sv[2 * c], sv[2 * c + 1]), sc2, nm2));
                        const float p0 = ex2_approx(xv.x);
                        const float p1 = ex2_approx(xv.y);
                        const uint32_t pr = pack_bf16x2(p0, p1);
                        pk[c] = pr;
                        if constexpr (kTree) {
                            lacc[0] = f2_add(lacc[0], f2_pack(p0, p1));
                            lacc[1] = f2_add(lacc[1], f2_pack(__uint_as_float(pr << 16),
                                                              __uint_as_float(pr & 0xffff0000u)));
                        } else {
                            lacc[c & 1] = f2_add(lacc[c & 1], f2_pack(p0, p1));
                        }
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
                        const uint32_t ta = tmem + lane_base + kTmemO + ob * 128 + o_col + c * 32;
                        tmem_load_chunk<M, D / 2>(ta, ov);
                        tmem_wait_ld();
#pragma unroll
                        for (int q = 0; q < 32; ++q) ov[q] *= alpha;
                        tmem_store_chunk<M, D / 2>(ta, ov);
                    }
                    tmem_wait_st();
                }
                // P row -> shared memory, K-major with the 128-byte swizzle.
                if (stage_busy) {
                    ok = release_stage();
                    if (!ok) break;
                }
                {
                    const uint32_t pbase = sbase + C::kOffP + pb * C::kPBuf;
#pragma unroll
                    for (int u = 0; u < NC / 8; ++u) {
                        const int slab = (C::TPR == 2) ? half : (u >> 3);
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
                    if (tid < kBN && tid >= tile_keys) {
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

            // ---- end of the piece
            {
                const float2 la = f2_unpack(lacc[0]), lb = f2_unpack(lacc[1]);
                float l, lr;
                if constexpr (kTree) {
                    l = la.x + la.y;
                    lr = lb.x + lb.y;
                    if constexpr (M == 64) lr += __shfl_xor_sync(0xffffffffu, lr, 16);
                    if constexpr (W8) {
                        float o1, o2;
                        ok = pair_exchange(lr, o1);
                        ok = ok && pair_exchange(l, o2);
                        if (!ok) break;
                        lr += o1;
                        l += o2;
                    }
                } else {
                    l = (la.x + la.y) + (lb.x + lb.y);
                    if constexpr (W8) {
                        float o2;
                        ok = pair_exchange(l, o2);
                        if (!ok) break;
                        l += o2;
                    }
                }
                if constexpr (M == 64) l += __shfl_xor_sync(0xffffffffu, l, 16);
                if constexpr (!kTree) lr = l;
                if (pend) page_bad |= pend_pg < 0 || pend_pg >= prm.num_pages;
                Epi e;
                e.lastg = g - 1;
                e.ob = ob;
                e.inv_l = lr > 0.f ? 1.f / lr : 0.f;
                e.lse2 = l > 0.f ? m_used + log2f(l) : -INFINITY;
                e.complete = pc.a == 0 && pc.e == pc.nt;
                e.owner = kOwner && prm.owner_merge && pc.a == 0 && pc.e < pc.nt;
                // every warp checked every page of the piece
                e.bad = shape_bad || __any_sync(0xffffffffu, page_bad);
                e.orow = ((long)rr * B + node) * prm.Hq + (long)pc.h * G + row % G;
                e.slot = 2 * b + (k == 0 ? 0 : 1);
                e.r = rr;  // (the 64-row tile has one row tile: rr * B is its first token)
                e.h = pc.h;
                e.k = k;
                if (e.bad && tid == 0) report_status(prm.dev_status, BDSA_DEVICE_OUT_OF_RANGE);
                if constexpr (kOwner) {
                    if (e.owner) {
                        ok = owner_gather(e, pc, lr);
                        if (!ok) break;
                    } else {
#pragma unroll
                        for (int c = 0; c < OC; ++c) madd[c] = 0.f;
                    }
                }
                ok = epilogue(e);
                if (!ok) break;
            }
            x += pc.e - pc.a;
            if (pc.e == pc.nt) next_unit<kTree>(cur, prm);
        }
    }

    if (tid == 0) bulk_wait_group0();  // epilogue tile stores complete
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// Merge the partials of every unit cut between CTAs.  Block b handles the
// unit whose first interior cut is the start of attention CTA b's range: it
// derives that unit and the slots of its pieces from the context lengths (the
// same schedule as the attention kernel, computed while the attention runs),
// waits until each piece's ready word carries the call's ticket, then merges
// the pieces in tile order, and ends with griddepcontrol.wait.  Four
// threads share a row, their 16-byte columns interleaved so each warp load
// reads whole 32-byte sectors, and walk the pieces with all of a piece's
// loads in flight.  A unit any of whose pieces saw a page id outside the pool
// is written as zeros (lse -inf).
constexpr int kMergeThreads = 256;
constexpr int kMergeTPR = 4;      // threads per row
constexpr int kMergeSlots = 16;   // piece slots listed in shared memory
constexpr uint64_t kMergeWaitNs = 20000000ull;  // 20 ms, then wait for the whole grid

// At most 64 registers a thread (launch bound of 4 CTAs an SM): two merge warps
// must fit on each SM sub-partition beside two attention warps, so that the
// merge CTAs become resident, and compute the schedule, while the attention
// grid still runs.
template <int D, bool kRT>
__global__ void __launch_bounds__(kMergeThreads, 4) attn_merge_kernel(const Params prm) {
    __shared__ Sched sch;
    __shared__ int s_slot[kMergeSlots];
    __shared__ int s_np;
    const int b = blockIdx.x, S = gridDim.x;
    schedule<kMergeThreads, kRT>(prm, b, S, &sch);
    const long W = sch.W, Wc = sch.Wc, x0 = sch.x0;
    // This grid must complete after the attention grid, so that a kernel that
    // waits on it sees every row: with published partials every CTA ends with
    // griddepcontrol.wait; otherwise the merging CTAs wait before they start,
    // and CTA 0 waits even when it has nothing to merge.
    const bool hold = prm.early_merge || b == 0;
    if (x0 >= W) {
        if (hold) grid_dependency_wait();
        return;
    }
    const long u_off = sch.u_off0, cu = sch.cu0;
    // the cut at this CTA's start splits the unit's tiles, and CTA b - 1 holds
    // the unit's first tile (so this is the unit's first cut)
    if (!(u_off < x0 && range_start(b - 1, Wc, S, prm.magic_S) <= cu + prm.unit_cost)) {
        if (hold) grid_dependency_wait();
        return;
    }
    const int rv = sch.r0, h = vreq_h0<kRT>(prm, rv) + sch.u0;
    const int r = vreq_r<kRT>(prm, rv), node0 = vreq_node0<kRT>(prm, rv);
    const int b_first = cta_of(cu + prm.unit_cost, Wc, S);
    const int b_last = cta_of(cu + prm.unit_cost + sch.nt0 - 1, Wc, S);
    // Partial slots of the unit's pieces, in tile order.  Every CTA from
    // b_first to b_last with a non-empty cost range holds one; it is that
    // CTA's first piece (slot 2bb) unless tiles of an earlier unit precede it
    // in the range (2bb + 1).
    if (threadIdx.x == 0) {
        int n = 0;
        for (int bb = b_first; bb <= b_last && n < kMergeSlots; ++bb) {
            const long cb = range_start(bb, Wc, S, prm.magic_S);
            if (cb < range_start(bb + 1, Wc, S, prm.magic_S))
                s_slot[n++] = 2 * bb + (cb >= cu ? 0 : 1);
        }
        s_np = n;
    }
    // Wait until every piece of the unit is published (ready word == this
    // call's ticket, written after the piece's stores and a GPU-wide fence),
    // so that the merge overlaps the attention CTAs still streaming.  All the
    // attention CTAs are resident (this grid starts only once each of them has
    // passed its launch_dependents), so the words do get written; the wait is
    // still bounded, and past the limit the merge waits for the whole
    // attention grid instead, by when every slot is final.
    if (!prm.early_merge) {
        grid_dependency_wait();  // the attention grid's partials
    } else if (threadIdx.x == 0) {
        const uint64_t t0 = global_timer_ns();
        bool late = false;
        for (int bb = b_first; bb <= b_last && !late; ++bb) {
            const long cb = range_start(bb, Wc, S, prm.magic_S);
            if (!(cb < range_start(bb + 1, Wc, S, prm.magic_S))) continue;
            const uint64_t *w = prm.part_ready + 2 * bb + (cb >= cu ? 0 : 1);
            while (ld_acquire_gpu_u64(w) != prm.ticket) {
                if (global_timer_ns() - t0 > kMergeWaitNs) {
                    late = true;
                    break;
                }
                __nanosleep(256);
            }
        }
        if (late) grid_dependency_wait();
    }
    __syncthreads();
    const int np = s_np;
    constexpr int C4 = D / 4;
    constexpr int F4 = C4 / kMergeTPR;  // 16-byte columns per thread
    const int items = prm.rows * kMergeTPR;
    for (int it = threadIdx.x; it < items; it += kMergeThreads) {
        const int row = it / kMergeTPR, sub = it % kMergeTPR;
        float mmax = -INFINITY, den = 0.f;
        float4 acc[F4];
#pragma unroll
        for (int v = 0; v < F4; ++v) acc[v] = make_float4(0.f, 0.f, 0.f, 0.f);
        bool bad = false;
        // pieces past the listed ones (only when a unit spans more than
        // kMergeSlots CTAs) are enumerated on the fly, after the last listed CTA
        int bb_next = np > 0 ? s_slot[np - 1] / 2 + 1 : b_first;
        for (int q = 0;; ++q) {
            int sl;
            if (q < np) {
                sl = s_slot[q];
            } else {
                if (np < kMergeSlots) break;
                while (bb_next <= b_last && range_start(bb_next, Wc, S, prm.magic_S) >=
                                               range_start(bb_next + 1, Wc, S, prm.magic_S))
                    ++bb_next;
                if (bb_next > b_last) break;
                const long cb = range_start(bb_next, Wc, S, prm.magic_S);
                sl = 2 * bb_next + (cb >= cu ? 0 : 1);
                ++bb_next;
            }
            const float4 *src =
                reinterpret_cast<const float4 *>(prm.part_o + ((long)sl * prm.rows + row) * D);
            float4 po[F4];
#pragma unroll
            for (int v = 0; v < F4; ++v) po[v] = __ldcg(src + sub + kMergeTPR * v);
            const float ls = __ldcg(prm.part_lse + (long)sl * prm.rows + row);
            bad = bad || __ldcg(prm.part_bad + sl) != 0;
            if (ls == -INFINITY) continue;  // no key of this piece is visible to the row
            const float m_new = fmaxf(mmax, ls);
            const float sc = (mmax == -INFINITY) ? 0.f : exp2f(mmax - m_new);
            const float w = exp2f(ls - m_new);
            den = den * sc + w;
#pragma unroll
            for (int v = 0; v < F4; ++v) {
                acc[v].x = acc[v].x * sc + w * po[v].x;
                acc[v].y = acc[v].y * sc + w * po[v].y;
                acc[v].z = acc[v].z * sc + w * po[v].z;
                acc[v].w = acc[v].w * sc + w * po[v].w;
            }
            mmax = m_new;
        }
        const bool ok = den > 0.f && !bad;
        const float inv = ok ? 1.f / den : 0.f;
        const int node = node0 + row / prm.G;
        if (node >= prm.B) continue;  // a row tile's rows past the last node
        const long orow = ((long)r * prm.B + node) * prm.Hq + (long)h * prm.G + row % prm.G;
        uint2 *dst = reinterpret_cast<uint2 *>(prm.out + orow * D);
#pragma unroll
        for (int v = 0; v < F4; ++v) {
            uint2 w2 = make_uint2(0u, 0u);  // a bad unit's partials may hold anything
            if (ok) {
                w2.x = pack_bf16x2(acc[v].x * inv, acc[v].y * inv);
                w2.y = pack_bf16x2(acc[v].z * inv, acc[v].w * inv);
            }
            dst[sub + kMergeTPR * v] = w2;
        }
        if (sub == 0 && prm.lse) prm.lse[orow] = ok ? (mmax + log2f(den)) * kLn2 : -INFINITY;
    }
    if (prm.early_merge) grid_dependency_wait();
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

// A ticket unique to each call and never 0: a partial slot's ready word holds
// the ticket of the call that last wrote it, so it cannot show the current
// call's ticket before this call publishes the slot.  The counter starts at a
// value mixed from the clock (the splitmix64 finaliser), so that a workspace
// left by another process is as unlikely to match.
uint64_t next_ticket() {
    static std::atomic<uint64_t> counter{[] {
        uint64_t x = (uint64_t)std::chrono::steady_clock::now().time_since_epoch().count();
        x += 0x9E3779B97F4A7C15ull;
        x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ull;
        x = (x ^ (x >> 27)) * 0x94D049BB133111EBull;
        return x ^ (x >> 31);
    }()};
    uint64_t t;
    do {
        t = counter.fetch_add(1, std::memory_order_relaxed) + 1;
    } while (t == 0);
    return t;
}

// Test hook for the bounded waits: with BDSA_TEST_EXPIRE_OWNER_WAITS=1 in the
// environment, the owner merge (64-row tile) waits for a ticket no CTA
// publishes, so each owner CTA gives up after the wait limit (1 s), records
// BDSA_DEVICE_TIMEOUT in dev_status and exits cleanly (no copy or MMA in
// flight: its other pieces are done); the units it owns are left unwritten.
// Read at every call; never set outside tests.
bool expire_owner_waits() {
    const char *v = getenv("BDSA_TEST_EXPIRE_OWNER_WAITS");
    return v != nullptr && v[0] == '1' && v[1] == '\0';
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

// Virtual tiles a unit switch costs in the schedule (A/B over the bench's
// workloads against the cost two, which every tile size had before): three
// for the DRAFT / VERIFY tiles (Qwen3-8B-shaped verify call 64.5 -> 63.7 us,
// long-context verify 331.2 -> 330.0 us, LLaDA2.0-style draft and Uno within
// noise) and four for TREE calls, whose units are short row tiles (481-node
// trees 1053 -> 994 us; three: 1009, five: 998).
int unit_cost_for(int M, bool tree) {
    (void)M;
    return tree ? 4 : 3;
}

template <int D, int M>
int launch_impl(const AttnArgs &a, const AttnPlan &plan, cudaStream_t stream) {
    using C = Cfg<D, M, M == 128>;
    EncodeTiledFn enc = encode_fn();
    if (enc == nullptr) return BDSA_CUDA_ERROR;
    const int G = a.Hq / a.Hkv;
    // Row tiles (TREE with more than M rows): npt nodes a tile
    const int npt = G * a.B <= M ? a.B : M / G;
    const int n_rt = (a.B + npt - 1) / npt;
    if (n_rt > 1 && (long)a.bs * a.Hkv * n_rt > INT32_MAX) return BDSA_UNSUPPORTED;
    CUtensorMap tq, tk, tv;
    {
        // q[(token*Hq + h*G + g)*D + d] as a 4-D tensor (d, g, h, token); a box
        // is one row tile of one KV head
        cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)G, (cuuint64_t)a.Hkv,
                              (cuuint64_t)a.bs * a.B};
        cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)G * D * 2,
                                 (cuuint64_t)a.Hq * D * 2};
        cuuint32_t box[4] = {64, (cuuint32_t)G, 1, (cuuint32_t)npt};
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
    CUtensorMap tout, tpart;
    {
        // out has q's layout; the epilogue stores a whole unit's rows per box
        // (the 64-row tile, whose unit is one row tile: npt = B).
        cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)G, (cuuint64_t)a.Hkv,
                              (cuuint64_t)a.bs * a.B};
        cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)G * D * 2,
                                 (cuuint64_t)a.Hq * D * 2};
        cuuint32_t box[4] = {64, (cuuint32_t)G, 1, (cuuint32_t)npt};
        cuuint32_t es[4] = {1, 1, 1, 1};
        if (enc(&tout, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, a.out, dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
            CUDA_SUCCESS)
            return BDSA_CUDA_ERROR;
    }
    {
        // partial slots [2 * grid * rows, D] fp32, stored 32 columns x rows per box.
        cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)2 * plan.grid * plan.rows};
        cuuint64_t strides[1] = {(cuuint64_t)D * 4};
        cuuint32_t box[2] = {32, (cuuint32_t)plan.rows};
        cuuint32_t es[2] = {1, 1};
        if (enc(&tpart, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, ws + plan.off_part_o, dims, strides,
                box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
            CUDA_SUCCESS)
            return BDSA_CUDA_ERROR;
    }
    Params prm;
    prm.block_table = a.block_table;
    prm.seq_lens = a.seq_lens;
    prm.part_bad = reinterpret_cast<int32_t *>(ws + plan.off_part_bad);
    prm.part_ready = reinterpret_cast<uint64_t *>(ws + plan.off_part_ready);
    prm.ticket = next_ticket();
    prm.owner_ticket = expire_owner_waits() ? (~prm.ticket | 1ull) : prm.ticket;
    // A CUDA graph would replay this call's ticket, so while the stream is
    // being captured the merge waits for the whole attention grid instead.
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) return BDSA_CUDA_ERROR;
    prm.early_merge = M == 128 && cap == cudaStreamCaptureStatusNone;
    // The owner of each cut unit merges it inside the attention launch.  Its
    // wait needs every CTA of the grid resident at once, so only a grid of at
    // most one CTA per SM takes this path; a larger one (a caller's num_sms
    // above the device's) keeps the separate merge launch, and so do TREE
    // calls with the 128-row tile: against the merge launch the owner merge
    // took the Qwen3-8B-shaped verify call 66.2 -> 63.6 us (64-row tile), the
    // LLaDA2.0-style draft 121.4 -> 109.1 us and long-context verify 338.6 ->
    // 330.8 us (128-row tile), but 481-node trees 1052 -> 1110 us.
    prm.owner_merge = plan.grid <= device_num_sms(0) && (M == 64 || a.mode != BDSA_MODE_TREE);
    prm.out = a.out;
    prm.out_v8 = (reinterpret_cast<uintptr_t>(a.out) & 31) == 0;
    prm.lse = a.lse;
    prm.tree_mask = a.tree_mask;
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
    prm.rows = G * npt;
    prm.npt = npt;
    prm.n_rt = n_rt;
    prm.bs_v = n_rt == 1 ? a.bs : a.bs * a.Hkv * n_rt;
    prm.hu = n_rt == 1 ? a.Hkv : 1;
    prm.mask_words = (a.B + 63) / 64;
    prm.page_size = a.page_size;
    int lg = 0;
    while ((1 << lg) < a.page_size) ++lg;
    prm.log2_ps = lg;
    prm.box_rows = box_rows;
    prm.mode = a.mode;
    prm.scale_log2 = a.scale * 1.4426950408889634f;
    prm.magic_S = UINT64_MAX / (uint64_t)plan.grid;
    prm.unit_cost = unit_cost_for(M, n_rt > 1 || a.mode == BDSA_MODE_TREE);
    AppendParams app;
    app.k_new = a.k_new;
    app.v_new = a.v_new;
    app.k_cache = const_cast<uint16_t *>(a.k_cache);
    app.v_cache = const_cast<uint16_t *>(a.v_cache);
    const bool append = a.k_new != nullptr;
    const bool tree = a.mode == BDSA_MODE_TREE;
    auto kernel = tree ? block_attn_kernel<D, M, false, true>
                       : (append ? block_attn_kernel<D, M, true, false>
                                 : block_attn_kernel<D, M, false, false>);
    const int inst = tree ? 2 : (append ? 1 : 0);
    const int smem = C::kSmem;
    const int threads = append ? C::kThreadsAppend : C::kThreads;
    static bool attr_set[3] = {false, false, false};  // per instantiation
    if (!attr_set[inst]) {
        if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
            cudaSuccess)
            return BDSA_CUDA_ERROR;
        attr_set[inst] = true;
    }
    if (launch_pdl(kernel, dim3(plan.grid), dim3(threads), (size_t)smem, stream, tq, tk, tv, tout,
                   tpart, prm, app) != cudaSuccess)
        return BDSA_CUDA_ERROR;
    if (prm.owner_merge) return BDSA_OK;
    if (launch_pdl(tree ? attn_merge_kernel<D, true> : attn_merge_kernel<D, false>,
                   dim3(plan.grid), dim3(kMergeThreads), 0, stream,
                   prm) != cudaSuccess)
        return BDSA_CUDA_ERROR;
    return BDSA_OK;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

AttnPlan attn_plan(int bs, int B, int Hq, int Hkv, int D, int max_ctx_len, int num_sms) {
    (void)max_ctx_len;
    AttnPlan p;
    p.grid = num_sms > 0 ? num_sms : 1;
    // rows a unit: G * B, or one 128-row tile of whole nodes when more (TREE)
    const int G = Hq / Hkv;
    p.rows = G * B <= 128 ? G * B : G * (128 / G);
    size_t off = 0;
    (void)bs;
    p.off_part_bad = off;
    off += align256((size_t)2 * p.grid * sizeof(int32_t));
    p.off_part_ready = off;
    off += align256((size_t)2 * p.grid * sizeof(uint64_t));
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
