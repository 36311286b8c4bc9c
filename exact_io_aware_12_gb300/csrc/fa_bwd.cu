// Backward kernels of exact IO-aware attention for sm_103a.
//
// Method (tonho.wtf "flash attention" entry, section "como funciona",
// backward paragraph; "FlashAttention: O Que E e Como Acelera LLMs na
// Pratica", pillar 2): the backward keeps only O and the per-row statistics
// (packed as LSE), rebuilds S and P on chip, and replaces the softmax
// Jacobian's row sum by D_i = dO_i . O_i.  With dP = dO V^T and
// dS = P o (dP - D):  dV = P^T dO,  dK = tau dS^T Q,  dQ = tau dS K.
//
// Three kernels:
//   bwd_pre   D_i = sum_k dO_ik O_ik (fp32) and a zeroed fp32 dQ accumulator.
//   bwd_main  one CTA per (128-key tile, batch*head); it walks the query tiles
//             that can see its keys (all of them, or those at or below the
//             diagonal when causal):
//               S^T  = K Q_i^T            tcgen05, both operands in smem
//               dP^T = V dO_i^T           tcgen05
//               P^T  = exp2(c S^T - log2e LSE_i)   elementwise warps, written
//                                         back to tensor memory as bf16 over S^T
//               dV  += P^T dO_i           tcgen05, A read from tensor memory
//               dS^T = P^T o (dP^T - D_i) elementwise warps, to smem (and at
//                                         d = 128 to tensor memory beside P^T)
//               dQ_i = dS K               tcgen05, A = dS^T from smem (MN-major)
//               dK  += dS^T Q_i           tcgen05, A from tensor memory (d = 128)
//                                         or the smem tile (d = 64)
//             the elementwise warps (NWG warpgroups: four at d = 128, two at
//             d = 64, each a share of the query and d columns) also read dQ_i out of
//             tensor memory into fp32 smem tiles that the reducer warp adds
//             into the accumulator with TMA bulk reductions (no per-element
//             atomics); at the end they write dK (scaled by tau) and dV.  The
//             loader warp issues the TMA copies, the MMA warp the MMAs.
//             Short d = 64 problems without a mask run it persistently: one CTA
//             per SM walks a list of (key tile, batch*head) items, with the next
//             item's K/V in a second buffer and its first S^T / dP^T issued while
//             the elementwise warps write the current item's dK and dV.
//   bwd_post  dQ = bf16(tau * accumulator).
// Tensor memory (512 columns): dV and dK accumulators (d each), S^T (128),
// dP^T (128).  P^T (bf16, two per column) is written over the first half of
// each warpgroup's S^T columns, and at d = 128 dS^T over the second half, so
// the dV (and at d = 128 the dK) MMA reads its A operand from tensor memory;
// the next S^T goes out right after dK.  For d = 128 the dQ tile reuses the
// dP^T columns once dS^T has been formed, so the next dP^T waits until dQ has
// been read out.  For d = 64, dQ has 64 columns of its own.
#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>
#include <type_traits>

#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int kBQ = 128;  // query rows per step
constexpr int kBK = 128;  // keys per CTA
// NWG elementwise warpgroups (warps 0 .. 4 NWG - 1), then the loader, MMA and
// reducer warps.
constexpr int bwd_threads(int nwg) { return 32 * (4 * nwg + 3); }
constexpr float kLog2e = 1.44269504088896341f;
// Which query tiles a key tile visits beyond causality.
enum : int { kMaskNone = 0, kMaskWindow = 1, kMaskBlocks = 2 };
constexpr int kMaskWords = kMaxMaskBlocks / 32;
constexpr int kBwdPersistMaxN = 2048;  // d = 64, no mask, up to this length: the persistent kernel

// Block-mask backward: a key tile visited by many query tiles (the global anchors of
// a local + global mask are visited by every one) sets the kernel's length alone
// when the rest of the work is short, so its query list is split into chunks that
// extra CTAs run.  A plan kernel picks the chunks from the mask; each chunk adds
// its dQ into the accumulator as usual and writes its partial dK, dV (fp32) to a
// slot, and the last chunk of a tile to finish adds the slots in chunk order (a
// fixed order: the result does not depend on which chunk finishes last) and writes
// dK, dV.  The plan and the slots live in the dQ output, which only the dQ
// conversion kernel writes, afterwards.  Only problems of at most kSplitTilesPerSm
// key tiles per SM are planned: measured on GB300 (16 heads of 16k tokens, a local
// + global mask), with more tiles the busiest SM ran within 4% of the mean without
// a split, and a split that runs the anchors' later query tiles early lost L2 reuse
// (16% slower), while the plan itself costs about 15 us.
constexpr int kSplitTilesPerSm = 2;
constexpr int kSplitMaxChunks = 8;
constexpr int kSplitMinSteps = 16;     // a chunk of fewer query tiles is not worth a CTA
constexpr int kSplitCtaSteps = 2;      // a CTA's set-up and epilogue cost about two steps
constexpr int kPlanThreads = 1024;
// The plan's arrays in its buffer (byte offsets, each 256-aligned): the number of
// helper chunks in use (u32); per key tile in launch order kt * BH + bh its chunk
// count (u8, 1: not split), first partial slot (u32) and finished chunks (u32);
// per helper CTA its (key tile, chunk) (2 x u32); then the partial slots, each
// [dV, dK][D / 4][128 keys][4] fp32 (a warp's 32 key rows of four columns are
// contiguous).
struct SplitPlan {
    size_t hdr, nchunk, slot, help, arrive, part;
};
__host__ __device__ __forceinline__ SplitPlan split_layout(int n_tiles, int n_help) {
    const auto up = [](size_t x) { return (x + 255) / 256 * 256; };
    SplitPlan s;
    s.hdr = 0;
    s.nchunk = 256;
    s.slot = s.nchunk + up(static_cast<size_t>(n_tiles));
    s.help = s.slot + up(4 * static_cast<size_t>(n_tiles));
    s.arrive = s.help + up(8 * static_cast<size_t>(n_help));
    s.part = s.arrive + up(4 * static_cast<size_t>(n_tiles));
    return s;
}

template <int D>
struct BwdLayout {
    static constexpr int kTile = kBK * D * 2;  // one bf16 [128 x D] tile
    static constexpr int kBox = 128 * 128;     // [128 rows x 64 bf16] or [128 x 32 fp32]
    static constexpr int kBoxes = D / 64;
    static constexpr int kK = 0;
    static constexpr int kV = kTile;
    static constexpr int kStage0 = 2 * kTile;    // stage s: Q at +0, dO at +kTile
    static constexpr int kStageBytes = 2 * kTile;
    static constexpr int kDS = kStage0 + 2 * kStageBytes;  // dS^T [128 keys x 128 queries] bf16
    static constexpr int kDSBytes = 128 * 128 * 2;
    static constexpr int kVec = kDS + kDSBytes;  // lse2[2][128], dvec[2][128]
    static constexpr int kBars = kVec + 4 * 128 * 4;
    static constexpr int kBytes = kBars + 512;
    // tensor-memory columns
    static constexpr uint32_t kTmDV = 0, kTmDK = D, kTmS = 2 * D, kTmDP = 2 * D + 128;
    static constexpr bool kDQAliasDP = (D == 128);
    // dK's A operand: dS^T from tensor memory (beside P^T) at d = 128, where it
    // saves the shared-memory reads of an SS MMA; from the smem dS^T tile at
    // d = 64, where the extra tensor-memory store costs the elementwise phase
    // more than it saves
    static constexpr bool kDSInTmem = (D == 128);
    static constexpr uint32_t kTmDQ = kDQAliasDP ? kTmDP : 2 * D + 256;
    // persistent kernel: a second K/V buffer (K at +0, V at +kTile), so the next
    // work item's tiles load during this one, and a dV/dK staging area of its own
    static constexpr int kKV1 = (kBytes + 1023) / 1024 * 1024;
    static constexpr int kStageKV = kKV1 + 2 * kTile;
    static constexpr int kBytesPersist = kStageKV + 2 * kTile;
};

struct BwdBarriers {
    uint64_t kv_full[2];   // K/V buffer b loaded (one buffer unless persistent)
    uint64_t kv_empty[2];  // persistent: the MMAs of the item in K/V buffer b are done
    uint64_t q_full[2];    // Q tile (and the LSE / D vectors) of stage s loaded
    uint64_t do_full[2];   // dO tile of stage s loaded
    uint64_t q_empty[2];   // stage s's Q half free: MMAs done, staged dQ half read
    uint64_t do_empty[2];  // stage s's dO half free: MMAs done, staged dQ half read
    uint64_t s_full;
    uint64_t dp_full;
    uint64_t p_ready;
    uint64_t ds_ready;
    uint64_t dq_full;
    uint64_t dq_drained;
    uint64_t dq_staged_q;   // the warpgroups of dQ columns [0, D/2) staged them (over Q)
    uint64_t dq_staged_do;  // the warpgroups of dQ columns [D/2, D) staged them (over dO)
    uint64_t dk_done;
    uint32_t tmem_base;
    int abort_flag;
    int last_chunk;              // split key tile: this CTA's chunk finished last
    int sp_tile, sp_chunk, sp_nchunk;  // split plan: key tile, chunk, chunks (1: not split)
    uint32_t qbits[kMaskWords];  // kMaskBlocks: bit i = this key tile is visited by query tile i
};

struct BwdParams {
    const float* LSE;
    const float* Dvec;
    int N;
    int n_kv;
    int window;        // causal sliding window in keys (0 = none)
    float scale_log2;  // tau * log2(e)
    float tau;
    unsigned int* err;
    unsigned long long wait_limit_ns;
    const uint8_t* blocks;          // block mask [heads][n_kv][n_kv] (kMaskBlocks)
    long long blocks_head_stride;   // bytes between heads' masks (0: one mask)
    int head_group;                 // heads whose key tiles are interleaved in launch order
    int BH;                         // persistent: batch*heads
    int items;                      // persistent: work items (BH key tiles each)
    uint8_t* plan;                  // block mask: the split plan's buffer (layout: split_layout)
    int plan_tiles;                 // its key tiles (BH * n_kv), 0: no plan
    int plan_help;                  // its helper CTAs, launched first
};

enum : uint32_t {
    kSiteProd = 21, kSiteMmaKV = 22, kSiteMmaQ = 23, kSiteMmaP = 24, kSiteMmaDS = 25,
    kSiteMmaDrain = 26, kSiteDsS = 27, kSiteDsQ = 28, kSiteDsDP = 29, kSiteDsDQ = 30,
    kSiteDrain = 31, kSiteReduce = 32
};

__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }

constexpr uint32_t kDescHi = sw128_desc_hi(1024);  // every operand tile: 8-row groups 1 KB apart
constexpr uint32_t kLboMN = 128 * 128;               // MN-major: next 64-element column chunk

// D = A B^T, both K-major tiles of 128 rows x Dk (two 64-column boxes when Dk = 128).
// a_lo / b_lo: low descriptor halves (K-major) of the tiles.
template <int Dk>
__device__ __forceinline__ void mma_rows_rows(uint32_t tmem_d, uint32_t a_lo, uint32_t b_lo) {
    constexpr uint32_t id = idesc_bf16(128, 128, false, false);
#pragma unroll
    for (int k = 0; k < Dk / 16; ++k) {
        const uint32_t off = ((k / 4) * (128 * 128) + (k % 4) * 32) >> 4;
        if (k == 0) mma_ss_warp<0>(tmem_d, a_lo + off, b_lo + off, kDescHi, id);
        else mma_ss_warp<1>(tmem_d, a_lo + off, b_lo + off, kDescHi, id);
    }
}

// D (+)= A_tmem[128 x 128] B, B an MN-major smem tile [128 rows(K) x N] (N = Dn).
// A (bf16, packed two per column): each warpgroup owns QC consecutive K-columns
// (queries) and writes them packed over the first QC/2 of its QC fp32 columns,
// so K-columns [g QC, (g + 1) QC) sit at tensor-memory columns [g QC, g QC + QC/2).
template <int Dn, int QC>
__device__ __forceinline__ void mma_tmem_a(uint32_t tmem_d, uint32_t tmem_a, uint32_t b_lo,
                                           bool accumulate) {
    constexpr uint32_t id = idesc_bf16(128, Dn, false, true);
    if (accumulate) mma_ts_warp<1>(tmem_d, tmem_a, b_lo, kDescHi, id);
    else mma_ts_warp<0>(tmem_d, tmem_a, b_lo, kDescHi, id);
#pragma unroll
    for (int k = 1; k < 128 / 16; ++k)
        mma_ts_warp<1>(tmem_d, tmem_a + (16 * k / QC) * QC + (16 * k % QC) / 2,
                       b_lo + ((k * 2048) >> 4), kDescHi, id);
}

// D (+)= A B with A a K-major smem tile [128 rows(M) x 128(K)] (two 64-column
// boxes) and B an MN-major smem tile [128 rows(K) x Dn].
template <int Dn>
__device__ __forceinline__ void mma_rows_mn(uint32_t tmem_d, uint32_t a_lo, uint32_t b_lo,
                                            bool accumulate) {
    constexpr uint32_t id = idesc_bf16(128, Dn, false, true);
    if (accumulate) mma_ss_warp<1>(tmem_d, a_lo, b_lo, kDescHi, id);
    else mma_ss_warp<0>(tmem_d, a_lo, b_lo, kDescHi, id);
#pragma unroll
    for (int k = 1; k < 128 / 16; ++k)
        mma_ss_warp<1>(tmem_d, a_lo + (((k / 4) * (128 * 128) + (k % 4) * 32) >> 4),
                       b_lo + ((k * 2048) >> 4), kDescHi, id);
}

// D = A B with A MN-major [128(K) x 128(M)] and B MN-major [128(K) x Dn].
template <int Dn>
__device__ __forceinline__ void mma_mn_mn(uint32_t tmem_d, uint32_t a_lo, uint32_t b_lo) {
    constexpr uint32_t id = idesc_bf16(128, Dn, true, true);
    mma_ss_warp<0>(tmem_d, a_lo, b_lo, kDescHi, id);
#pragma unroll
    for (int k = 1; k < 128 / 16; ++k)
        mma_ss_warp<1>(tmem_d, a_lo + ((k * 2048) >> 4), b_lo + ((k * 2048) >> 4), kDescHi, id);
}

// MASK: kMaskNone; kMaskWindow, a causal sliding window of p.window keys (only
// with CAUSAL); kMaskBlocks, the block mask p.blocks.  PERSIST: one CTA per SM
// walks a list of (key tile, batch*head) work items (no mask).
template <int D, bool CAUSAL, int MASK, int NWG, bool PERSIST = false, bool SPLIT = false>
__global__ void __launch_bounds__(bwd_threads(NWG), 1)
fa_bwd_main_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                   const __grid_constant__ CUtensorMap tmdQacc,
                   const __grid_constant__ CUtensorMap tmdK, const __grid_constant__ CUtensorMap tmdV,
                   const BwdParams p) {
    using L = BwdLayout<D>;
    static_assert(sizeof(BwdBarriers) <= L::kBytes - L::kBars, "barrier block overflows its slot");
    static_assert(NWG == 2 || NWG == 4, "two or four elementwise warpgroups");
    static_assert((D / NWG) % 16 == 0, "each warpgroup drains whole 16-column chunks");
    static_assert(!PERSIST || MASK == kMaskNone, "the persistent kernel takes no mask");
    constexpr int kProducerWarp = 4 * NWG, kMmaWarp = 4 * NWG + 1, kReducerWarp = 4 * NWG + 2;
    constexpr int kQC = 128 / NWG;      // query columns of P^T / dS^T per warpgroup
    constexpr int kDC = D / NWG;        // d-columns of dQ, dK, dV per warpgroup
    constexpr int kEW = 128 * NWG;      // elementwise threads
    constexpr bool LOCAL = MASK == kMaskWindow;
    constexpr bool SPARSE = MASK == kMaskBlocks;
    // a block mask with a split plan (its own instance: the plan's code stays out of
    // the plain block-mask kernel)
    constexpr bool SPLIT_ = SPARSE && SPLIT;
    static_assert(!SPLIT || SPARSE, "a split plan needs a block mask");
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t sbase = smem_addr(smem);
    BwdBarriers& sh = *reinterpret_cast<BwdBarriers*>(smem + L::kBars);
    float* lse2_s = reinterpret_cast<float*>(smem + L::kVec);        // [2][128]
    float* dvec_s = reinterpret_cast<float*>(smem + L::kVec + 1024);  // [2][128]

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // Block mask with a split plan: this CTA's key tile (launch order kt * BH + bh)
    // and its chunk of the tile's query list.  The first n_help CTAs are helpers,
    // each running one chunk > 0 of a split tile, or nothing; launched first, the
    // long tiles' chunks start before the short tiles fill the machine.  The plan
    // is written by the plan kernel, launched just before: a helper waits for it
    // here, a key tile's own CTA reads its chunk count later, beside its mask loads.
    int sp_tile = -1, sp_chunk = 0;
    if constexpr (SPLIT_) {
        const int e = static_cast<int>(blockIdx.x);
        if (e < p.plan_help) {
            griddep_wait();
            const SplitPlan pl = split_layout(p.plan_tiles, p.plan_help);
            if (e >= static_cast<int>(*reinterpret_cast<const uint32_t*>(p.plan + pl.hdr))) return;
            const uint32_t* help = reinterpret_cast<const uint32_t*>(p.plan + pl.help);
            sp_tile = static_cast<int>(help[2 * e]);
            sp_chunk = static_cast<int>(help[2 * e + 1]);
        } else {
            sp_tile = e - p.plan_help;
        }
    }
    // Work item k of this CTA: (batch*head, key tile), or false past the last.
    // Without PERSIST a CTA has one item, set by its launch position: the launch
    // order (x fastest) walks groups of p.head_group heads; inside a group the key
    // tiles go in order (tile 0 has the most query tiles when causal), the group's
    // heads interleaved.  So the CTAs resident at one time work on a few heads,
    // whose Q, dO and fp32 dQ accumulator stay in L2.  With PERSIST, CTA c of G
    // takes items c, 2G - 1 - c, 2G + c, ... of the list ordered by key tile, then
    // head (heaviest first when causal): a snake that balances heavy and light
    // items without a shared counter.  (The head-grouped order measured slower
    // here: at these sizes the balance matters more than the L2 reuse.)
    auto item_at = [&](int k, int& ibh, int& ikv) -> bool {
        if constexpr (PERSIST) {
            const int G = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
            const long long i = static_cast<long long>(k) * G + ((k & 1) ? G - 1 - c : c);
            if (i >= p.items) return false;
            ikv = static_cast<int>(i / p.BH);
            ibh = static_cast<int>(i - static_cast<long long>(ikv) * p.BH);
            return true;
        }
        if (k > 0) return false;
        if (SPLIT_) {
            ikv = sp_tile / p.BH;
            ibh = sp_tile - ikv * p.BH;
            return true;
        }
        const long long i = blockIdx.x + static_cast<long long>(gridDim.x) * blockIdx.y;
        const long long per_group = static_cast<long long>(p.head_group) * p.n_kv;
        const int g = static_cast<int>(i / per_group);
        const int j = static_cast<int>(i - g * per_group);
        const int heads = min(p.head_group, p.BH - g * p.head_group);
        ikv = j / heads;
        ibh = g * p.head_group + (j - ikv * heads);
        return true;
    };
    int bh = 0, kv_tile = 0;  // item 0 (every CTA has one)
    item_at(0, bh, kv_tile);
    const int N = p.N;
    const int kv_start = kv_tile * kBK;
    const int n_q = (N + kBQ - 1) / kBQ;
    // Query tiles that see this key tile: from the diagonal when causal, and with
    // a sliding window only up to the tile holding query (last key + window - 1).
    const int window = (CAUSAL && LOCAL) ? p.window : 0;
    const int first = CAUSAL ? kv_tile : 0;
    const int last = window > 0 ? min(n_q - 1, (kv_start + kBK - 1 + window - 1) / kBQ) : n_q - 1;
    int n_steps = last - first + 1;  // with a block mask: counted below
    // an item's first query tile and step count (item 0: first and n_steps)
    auto first_of = [&](int ikv) { return PERSIST ? (CAUSAL ? ikv : 0) : first; };
    auto steps_of = [&](int ikv) { return PERSIST ? n_q - (CAUSAL ? ikv : 0) : n_steps; };

    if (sbase & 1023u) {  // the swizzled tiles need 1024-byte alignment
        if (threadIdx.x == 0) atomicCAS(p.err, 0u, 1u | (0xAAu << 8));
        return;
    }

    const uint32_t bar_kv = smem_addr(&sh.kv_full[0]);
    const uint32_t bar_kve = smem_addr(&sh.kv_empty[0]);
    const uint32_t bar_qf = smem_addr(&sh.q_full[0]);
    const uint32_t bar_df = smem_addr(&sh.do_full[0]);
    const uint32_t bar_qe = smem_addr(&sh.q_empty[0]);
    const uint32_t bar_de = smem_addr(&sh.do_empty[0]);
    const uint32_t bar_s = smem_addr(&sh.s_full);
    const uint32_t bar_dp = smem_addr(&sh.dp_full);
    const uint32_t bar_p = smem_addr(&sh.p_ready);
    const uint32_t bar_ds = smem_addr(&sh.ds_ready);
    const uint32_t bar_dq = smem_addr(&sh.dq_full);
    const uint32_t bar_dr = smem_addr(&sh.dq_drained);
    const uint32_t bar_sgq = smem_addr(&sh.dq_staged_q);
    const uint32_t bar_sgd = smem_addr(&sh.dq_staged_do);
    const uint32_t bar_dk = smem_addr(&sh.dk_done);

    if (threadIdx.x == 0) {
        sh.abort_flag = 0;
        if constexpr (SPLIT_) {
            sh.sp_tile = sp_tile;
            sh.sp_chunk = sp_chunk;
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar_kv + 8 * b, 1);
            mbar_init(bar_kve + 8 * b, 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar_qf + 8 * s, 32);
            mbar_init(bar_df + 8 * s, 1);
            mbar_init(bar_qe + 8 * s, 2);  // MMA commit + the reducer warp
            mbar_init(bar_de + 8 * s, 2);
        }
        mbar_init(bar_s, 1);
        mbar_init(bar_dp, 1);
        mbar_init(bar_p, kEW);
        mbar_init(bar_ds, kEW);
        mbar_init(bar_dq, 1);
        mbar_init(bar_dr, kEW);
        mbar_init(bar_sgq, kEW / 2);
        mbar_init(bar_sgd, kEW / 2);
        mbar_init(bar_dk, 1);
        mbar_init_fence();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_addr(&sh.tmem_base), 512);
        tmem_relinquish();
    }
    if (warp == kProducerWarp && lane == 0) {
        tma_prefetch_map(&tmQ);
        tma_prefetch_map(&tmK);
        tma_prefetch_map(&tmV);
        tma_prefetch_map(&tmdO);
        tma_prefetch_map(&tmdQacc);
    }
    if constexpr (SPARSE) {
        if (warp == kProducerWarp) {
            // bit i of qbits: query tile i's mask row has this key block set (and
            // i is at or below the diagonal when causal); one ballot per 32 tiles
            const uint8_t* m = p.blocks + bh * p.blocks_head_stride;
            int nch = 1;  // a split plan: this key tile's chunks (its load overlaps the mask loads)
            if constexpr (SPLIT_) {
                griddep_wait();
                nch = p.plan[split_layout(p.plan_tiles, p.plan_help).nchunk + sp_tile];
            }
            for (int w = 0; w * 32 < n_q; ++w) {
                const int i = w * 32 + lane;
                bool u = false;
                if (i < n_q && (!CAUSAL || i >= kv_tile))
                    u = m[static_cast<long long>(i) * p.n_kv + kv_tile] != 0;
                const uint32_t bits = __ballot_sync(0xffffffffu, u);
                if (lane == 0) sh.qbits[w] = bits;
            }
            if (SPLIT_ && lane == 0) sh.sp_nchunk = nch;
            // a split tile: keep the chunk's share of the list, the set bits with index
            // in [chunk c / n, (chunk + 1) c / n)
            if (nch > 1 && lane == 0) {
                int c = 0;
                for (int w = 0; w * 32 < n_q; ++w) c += __popc(sh.qbits[w]);
                const int lo = sp_chunk * c / nch, hi = (sp_chunk + 1) * c / nch;
                int seen = 0;
                for (int w = 0; w * 32 < n_q; ++w) {
                    uint32_t bits = sh.qbits[w], keep = 0u;
                    while (bits) {
                        const uint32_t bit = bits & (0u - bits);
                        if (seen >= lo && seen < hi) keep |= bit;
                        ++seen;
                        bits ^= bit;
                    }
                    sh.qbits[w] = keep;
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    griddep_launch_dependents();  // the dQ conversion kernel may be scheduled
    const uint32_t tmem = sh.tmem_base;
    const Watchdog wd{p.err, &sh.abort_flag, p.wait_limit_ns};
    constexpr uint32_t FULL = 0xffffffffu;
    if constexpr (SPARSE) {
        int c = 0;
        for (int w = 0; w * 32 < n_q; ++w) c += __popc(sh.qbits[w]);
        n_steps = c;
    }

    if (warp == kProducerWarp) {
        // ------------------------------------------------------- producer --
        // Steps are numbered across work items (gs): the Q/dO stage and the
        // barrier phases follow gs, the K/V buffer follows the item.
        bool pok = true;
        int gs = 0;
        int ibh = 0, ikv = 0;
        for (int k = 0; pok && item_at(k, ibh, ikv); ++k) {
            const int kb = PERSIST ? (k & 1) : 0;
            const int ifirst = first_of(ikv), isteps = steps_of(ikv);
            // the buffer's previous item (k - 2) must be done with it
            if (PERSIST && k >= 2 && !mbar_wait(bar_kve + 8 * kb, ((k >> 1) - 1) & 1, wd, kSiteProd)) break;
            // a key tile that no query tile visits (block mask) loads nothing: its
            // epilogue writes zero dK, dV over the K and V tiles
            if (lane == 0 && (!SPARSE || isteps > 0)) {
                const uint32_t kv_buf = sbase + (kb ? L::kKV1 : L::kK);
                mbar_arrive_expect_tx(bar_kv + 8 * kb, 2 * L::kTile);
                for (int b = 0; b < L::kBoxes; ++b) {
                    tma_load_3d(kv_buf + b * L::kBox, &tmK, bar_kv + 8 * kb, b * 64, ikv * kBK, ibh);
                    tma_load_3d(kv_buf + L::kTile + b * L::kBox, &tmV, bar_kv + 8 * kb, b * 64, ikv * kBK,
                                ibh);
                }
            }
            // LSE comes from the forward and D from the D kernel launched just before
            // this one, which may still be running (dependent launch): wait for it
            if (k == 0) griddep_wait();
            int qsp = -1;  // block mask: the query tile of the last step
            for (int s = 0; s < isteps; ++s, ++gs) {
                if constexpr (!PERSIST) gs = s;  // one item: the two counts agree
                const int st = gs & 1;
                int qtile = ifirst + s;
                if constexpr (SPARSE) {
                    qsp = next_set_bit(sh.qbits, nullptr, qsp + 1, n_q);
                    qtile = qsp;
                }
                const int q_start = qtile * kBQ;
                const int64_t row0 = static_cast<int64_t>(ibh) * N;
                // this step's LSE and D into registers first: their latency overlaps
                // the wait for the stage (stored negated: the softmax warps add them
                // with paired fp32 ops)
                float lv[4], dv[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int q = q_start + lane * 4 + e;
                    lv[e] = q < N ? -p.LSE[row0 + q] * kLog2e : -INFINITY;
                    dv[e] = q < N ? -p.Dvec[row0 + q] : 0.f;
                }
                // the two halves of the stage are refilled as each is freed: dO (whose
                // staged dQ half is added first), then Q with the vectors
                const uint32_t stage = sbase + L::kStage0 + st * L::kStageBytes;
                if (gs >= 2 && !mbar_wait(bar_de + 8 * st, ((gs >> 1) - 1) & 1, wd, kSiteProd)) {
                    pok = false;
                    break;
                }
                if (lane == 0) {
                    mbar_arrive_expect_tx(bar_df + 8 * st, L::kTile);
                    for (int b = 0; b < L::kBoxes; ++b)
                        tma_load_3d(stage + L::kTile + b * L::kBox, &tmdO, bar_df + 8 * st, b * 64,
                                    q_start, ibh);
                }
                if (gs >= 2 && !mbar_wait(bar_qe + 8 * st, ((gs >> 1) - 1) & 1, wd, kSiteProd)) {
                    pok = false;
                    break;
                }
                if (lane == 0) {  // the bulk copy first, then the vectors
                    mbar_expect_tx(bar_qf + 8 * st, L::kTile);
                    for (int b = 0; b < L::kBoxes; ++b)
                        tma_load_3d(stage + b * L::kBox, &tmQ, bar_qf + 8 * st, b * 64, q_start, ibh);
                }
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    lse2_s[st * 128 + lane * 4 + e] = lv[e];
                    dvec_s[st * 128 + lane * 4 + e] = dv[e];
                }
                mbar_arrive(bar_qf + 8 * st);  // 32 arrivals; the phase also waits for the copy
            }
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA --
        // The whole warp runs this loop; each MMA and commit is issued by one
        // elected lane (see mma_ss_warp).
        {
            // low descriptor halves: K-major (LBO unused) and MN-major (LBO = 16 KB);
            // K and V per buffer (buffer 1 only in the persistent kernel)
            const uint32_t k_lo0 = sw128_desc_lo(sbase + L::kK, 16), k_lo1 = sw128_desc_lo(sbase + L::kKV1, 16);
            const uint32_t k_mn0 = sw128_desc_lo(sbase + L::kK, kLboMN);
            const uint32_t k_mn1 = sw128_desc_lo(sbase + L::kKV1, kLboMN);
            const uint32_t v_lo0 = sw128_desc_lo(sbase + L::kV, 16);
            const uint32_t v_lo1 = sw128_desc_lo(sbase + L::kKV1 + L::kTile, 16);
            const uint32_t ds_mn = sw128_desc_lo(sbase + L::kDS, kLboMN);
            const uint32_t ds_lo = sw128_desc_lo(sbase + L::kDS, 16);
            const uint32_t q_lo0 = sw128_desc_lo(sbase + L::kStage0, 16);
            const uint32_t q_mn0 = sw128_desc_lo(sbase + L::kStage0, kLboMN);
            const uint32_t do_lo0 = sw128_desc_lo(sbase + L::kStage0 + L::kTile, 16);
            const uint32_t do_mn0 = sw128_desc_lo(sbase + L::kStage0 + L::kTile, kLboMN);
            constexpr uint32_t kStageStep = L::kStageBytes >> 4;
            bool ok = (!SPARSE || n_steps > 0) &&
                      __all_sync(0xffffffffu, mbar_wait(bar_kv, 0, wd, kSiteMmaKV) &&
                                                  mbar_wait(bar_qf, 0, wd, kSiteMmaQ));
            if (ok) {
                tc_fence_after();
                mma_rows_rows<D>(tmem + L::kTmS, k_lo0, q_lo0);     // S^T
                mma_commit_warp(bar_s);
                ok = __all_sync(0xffffffffu, mbar_wait(bar_df, 0, wd, kSiteMmaQ));
                if (ok) {
                    tc_fence_after();
                    mma_rows_rows<D>(tmem + L::kTmDP, v_lo0, do_lo0);   // dP^T
                    mma_commit_warp(bar_dp);
                }
            }
            int gs = 0;  // steps across work items
            int ibh = 0, ikv = 0;
            for (int k = 0; ok && item_at(k, ibh, ikv); ++k) {
                const int kb = PERSIST ? (k & 1) : 0;
                const int isteps = steps_of(ikv);
                int nbh = 0, nkv = 0;
                const bool has_next = PERSIST && item_at(k + 1, nbh, nkv);
                for (int s = 0; ok && s < isteps; ++s, ++gs) {
                    if constexpr (!PERSIST) gs = s;  // one item: the two counts agree
                    const int st = gs & 1;
                    const uint32_t so = st * kStageStep;
                    if (!__all_sync(0xffffffffu, mbar_wait(bar_p, gs & 1, wd, kSiteMmaP))) { ok = false; break; }
                    tc_fence_after();
                    mma_tmem_a<D, kQC>(tmem + L::kTmDV, tmem + L::kTmS, do_mn0 + so, s > 0);   // dV
                    mma_commit_warp(bar_de + 8 * st);  // the last MMA that reads this dO
                    if (!__all_sync(0xffffffffu, mbar_wait(bar_ds, gs & 1, wd, kSiteMmaDS))) { ok = false; break; }
                    tc_fence_after();
                    // d = 64: the dQ columns are reused every step
                    if (!L::kDQAliasDP && gs > 0) {
                        if (!__all_sync(0xffffffffu, mbar_wait(bar_dr, (gs - 1) & 1, wd, kSiteMmaDrain))) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                    }
                    // dQ first: its drain is on the elementwise warps' path; dK and the
                    // next S^T run while they drain it
                    mma_mn_mn<D>(tmem + L::kTmDQ, ds_mn, kb ? k_mn1 : k_mn0);                        // dQ
                    mma_commit_warp(bar_dq);
                    if constexpr (L::kDSInTmem)
                        mma_tmem_a<D, kQC>(tmem + L::kTmDK, tmem + L::kTmS + kQC / 2, q_mn0 + so, s > 0);  // dK
                    else
                        mma_rows_mn<D>(tmem + L::kTmDK, ds_lo, q_mn0 + so, s > 0);           // dK
                    mma_commit_warp(bar_dk);           // d = 64: also, the dS^T tile is free again
                    mma_commit_warp(bar_qe + 8 * st);
                    const bool last_step = s + 1 == isteps;
                    // the last MMA that reads this item's K and V has been issued
                    if (PERSIST && last_step) mma_commit_warp(bar_kve + 8 * kb);
                    if (!last_step || has_next) {
                        // the next step: this item's, or the next item's first (its K, V
                        // in the other buffer)
                        const int nkb = last_step ? (k + 1) & 1 : kb;
                        if (last_step) {
                            if (!__all_sync(0xffffffffu,
                                            mbar_wait(bar_kv + 8 * nkb, ((k + 1) >> 1) & 1, wd, kSiteMmaKV))) {
                                ok = false;
                                break;
                            }
                        }
                        const int st1 = (gs + 1) & 1;
                        const uint32_t so1 = st1 * kStageStep;
                        if (!__all_sync(0xffffffffu, mbar_wait(bar_qf + 8 * st1, ((gs + 1) >> 1) & 1, wd, kSiteMmaQ))) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        // S^T over P^T and dS^T, which only the dV and dK MMAs above
                        // read (the tensor pipe runs in issue order)
                        mma_rows_rows<D>(tmem + L::kTmS, nkb ? k_lo1 : k_lo0, q_lo0 + so1);     // S^T next
                        mma_commit_warp(bar_s);
                        // d = 128: dP^T over the dQ tile, once it has been read out
                        if (L::kDQAliasDP) {
                            if (!__all_sync(0xffffffffu, mbar_wait(bar_dr, gs & 1, wd, kSiteMmaDrain))) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                        }
                        if (!__all_sync(0xffffffffu, mbar_wait(bar_df + 8 * st1, ((gs + 1) >> 1) & 1, wd, kSiteMmaQ))) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        mma_rows_rows<D>(tmem + L::kTmDP, nkb ? v_lo1 : v_lo0, do_lo0 + so1);   // dP^T next
                        mma_commit_warp(bar_dp);
                    }
                }
            }
        }
        __syncwarp();
    } else if (warp == kReducerWarp) {
        // ---------------------------------------------------------- reducer --
        // Adds each step's staged fp32 dQ tiles into the accumulator (TMA bulk
        // reduce-add) and, once the reads are done, hands the stage back to the
        // producer; waiting here keeps that wait off the softmax warps' path.
        if (lane == 0) {
            griddep_wait();  // the accumulator is zeroed by the D kernel
            bool ok = true;
            int gs = 0;  // steps across work items
            int ibh = 0, ikv = 0;
            for (int k = 0; item_at(k, ibh, ikv); ++k) {
                const int ifirst = first_of(ikv), isteps = steps_of(ikv);
                int qsp = -1;  // block mask: the query tile of the last step
                for (int s = 0; s < isteps; ++s, ++gs) {
                    if constexpr (!PERSIST) gs = s;  // one item: the two counts agree
                    const int st = gs & 1;
                    int qtile = ifirst + s;
                    if constexpr (SPARSE) {
                        qsp = next_set_bit(sh.qbits, nullptr, qsp + 1, n_q);
                        qtile = qsp;
                    }
                    const uint32_t src = sbase + L::kStage0 + st * L::kStageBytes;
                    const int q_start = qtile * kBQ;
                    // dQ columns [D/2, D) were staged over dO (first), [0, D/2) over Q
                    // (once dK is done)
                    if (ok) ok = mbar_wait(bar_sgd, gs & 1, wd, kSiteReduce);
                    if (ok) {
                        for (int b = D / 64; b < D / 32; ++b)
                            tma_reduce_add_3d(&tmdQacc, src + b * L::kBox, b * 32, q_start, ibh);
                        bulk_commit();
                    }
                    if (ok) ok = mbar_wait(bar_sgq, gs & 1, wd, kSiteReduce);
                    if (ok) {
                        for (int b = 0; b < D / 64; ++b)
                            tma_reduce_add_3d(&tmdQacc, src + b * L::kBox, b * 32, q_start, ibh);
                        bulk_commit();
                        bulk_wait_read<1>();
                    }
                    mbar_arrive(bar_de + 8 * st);
                    if (ok) bulk_wait_read<0>();
                    mbar_arrive(bar_qe + 8 * st);
                }
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------- elementwise warpgroups 0 .. NWG-1 --
        // Warpgroup h owns query columns [kQC h, kQC (h + 1)) of P^T and dS^T, and
        // d-columns [kDC h, kDC (h + 1)) of the dQ drain and the dK/dV epilogue.
        // A failed wait poisons the rest of the work (ok = false) but every
        // thread still reaches every named barrier, so none can be left waiting.
        const int h = warp >> 2;
        const int r = threadIdx.x & 127;  // key row (P^T, dS^T, dK, dV) / query row (dQ)
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + lane_off + L::kTmS + kQC * h;
        const uint32_t tDP = tmem + lane_off + L::kTmDP + kQC * h;
        const uint32_t tDQ = tmem + lane_off + L::kTmDQ + kDC * h;
        const float sl2 = p.scale_log2;
        // this row of the dS^T tile: the box (64 query columns) holding this warpgroup's
        // columns, and their first 16-byte chunk in it
        uint8_t* ds_row = smem + L::kDS + (kQC * h / 64) * (128 * 128) + r * 128;
        const int ds_chunk0 = (kQC * h % 64) / 8;
        constexpr int kDrainChunks = kDC / 16;  // 16-column fp32 chunks of dQ per warpgroup
        bool ok = true;
        int gs = 0;  // steps across work items
        int ibh = 0, ikv = 0;
        for (int k = 0; item_at(k, ibh, ikv); ++k) {
            const int ifirst = first_of(ikv), isteps = steps_of(ikv);
            const int kvs = ikv * kBK;
            const int kg = kvs + r;
            int qsp = -1;  // block mask: the query tile of the last step
            for (int s = 0; s < isteps; ++s, ++gs) {
                if constexpr (!PERSIST) gs = s;  // one item: the two counts agree
                const int st = gs & 1;
                int qtile = ifirst + s;
                if constexpr (SPARSE) {
                    qsp = next_set_bit(sh.qbits, nullptr, qsp + 1, n_q);
                    qtile = qsp;
                }
                const int q_start = qtile * kBQ;
                // P^T = exp2(c S^T - log2e LSE), bf16, over this warpgroup's S^T columns.
                // -log2(e) LSE per query, pairs of adjacent queries as one 64-bit value,
                // read four queries per 16-byte broadcast load; the first chunk's are
                // read as soon as the stage (with the vectors) is in, before S^T is
                const ulonglong2* nl4 = reinterpret_cast<const ulonglong2*>(lse2_s + st * 128 + kQC * h);
                ulonglong2 nl0[8];
                uint32_t pkeep[16];  // the first chunk's packed P^T, reused by dS^T below
                if (ok) ok = __all_sync(FULL, mbar_wait_sleep(bar_qf + 8 * st, (gs >> 1) & 1, wd, kSiteDsQ));
                if (ok) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) nl0[i] = nl4[i];
                }
                if (ok) ok = __all_sync(FULL, mbar_wait_sleep(bar_s, gs & 1, wd, kSiteDsS));
                if (ok) {
                    tc_fence_after();
                    const bool diag = CAUSAL && (q_start == kvs);
                    // window edge: query q no longer sees key kg once q >= kg + window
                    const bool wedge = window > 0 && q_start + kBQ - 1 >= kvs + window;
                    const int qh = q_start + kQC * h;
                    const uint64_t c2 = f2_pack(sl2, sl2);
                    // most tiles need no mask: the loop is built twice, and the masked
                    // copy runs only on the diagonal, window-edge and ragged-end tiles
                    const bool masked = diag || wedge || kvs + kBK > N;
                    // this key row's visible query columns q (offsets in the warpgroup's
                    // slice) are lo <= q < hi: above the diagonal q < kg - qh is hidden,
                    // past the window edge q >= kg + window - qh, and a key row past a
                    // ragged end sees none
                    const int lo = kg >= N ? (1 << 30) : (diag ? kg - qh : -(1 << 30));
                    const int hi = (LOCAL && wedge) ? kg + window - qh : (1 << 30);
#pragma unroll
                    for (int c = 0; c < kQC / 32; ++c) {
                        uint32_t sv[32];
                        tmem_ld32(tS + 32 * c, sv);
                        tmem_ld_wait(sv);
                        uint32_t pk[16];
                        ulonglong2 nl[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) nl[i] = c == 0 ? nl0[i] : nl4[8 * c + i];
                        auto p_pairs = [&](auto with_mask) {
#pragma unroll
                            for (int i = 0; i < 16; ++i) {
                                const int q = 32 * c + 2 * i;
                                const uint64_t nlq = (i & 1) ? nl[i >> 1].y : nl[i >> 1].x;
                                const float2 x = f2_unpack(
                                    ffma2(f2_pack(u2f(sv[2 * i]), u2f(sv[2 * i + 1])), c2, nlq));
                                float p0 = ex2(x.x);
                                float p1 = ex2(x.y);
                                if constexpr (decltype(with_mask)::value) {
                                    if (q < lo || q >= hi) p0 = 0.f;
                                    if (q + 1 < lo || q + 1 >= hi) p1 = 0.f;
                                }
                                pk[i] = pack_bf16(p0, p1);
                            }
                        };
                        if (masked) p_pairs(std::true_type{});
                        else p_pairs(std::false_type{});
                        tmem_st16(tS + 16 * c, pk);
                        if (c == 0) {
#pragma unroll
                            for (int i = 0; i < 16; ++i) pkeep[i] = pk[i];
                        }
                    }
                    tmem_st_wait();
                    tc_fence_before();
                }
                mbar_arrive(bar_p);

                // dS^T = P^T o (dP^T - D), to the smem tile that the dQ MMA reads (and at
                // d = 64 the dK MMA), once the MMAs of the previous step are done with
                // it, and at d = 128 also to tensor memory beside P^T (dK's A operand).
                // -D per query, pairs of adjacent queries as one 64-bit value (16-byte
                // loads); the first chunk's are read before the wait for dP^T
                const ulonglong2* nd4 = reinterpret_cast<const ulonglong2*>(dvec_s + st * 128 + kQC * h);
                ulonglong2 nd0[8];
                if (ok) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) nd0[i] = nd4[i];
                }
                if (ok)
                    ok = __all_sync(FULL, mbar_wait_sleep(bar_dp, gs & 1, wd, kSiteDsDP) &&
                                              (gs == 0 || mbar_wait_sleep(L::kDSInTmem ? bar_dq : bar_dk,
                                                                          (gs - 1) & 1, wd, kSiteDsDQ)));
                if (ok) {
                    tc_fence_after();
#pragma unroll
                    for (int c = 0; c < kQC / 32; ++c) {
                        uint32_t dp[32], pk[16];
                        tmem_ld32(tDP + 32 * c, dp);
                        if (c == 0) {
#pragma unroll
                            for (int i = 0; i < 16; ++i) pk[i] = pkeep[i];
                        } else {
                            tmem_ld16(tS + 16 * c, pk);
                            tmem_ld_wait(pk);
                        }
                        tmem_ld_wait(dp);
                        uint32_t ds[16];
                        ulonglong2 nd[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) nd[i] = c == 0 ? nd0[i] : nd4[8 * c + i];
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const uint64_t ndq = (i & 1) ? nd[i >> 1].y : nd[i >> 1].x;
                            // dP - D in fp32, rounded to bf16, times the bf16 P
                            const float2 t = f2_unpack(
                                fadd2(f2_pack(u2f(dp[2 * i]), u2f(dp[2 * i + 1])), ndq));
                            ds[i] = mul_bf16x2(pk[i], pack_bf16(t.x, t.y));
                        }
                        if constexpr (L::kDSInTmem) tmem_st16(tS + kQC / 2 + 16 * c, ds);
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4) {
                            const int chunk = ds_chunk0 + 4 * c + q4;
                            *reinterpret_cast<uint4*>(ds_row + ((chunk ^ (r & 7)) << 4)) =
                                make_uint4(ds[4 * q4], ds[4 * q4 + 1], ds[4 * q4 + 2], ds[4 * q4 + 3]);
                        }
                    }
                    fence_async_shared();
                    if constexpr (L::kDSInTmem) tmem_st_wait();
                    tc_fence_before();
                }
                mbar_arrive(bar_ds);

                // dQ drain: this warpgroup's D/2 columns -> fp32 tiles -> bulk reduce-add
                if (ok) ok = __all_sync(FULL, mbar_wait_sleep(bar_dq, gs & 1, wd, kSiteDrain));
                uint8_t* stage = smem + L::kStage0 + st * L::kStageBytes;
                uint32_t acc[kDrainChunks][16];
                if (ok) {
                    tc_fence_after();
#pragma unroll
                    for (int b = 0; b < kDrainChunks; ++b) tmem_ld16(tDQ + 16 * b, acc[b]);
#pragma unroll
                    for (int b = 0; b < kDrainChunks; ++b) tmem_ld_wait(acc[b]);
                    tc_fence_before();
                    mbar_arrive(bar_dr);
                    // stage fp32 boxes of [128 x 32] over this step's Q (the first half of the
                    // warpgroups, dQ columns [0, D/2)) and dO (the second half): dO is free
                    // (dV, dP^T done before dQ), Q once dK is
                    if (h < NWG / 2) ok = __all_sync(FULL, mbar_wait_sleep(bar_dk, gs & 1, wd, kSiteDrain));
                } else {
                    mbar_arrive(bar_dr);
                }
                if (ok) {
#pragma unroll
                    for (int b = 0; b < kDrainChunks; ++b) {
                        // columns h kDC + 16 b ..: box (32 columns) and first 16-byte chunk in it
                        const int col = h * kDC + 16 * b;
                        uint8_t* box = stage + (col / 32) * L::kBox + r * 128;
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            *reinterpret_cast<uint4*>(box + ((((col % 32) / 4 + j) ^ (r & 7)) << 4)) =
                                make_uint4(acc[b][4 * j], acc[b][4 * j + 1], acc[b][4 * j + 2],
                                           acc[b][4 * j + 3]);
                    }
                    fence_async_shared();
                }
                mbar_arrive(h >= NWG / 2 ? bar_sgd : bar_sgq);  // the reducer adds the staged tiles into dQ
            }
            // dK = tau * dK_acc and dV (this warpgroup's D/2 columns), staged over the K
            // and V tiles, which no MMA reads any more: the commit after the last dK
            // covers every MMA of this CTA (warpgroup 1 has not waited for it yet).  The
            // persistent kernel stages them apart (the next item's MMAs may be running);
            // its next item's first dV and dK MMAs wait for this warpgroup's arrivals
            // after these reads.
            if (ok && isteps > 0)
                ok = __all_sync(FULL, mbar_wait_sleep(bar_dk, (gs - 1) & 1, wd, kSiteDrain));
            if constexpr (PERSIST) {
                // the previous item's dK/dV store has read the staging area (thread 0
                // issued it and went on without waiting)
                if (threadIdx.x == 0) bulk_wait_read<0>();
                named_bar_sync(5, kEW);
            }
            // A split key tile: this chunk's partial dV and dK (fp32) go to its slot, and
            // the chunk that finishes last writes dK, dV from the sum of the slots, taken
            // in chunk order.  (Each chunk writes its slot, fences, then counts itself in;
            // the last one fences again before it reads the others' slots.)
            bool store = true;
            const int nchunks = SPLIT_ ? sh.sp_nchunk : 1;
            const bool split = SPLIT_ && nchunks > 1;
            const int tile = SPLIT_ ? sh.sp_tile : 0;
            const SplitPlan pl = split_layout(p.plan_tiles, p.plan_help);
            float* part = split ? reinterpret_cast<float*>(p.plan + pl.part) +
                                      static_cast<size_t>(reinterpret_cast<const uint32_t*>(p.plan + pl.slot)[tile]) *
                                          2 * 128 * D
                                : nullptr;
            if (split) {
                if (ok) {
                    tc_fence_after();
                    float* mine = part + static_cast<size_t>(sh.sp_chunk) * 2 * 128 * D;
#pragma unroll
                    for (int which = 0; which < 2; ++which) {
                        const uint32_t src = tmem + lane_off + (which ? L::kTmDK : L::kTmDV);
#pragma unroll
                        for (int cc = 0; cc < kDC; cc += 16) {
                            const int c0 = h * kDC + cc;
                            uint32_t o[16];
                            tmem_ld16(src + c0, o);
                            tmem_ld_wait(o);
                            // slot layout [dV, dK][column / 4][key row][4]: a warp's 32 rows
                            // of one float4 column group are 512 contiguous bytes
                            float4* dst4 = reinterpret_cast<float4*>(mine + static_cast<size_t>(which) * 128 * D) +
                                           (c0 / 4) * 128 + r;
#pragma unroll
                            for (int q = 0; q < 4; ++q)
                                dst4[q * 128] = make_float4(u2f(o[4 * q]), u2f(o[4 * q + 1]), u2f(o[4 * q + 2]),
                                                            u2f(o[4 * q + 3]));
                        }
                    }
                }
                __threadfence();
                named_bar_sync(4, kEW);
                if (threadIdx.x == 0)
                    sh.last_chunk =
                        ok && atomicAdd(reinterpret_cast<unsigned int*>(p.plan + pl.arrive) + tile, 1u) ==
                                  static_cast<unsigned>(nchunks - 1);
                named_bar_sync(4, kEW);
                store = sh.last_chunk != 0;
                if (store) __threadfence();
            }
            if (ok && store) {
                tc_fence_after();
                const uint32_t tDV = tmem + lane_off + L::kTmDV, tDK = tmem + lane_off + L::kTmDK;
#pragma unroll
                for (int which = 0; which < 2; ++which) {
                    uint8_t* dst = smem + (PERSIST ? L::kStageKV + (which ? L::kTile : 0) : (which ? L::kK : L::kV));
                    const float scale = which ? p.tau : 1.f;
                    const uint32_t src = which ? tDK : tDV;
#pragma unroll
                    for (int cc = 0; cc < kDC; cc += 16) {
                        const int c0 = h * kDC + cc;
                        uint32_t o[16];
                        if (split) {
                            // 8 columns of every chunk's slot in flight at once (the slots
                            // were written by other SMs, possibly on the other die), then
                            // added in chunk order; each load instruction reads 512
                            // contiguous bytes
                            float f[16];
#pragma unroll
                            for (int i = 0; i < 16; ++i) f[i] = 0.f;
#pragma unroll
                            for (int hq = 0; hq < 2; ++hq) {
                                float4 v[kSplitMaxChunks][2];
#pragma unroll
                                for (int c = 0; c < kSplitMaxChunks; ++c) {
                                    if (c < nchunks) {
                                        const float4* src4 =
                                            reinterpret_cast<const float4*>(
                                                part + (static_cast<size_t>(c) * 2 + which) * 128 * D) +
                                            (c0 / 4 + 2 * hq) * 128 + r;
                                        v[c][0] = __ldcg(src4);
                                        v[c][1] = __ldcg(src4 + 128);
                                    }
                                }
#pragma unroll
                                for (int c = 0; c < kSplitMaxChunks; ++c) {
                                    if (c < nchunks) {
#pragma unroll
                                        for (int e = 0; e < 2; ++e) {
                                            f[8 * hq + 4 * e] += v[c][e].x;
                                            f[8 * hq + 4 * e + 1] += v[c][e].y;
                                            f[8 * hq + 4 * e + 2] += v[c][e].z;
                                            f[8 * hq + 4 * e + 3] += v[c][e].w;
                                        }
                                    }
                                }
                            }
#pragma unroll
                            for (int i = 0; i < 16; ++i) o[i] = __float_as_uint(f[i]);
                        } else if (!SPARSE || isteps > 0) {
                            tmem_ld16(src + c0, o);
                            tmem_ld_wait(o);
                        } else {
#pragma unroll
                            for (int i = 0; i < 16; ++i) o[i] = 0u;  // no query sees these keys
                        }
                        const int box = c0 / 64;
#pragma unroll
                        for (int q = 0; q < 2; ++q) {
                            const int chunk = (c0 % 64) / 8 + q;
                            uint4 v;
                            v.x = pack_bf16(u2f(o[8 * q + 0]) * scale, u2f(o[8 * q + 1]) * scale);
                            v.y = pack_bf16(u2f(o[8 * q + 2]) * scale, u2f(o[8 * q + 3]) * scale);
                            v.z = pack_bf16(u2f(o[8 * q + 4]) * scale, u2f(o[8 * q + 5]) * scale);
                            v.w = pack_bf16(u2f(o[8 * q + 6]) * scale, u2f(o[8 * q + 7]) * scale);
                            *reinterpret_cast<uint4*>(dst + box * L::kBox + r * 128 +
                                                      ((chunk ^ (r & 7)) << 4)) = v;
                        }
                    }
                }
                fence_async_shared();
            }
            named_bar_sync(4, kEW);
            if (threadIdx.x == 0 && ok && store) {
                const uint32_t sv = sbase + (PERSIST ? L::kStageKV : L::kV);
                const uint32_t sk = sbase + (PERSIST ? L::kStageKV + L::kTile : L::kK);
                for (int b = 0; b < L::kBoxes; ++b) {
                    tma_store_3d(&tmdV, sv + b * L::kBox, b * 64, kvs, ibh);
                    tma_store_3d(&tmdK, sk + b * L::kBox, b * 64, kvs, ibh);
                }
                bulk_commit();
                if (!PERSIST) bulk_wait_read<0>();
            }
        }
        if (PERSIST && threadIdx.x == 0) bulk_wait_read<0>();  // the last item's store
    }

    // ------------------------------------------------------------ teardown --
    if (sh.abort_flag) drain_after_abort();
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// The split plan's inputs: the mask, the plan buffer (the dQ output) and the sizes.
struct PlanArgs {
    const uint8_t* blocks;
    long long head_stride;  // bytes between heads' masks (0: one mask)
    uint8_t* base;          // the plan buffer, laid out by split_layout
    int BH, n_kv, n_q, sms, n_help, n_slots, causal;
};

constexpr int kPlanWarps = kPlanThreads / 32;

__device__ __forceinline__ int block_sum(int v, int* red) {
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    __syncthreads();
    if (l == 0) red[w] = v;
    __syncthreads();
    int t = 0;
    for (int i = 0; i < kPlanWarps; ++i) t += red[i];
    return t;
}

// Exclusive prefix sum over the block of (a, b) pairs, in thread order.
__device__ __forceinline__ void block_scan2(int& a, int& b, int2* wsum) {
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    int ia = a, ib = b;
    for (int o = 1; o < 32; o <<= 1) {
        const int ya = __shfl_up_sync(0xffffffffu, ia, o), yb = __shfl_up_sync(0xffffffffu, ib, o);
        if (l >= o) {
            ia += ya;
            ib += yb;
        }
    }
    __syncthreads();
    if (l == 31) wsum[w] = make_int2(ia, ib);
    __syncthreads();
    if (w == 0) {
        int2 v = l < kPlanWarps ? wsum[l] : make_int2(0, 0);
        for (int o = 1; o < 32; o <<= 1) {
            const int ya = __shfl_up_sync(0xffffffffu, v.x, o), yb = __shfl_up_sync(0xffffffffu, v.y, o);
            if (l >= o) {
                v.x += ya;
                v.y += yb;
            }
        }
        if (l < kPlanWarps) wsum[l] = v;  // inclusive over warps
    }
    __syncthreads();
    const int2 before = w > 0 ? wsum[w - 1] : make_int2(0, 0);
    a = before.x + ia - a;
    b = before.y + ib - b;
}

// Split plan for the block-mask backward: one CTA of kPlanThreads threads.
// Counts each key tile's query tiles from the mask; takes one SM's share of the
// work, S = (query tiles + kSplitCtaSteps x key tiles) / SMs, as the chunk length T
// (at least kSplitMinSteps); splits a key tile of c > 1.5 T query tiles into
// ceil(c / T) chunks (at most kSplitMaxChunks), doubling T until the helper CTAs
// and partial slots suffice; and writes per key tile its chunk count and first
// slot, per helper its (key tile, chunk), zeroed arrival counters, and the number
// of helper chunks.  Key tiles are numbered in the main kernel's launch order,
// kt * BH + bh.
__global__ void __launch_bounds__(kPlanThreads, 1) fa_bwd_plan_kernel(const PlanArgs a) {
    // the previous kernels on the stream (the D kernel, and the dQ conversion of an
    // earlier call, which wrote this buffer) are done
    griddep_wait();
    __shared__ int red[kPlanWarps];
    __shared__ int2 wsum[kPlanWarps];
    __shared__ unsigned int cnt[kPlanThreads];  // [mask head][key tile]: query tiles
    const int n_tiles = a.BH * a.n_kv;          // at most kPlanThreads (the launcher's bound)
    const SplitPlan pl = split_layout(n_tiles, a.n_help);
    const int n_mh = a.head_stride ? a.BH : 1;
    cnt[threadIdx.x] = 0u;
    __syncthreads();
    // 1. query tiles per key tile.  A thread takes 16 neighbouring key tiles (one
    //    16-byte piece of a mask row when the rows allow) of one mask head over a
    //    slice of the query rows and adds its counts in.
    const int groups = (a.n_kv + 15) / 16;
    const int G = n_mh * groups;
    const int S = max(1, kPlanThreads / G);
    const int R = (a.n_q + S - 1) / S;
    const bool vec = (reinterpret_cast<uintptr_t>(a.blocks) & 15u) == 0 && (a.n_kv & 15) == 0 &&
                     (a.head_stride & 15) == 0;
    for (int u = threadIdx.x; u < G * S; u += kPlanThreads) {
        const int sl = u / G, g = u - sl * G;
        const int mh = g / groups, kt0 = (g - mh * groups) * 16;
        const uint8_t* m = a.blocks + mh * a.head_stride + kt0;
        const int q0 = sl * R, q1 = min(a.n_q, q0 + R);
        int c[16];
#pragma unroll
        for (int b = 0; b < 16; ++b) c[b] = 0;
#pragma unroll 4
        for (int qt = q0; qt < q1; ++qt) {
            const uint8_t* row = m + static_cast<long long>(qt) * a.n_kv;
            uint32_t wv[4] = {0u, 0u, 0u, 0u};
            if (vec) {
                const uint4 v = *reinterpret_cast<const uint4*>(row);
                wv[0] = v.x;
                wv[1] = v.y;
                wv[2] = v.z;
                wv[3] = v.w;
            } else {
#pragma unroll
                for (int b = 0; b < 16; ++b)
                    if (kt0 + b < a.n_kv && row[b] != 0) wv[b >> 2] |= 1u << (8 * (b & 3));
            }
#pragma unroll
            for (int b = 0; b < 16; ++b)  // causal: key tile kt0 + b counts query tiles from the diagonal
                c[b] += ((wv[b >> 2] >> (8 * (b & 3))) & 0xffu) != 0u && (!a.causal || qt >= kt0 + b);
        }
#pragma unroll
        for (int b = 0; b < 16; ++b)
            if (kt0 + b < a.n_kv && c[b] != 0) atomicAdd(&cnt[mh * a.n_kv + kt0 + b], static_cast<unsigned>(c[b]));
    }
    __syncthreads();
    // thread t plans key tile t (launch order kt * BH + bh)
    const int t = static_cast<int>(threadIdx.x);
    int my = 0;
    if (t < n_tiles) {
        const int kt = t / a.BH, bh = t - kt * a.BH;
        my = static_cast<int>(cnt[(a.head_stride ? bh : 0) * a.n_kv + kt]);
    }
    const long long work = static_cast<long long>(block_sum(my, red)) + static_cast<long long>(kSplitCtaSteps) * n_tiles;
    // 2. chunk length
    int T = static_cast<int>(max(static_cast<long long>(kSplitMinSteps), (work + a.sms - 1) / a.sms));
    auto chunks = [&](int c) { return 2 * c > 3 * T ? min(kSplitMaxChunks, (c + T - 1) / T) : 1; };
    int need_h = 0, need_s = 0;
    for (int it = 0; it < 16; ++it) {
        const int k = chunks(my);
        need_h = block_sum(k - 1, red);
        need_s = block_sum(k > 1 ? k : 0, red);
        if (need_h <= a.n_help && need_s <= a.n_slots) break;
        T *= 2;
    }
    if (need_h > a.n_help || need_s > a.n_slots) T = 1 << 28;  // no split at all
    // 3. exclusive prefix sums of helpers and slots in launch order
    const int k = chunks(my);
    int he = k - 1, se = k > 1 ? k : 0;
    block_scan2(he, se, wsum);
    if (t == kPlanThreads - 1) *reinterpret_cast<uint32_t*>(a.base + pl.hdr) = static_cast<uint32_t>(he + k - 1);
    // 4. the plan
    if (t < n_tiles) {
        a.base[pl.nchunk + t] = static_cast<uint8_t>(k);
        reinterpret_cast<uint32_t*>(a.base + pl.slot)[t] = static_cast<uint32_t>(se);
        reinterpret_cast<unsigned int*>(a.base + pl.arrive)[t] = 0u;
        uint32_t* help = reinterpret_cast<uint32_t*>(a.base + pl.help);
        for (int c = 1; c < k; ++c, ++he) {
            help[2 * he] = static_cast<uint32_t>(t);
            help[2 * he + 1] = static_cast<uint32_t>(c);
        }
    }
    // the main kernel, launched next as a dependent, reads the plan after its own wait
    griddep_launch_dependents();
}

// D_i = dO_i . O_i in fp32 and a zeroed dQ accumulator row; D/8 threads per row,
// each handling 8 bf16 of both inputs (16-byte loads).
template <int D>
__global__ void __launch_bounds__(256) fa_bwd_pre_kernel(const __nv_bfloat16* __restrict__ O,
                                                         const __nv_bfloat16* __restrict__ dO,
                                                         float* __restrict__ Dvec,
                                                         float* __restrict__ dQacc, int64_t rows) {
    // launched as a dependent of the previous kernel on the stream (usually the
    // forward, which writes O): wait for it
    griddep_wait();
    constexpr int TPR = D / 8;
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t row = tid / TPR;
    const int sub = static_cast<int>(tid % TPR);
    float acc = 0.f;
    if (row < rows) {
        const uint4 a = *reinterpret_cast<const uint4*>(O + row * D + sub * 8);
        const uint4 b = *reinterpret_cast<const uint4*>(dO + row * D + sub * 8);
        const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            acc = fmaf(u2f(aw[i] << 16), u2f(bw[i] << 16), acc);
            acc = fmaf(u2f(aw[i] & 0xffff0000u), u2f(bw[i] & 0xffff0000u), acc);
        }
        float4* z = reinterpret_cast<float4*>(dQacc + row * D + sub * 8);
        z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
        z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (row < rows && sub == 0) Dvec[row] = acc;
    // the main kernel may be scheduled once every CTA of this one is here: its
    // set-up and K, V loads overlap this kernel's last CTAs (it waits for this
    // kernel to finish before reading D or reducing into the accumulator)
    griddep_launch_dependents();
}

// dQ = bf16(tau * acc), 8 elements per thread, grid-stride.
__global__ void __launch_bounds__(256) fa_bwd_post_kernel(const float* __restrict__ acc,
                                                          __nv_bfloat16* __restrict__ dQ,
                                                          float tau, int64_t n8) {
    griddep_wait();  // the accumulator is complete once the main kernel is
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const float4 a = reinterpret_cast<const float4*>(acc)[2 * i];
        const float4 b = reinterpret_cast<const float4*>(acc)[2 * i + 1];
        uint4 o;
        o.x = pack_bf16(a.x * tau, a.y * tau);
        o.y = pack_bf16(a.z * tau, a.w * tau);
        o.z = pack_bf16(b.x * tau, b.y * tau);
        o.w = pack_bf16(b.z * tau, b.w * tau);
        reinterpret_cast<uint4*>(dQ)[i] = o;
    }
}


// Heads per launch-order group (a power of two, at most 16).  Measured on
// GB300, interleaved runs: causal problems do best with the group's Q, dO, K, V
// (bf16) and fp32 dQ accumulator near 128 MB (16k tokens, d = 128: 4 heads,
// 2.04 vs 2.12 ms with all 16 in flight), non-causal ones near 48 MB (1-2
// heads: 4.13 vs 4.45 ms), GPT-2-sized ones with 16.  A block mask keeps every
// head in flight: its few heavy key tiles (global anchors) must start first,
// and grouping left the last group's anchors as a tail (0.31 vs 0.50 ms).
int bwd_head_group(int BH, int N, int D, bool causal, int mask) {
    if (mask == kMaskBlocks) return BH;
    const double budget = (causal ? 128.0 : 48.0) * 1024 * 1024;
    const double per_head = static_cast<double>(N) * D * (4 * 2 + 4);
    int g = 1;
    while (g < 16 && 2.0 * g * per_head <= budget) g *= 2;
    return max(1, min(BH, g));
}

template <int D, bool CAUSAL, int MASK = kMaskNone>
cudaError_t launch_bwd_t(const BwdArgs& a, cudaStream_t stream) {
    using L = BwdLayout<D>;
    const int64_t rows = static_cast<int64_t>(a.BH) * a.N;
    // d = 128: four elementwise warpgroups (32 query columns each); d = 64: two
    // (four measured 4-8% slower there)
    constexpr int NWG = D == 128 ? 4 : 2;
    // short d = 64 problems without a mask, with more work items than SMs: the
    // persistent kernel, so that one item's set-up, first loads and epilogue
    // overlap the next's
    constexpr bool kCanPersist = D == 64 && MASK == kMaskNone;
    int sms = 0;
    if (kCanPersist || MASK == kMaskBlocks) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return cudaGetLastError();
    }
    const int n_kv = (a.N + kBK - 1) / kBK;
    // A block mask with few key tiles per SM: the split plan and the partial slots,
    // laid out in the dQ output (written only by the dQ conversion kernel, after the
    // main kernel); one helper CTA per SM
    PlanArgs pa{};
    const long long n_tiles = static_cast<long long>(a.BH) * n_kv;
    if (MASK == kMaskBlocks && a.dQ && n_tiles <= std::min<long long>(static_cast<long long>(kSplitTilesPerSm) * sms,
                                                                    kPlanThreads)) {
        const SplitPlan pl = split_layout(static_cast<int>(n_tiles), sms);
        const size_t dq_bytes = static_cast<size_t>(a.BH) * a.N * D * 2;
        const size_t slot_bytes = static_cast<size_t>(2) * 128 * D * 4;
        const long long n_slots = pl.part < dq_bytes ? static_cast<long long>((dq_bytes - pl.part) / slot_bytes) : 0;
        if (n_slots >= 2) {
            pa.blocks = a.blocks;
            pa.head_stride = a.blocks_head_stride;
            pa.base = static_cast<uint8_t*>(a.dQ);
            pa.BH = a.BH;
            pa.n_kv = n_kv;
            pa.n_q = (a.N + kBQ - 1) / kBQ;
            pa.sms = sms;
            pa.n_help = sms;
            pa.n_slots = static_cast<int>(std::min<long long>(n_slots, 1ll << 30));
            pa.causal = CAUSAL;
        }
    }
    // 1. D and a zeroed accumulator
    {
        constexpr int TPR = D / 8;
        const int64_t threads = rows * TPR;
        const unsigned blocks = static_cast<unsigned>((threads + 255) / 256);
        cudaError_t e = launch_dependent(fa_bwd_pre_kernel<D>, dim3(blocks), dim3(256), 0, stream,
                                         static_cast<const __nv_bfloat16*>(a.O),
                                         static_cast<const __nv_bfloat16*>(a.dO), a.D, a.dQacc, rows);
        if (e != cudaSuccess) return e;
    }
    // 2. main kernel
    {
        CUtensorMap tq, tk, tv, tdo, tacc, tdk, tdv;
        const auto BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
        if (!make_tile_map(&tq, a.Q, BF, 2, D, a.N, a.BH, 64, kBQ) ||
            !make_tile_map(&tk, a.K, BF, 2, D, a.N, a.BH, 64, kBK) ||
            !make_tile_map(&tv, a.V, BF, 2, D, a.N, a.BH, 64, kBK) ||
            !make_tile_map(&tdo, a.dO, BF, 2, D, a.N, a.BH, 64, kBQ) ||
            !make_tile_map(&tacc, a.dQacc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, D, a.N, a.BH, 32, kBQ) ||
            !make_tile_map(&tdk, a.dK, BF, 2, D, a.N, a.BH, 64, kBK) ||
            !make_tile_map(&tdv, a.dV, BF, 2, D, a.N, a.BH, 64, kBK))
            return cudaErrorInvalidValue;
        const long long items = static_cast<long long>(a.BH) * ((a.N + kBK - 1) / kBK);
        const bool persist = kCanPersist && a.N <= kBwdPersistMaxN && items > sms;
        constexpr auto kern = &fa_bwd_main_kernel<D, CAUSAL, MASK, NWG>;
        constexpr auto kern_p = &fa_bwd_main_kernel<D, CAUSAL, MASK, NWG, kCanPersist>;
        constexpr auto kern_s = &fa_bwd_main_kernel<D, CAUSAL, MASK, NWG, false, MASK == kMaskBlocks>;
        cudaError_t e = persist   ? set_max_dyn_smem_once<kern_p>(L::kBytesPersist)
                        : pa.base ? set_max_dyn_smem_once<kern_s>(L::kBytes)
                                  : set_max_dyn_smem_once<kern>(L::kBytes);
        if (e != cudaSuccess) return e;
        BwdParams p;
        p.LSE = a.LSE;
        p.Dvec = a.D;
        p.N = a.N;
        p.n_kv = n_kv;
        p.scale_log2 = a.tau * kLog2e;
        p.tau = a.tau;
        p.window = (a.window > 0 && a.window < a.N) ? a.window : 0;
        p.blocks = a.blocks;
        p.blocks_head_stride = a.blocks_head_stride;
        p.head_group = bwd_head_group(a.BH, a.N, D, CAUSAL, MASK);
        p.err = a.err;
        p.wait_limit_ns = a.wait_limit_ns;
        p.BH = a.BH;
        if (items > (1ll << 30)) return cudaErrorInvalidValue;
        p.items = static_cast<int>(items);
        p.plan = nullptr;
        p.plan_tiles = p.plan_help = 0;
        dim3 grid(static_cast<unsigned>(a.BH), static_cast<unsigned>(p.n_kv));
        if (persist) grid = dim3(static_cast<unsigned>(sms));
        if (a.ev_start) cudaEventRecord(a.ev_start, stream);
        if (pa.base) {
            e = launch_dependent(fa_bwd_plan_kernel, dim3(1), dim3(kPlanThreads), 0, stream, pa);
            if (e != cudaSuccess) return e;
            p.plan = pa.base;
            p.plan_tiles = static_cast<int>(n_tiles);
            p.plan_help = pa.n_help;
            grid = dim3(static_cast<unsigned>(n_tiles + pa.n_help));
        }
        e = persist   ? launch_dependent(kern_p, grid, dim3(bwd_threads(NWG)), L::kBytesPersist, stream, tq, tk,
                                         tv, tdo, tacc, tdk, tdv, p)
            : pa.base ? launch_dependent(kern_s, grid, dim3(bwd_threads(NWG)), L::kBytes, stream, tq, tk, tv, tdo,
                                         tacc, tdk, tdv, p)
                      : launch_dependent(kern, grid, dim3(bwd_threads(NWG)), L::kBytes, stream, tq, tk, tv, tdo,
                                         tacc, tdk, tdv, p);
        if (e == cudaSuccess && a.ev_stop) e = cudaEventRecord(a.ev_stop, stream);
        if (e != cudaSuccess) return e;
    }
    // 3. dQ = tau * accumulator
    {
        const int64_t n8 = rows * D / 8;
        int64_t blocks = (n8 + 255) / 256;
        if (blocks > 152 * 64) blocks = 152 * 64;
        return launch_dependent(fa_bwd_post_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0,
                                stream, static_cast<const float*>(a.dQacc),
                                static_cast<__nv_bfloat16*>(a.dQ), a.tau, n8);
    }
}

}  // namespace

cudaError_t launch_bwd(const BwdArgs& a, cudaStream_t stream) {
    if (a.blocks) {
        if (a.d == 64)
            return a.causal ? launch_bwd_t<64, true, kMaskBlocks>(a, stream)
                            : launch_bwd_t<64, false, kMaskBlocks>(a, stream);
        return a.causal ? launch_bwd_t<128, true, kMaskBlocks>(a, stream)
                        : launch_bwd_t<128, false, kMaskBlocks>(a, stream);
    }
    if (a.causal && a.window > 0 && a.window < a.N)
        return a.d == 64 ? launch_bwd_t<64, true, kMaskWindow>(a, stream)
                         : launch_bwd_t<128, true, kMaskWindow>(a, stream);
    if (a.d == 64) return a.causal ? launch_bwd_t<64, true>(a, stream) : launch_bwd_t<64, false>(a, stream);
    return a.causal ? launch_bwd_t<128, true>(a, stream) : launch_bwd_t<128, false>(a, stream);
}

}  // namespace fa
