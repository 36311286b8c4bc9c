// Forward kernel of exact IO-aware attention for sm_103a.
//
// Method (tonho.wtf "flash attention" entry, section "como funciona";
// "Atencao eficiente - FlashAttention, sparse e hibrida", "Insight 1 -
// Tiling" and "Insight 2 - Online softmax"): the scores of one query tile
// against one key block live only on chip; each row carries its running max m
// and sum l, and merging a new block rescales what was accumulated.  The N x N
// matrix never reaches device memory; only O and LSE = m + ln l are written.
//
// GB300 design (differs from the pages' A100 loop order, which walks key
// blocks outside and reloads O/m/l per query block):
//   - one CTA owns two 128-row query tiles of one (batch, head) and walks the
//     key blocks inside, so O, m and l never leave the chip;
//   - warp 8 streams K_j and V_j with TMA (128-byte swizzle) through a ring
//     of shared-memory slots guarded by full/empty mbarriers;
//   - warp 9 issues tcgen05.mma: S_t = Q_t K_j^T into tensor memory (fp32),
//     then O_t += P_t V_j with P_t read from tensor memory (bf16, written
//     over S_t's columns by the softmax warps);
//   - warps 0-3 / 4-7 run the online softmax of tile 0 / tile 1 (one thread
//     per row = one tensor-memory lane), so one tile's softmax overlaps the
//     other tile's MMAs;
//   - the exponent is taken with ex2 on tau*log2(e)-scaled scores; O is
//     rescaled only when a row's max grows by more than 2^8 (the stale max
//     is used for both O and l, so the final O / l is unchanged); the row
//     sums run as paired fp32 adds where the registers allow it;
//   - at d = 128 P is written over S, so a tile's next S waits for its P V;
//     at d = 64 (no mask) P has columns of its own and the next S is issued
//     as soon as the softmax has read S (PIPE below);
//   - causal: key blocks wholly above the diagonal are never loaded; the
//     diagonal block is masked element-wise.  Keys >= N in a ragged last
//     block are masked the same way;
//   - two-tile problems with a bf16 O (d = 128 sliding windows, d = 64 without a
//     mask, d = 128 without a mask up to 4096 tokens) run persistently when
//     there are more tile pairs than SMs (PERSIST below): one CTA per SM walks
//     a list of (batch*head, pair) items and keeps its barriers, tensor memory
//     and K/V ring; the next item's Q tiles and first K/V blocks load while the
//     current item's epilogue runs, and O is staged in a buffer of its own, so
//     an item change costs only the epilogue.
#include <cuda_bf16.h>

#include <cmath>

#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int kBM = 128;  // query rows per tile
constexpr int kBN = 128;  // keys per block
// TILES = 2 (the default): two query tiles per CTA, 10 warps, all 512 tensor-
// memory columns, one CTA per SM.  TILES = 1: one tile, 6 warps, 256 columns
// and a smaller ring (5 slots at d = 64, 2 at d = 128), so two CTAs share an SM
// and one's prologue and epilogue overlap the other's main loop: used for d = 64
// block masks (d = 64 short sequences and d = 128 block masks have persistent
// kernels of their own, fa_fwd_short.cu and fa_fwd_sparse.cu).
constexpr int threads_for(int tiles) { return tiles == 2 ? 320 : 192; }
constexpr float kLn2 = 0.69314718055994531f;
constexpr float kLog2e = 1.44269504088896341f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: P stays <= 2^8
// Which keys a query tile visits beyond causality.
enum : int { kMaskNone = 0, kMaskWindow = 1, kMaskBlocks = 2 };
constexpr int kMaskWords = kMaxMaskBlocks / 32;
constexpr int kSingleTileMaxN = 2048;  // d = 64 up to this length: one tile per CTA
constexpr int kPersistMaxN128 = 4096;  // d = 128 without a mask up to this length: the persistent pairs

template <int D, int TILES = 2>
struct FwdLayout {
    static constexpr int kTileBytes = kBM * D * 2;  // one 128-row bf16 tile
    static constexpr int kBoxBytes = 128 * 128;     // one [128 rows x 64 cols] bf16 TMA box
    static constexpr int kBoxes = D / 64;
    static constexpr int kStages = TILES == 2 ? ((D == 64) ? 8 : 4) : (D == 64 ? 5 : 2);
    static constexpr int kQ0 = 0;
    static constexpr int kQ1 = TILES == 2 ? kTileBytes : 0;
    static constexpr int kRing = TILES * kTileBytes;
    static constexpr int kBytes = kRing + kStages * kTileBytes;
    static constexpr int kDynSmem = kBytes + 1024;  // + alignment slack
    // persistent kernel: O of tile t is staged 64 columns (one TMA box) at a time in
    // a 16 KB area of its own at kBytes + t kBoxBytes, since Q_t is already loading
    // the next item's tile
    static constexpr int kDynSmemPersist = kBytes + 2 * kBoxBytes + 1024;
    static constexpr uint32_t kTmemS0 = 0, kTmemS1 = TILES == 2 ? 128 : 0;
    static constexpr uint32_t kTmemO0 = TILES == 2 ? 256 : 128, kTmemO1 = TILES == 2 ? 256 + D : 128;
    static constexpr uint32_t kTmemCols = TILES == 2 ? 512 : 256;
    // d = 64 leaves room for P (bf16, 64 columns per tile) beside S and O, so the
    // next block's S need not wait for P V (see PIPE in the kernel)
    static constexpr uint32_t kTmemP0 = TILES == 2 ? 384 : 192, kTmemP1 = TILES == 2 ? 448 : 192;
};

struct FwdParams {
    float* LSE;
    float* O32;
    __nv_bfloat16* O16;  // PERSIST: O written from registers
    int N;
    int n_pairs;
    float scale_log2;  // tau * log2(e)
    unsigned int* err;
    unsigned long long wait_limit_ns;
    int window;  // causal sliding window in keys (0 = none)
    const uint8_t* blocks;          // block mask [heads][n_kv][n_kv] (kMaskBlocks)
    long long blocks_head_stride;   // bytes between heads' masks (0: one mask)
    int BH;                         // PERSIST: batch*heads
    int items;                      // PERSIST: work items (BH pairs each)
};

struct FwdShared {
    uint64_t q_full;
    uint64_t q_empty;    // PERSIST: the item's MMAs are done; Q may take the next item's tiles
    uint64_t o_free[2];  // PERSIST: the softmax warps have read O_t out (one phase per item)
    uint64_t kv_full[8];
    uint64_t kv_empty[8];
    uint64_t s_full[2];
    uint64_t s_free[2];  // PIPE: the softmax has read S_t; its columns may take the next S
    uint64_t p_ready[2];
    uint64_t o_done[2];
    uint32_t tmem_base;
    int abort_flag;
    uint32_t use[2][kMaskWords];  // kMaskBlocks: bit j of use[t] = tile t visits key block j
};

// Wait-site ids recorded in the error word.
enum : uint32_t {
    kSiteProdEmpty = 1, kSiteMmaQ = 2, kSiteMmaKV = 3, kSiteMmaP = 4,
    kSiteSoftS = 5, kSiteSoftO = 6, kSiteEpi = 7, kSiteProdQ = 8, kSiteMmaOF = 9
};

__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }
__device__ __forceinline__ uint32_t f2u(float x) { return __float_as_uint(x); }

constexpr uint32_t kDescHi = sw128_desc_hi(1024);  // every operand tile: 8-row groups 1 KB apart

// S = Q K^T: both operands K-major [128 rows x D], D/64 boxes of 64 columns.
// q_lo / k_lo: low descriptor halves of the tiles' first box.
template <int D>
__device__ __forceinline__ void issue_s(uint32_t tmem_d, uint32_t q_lo, uint32_t k_lo) {
    constexpr uint32_t id = idesc_bf16(128, 128, false, false);
#pragma unroll
    for (int k = 0; k < D / 16; ++k) {
        const uint32_t off = ((k / 4) * (128 * 128) + (k % 4) * 32) >> 4;
        if (k == 0) mma_ss_warp<0>(tmem_d, q_lo + off, k_lo + off, kDescHi, id);
        else mma_ss_warp<1>(tmem_d, q_lo + off, k_lo + off, kDescHi, id);
    }
}

// O += P V: P from tensor memory, V an MN-major [128 keys x D] tile.
template <int D>
__device__ __forceinline__ void issue_pv(uint32_t tmem_o, uint32_t tmem_p, uint32_t v_lo,
                                         bool accumulate) {
    constexpr uint32_t id = idesc_bf16(128, D, false, true);
    if (accumulate) mma_ts_warp<1>(tmem_o, tmem_p, v_lo, kDescHi, id);
    else mma_ts_warp<0>(tmem_o, tmem_p, v_lo, kDescHi, id);
#pragma unroll
    for (int k = 1; k < kBN / 16; ++k)
        mma_ts_warp<1>(tmem_o, tmem_p + k * 8, v_lo + ((k * 2048) >> 4), kDescHi, id);
}

// One work item: query tiles q_start0 and q_start1 (q_start1 = N, no second
// tile, when TILES = 1) of head bh, and their key blocks [lo_t, hi_t): up to the
// diagonal when causal, and from the block holding key (first row - window + 1)
// with a sliding window.  The two ranges overlap or touch, so the loaders walk
// [jlo, jlo + nb) without gaps.  (A block mask recounts n_blk0, n_blk1 and nb.)
struct FwdItem {
    int bh, q_start0, q_start1, lo0, lo1, hi0, hi1, n_blk0, n_blk1, jlo, nb;
};

template <bool CAUSAL, int TILES>
__device__ __forceinline__ FwdItem fwd_item(int bh, int pair, int N, int n_kv, int window) {
    FwdItem it;
    it.bh = bh;
    it.q_start0 = pair * TILES * kBM;
    it.q_start1 = TILES == 2 ? it.q_start0 + kBM : N;
    it.hi0 = CAUSAL ? min(n_kv, it.q_start0 / kBN + 1) : n_kv;
    it.hi1 = it.q_start1 < N ? (CAUSAL ? min(n_kv, it.q_start1 / kBN + 1) : n_kv) : 0;
    it.lo0 = window > 0 ? max(0, it.q_start0 - window + 1) / kBN : 0;
    it.lo1 = window > 0 ? max(0, it.q_start1 - window + 1) / kBN : 0;
    it.n_blk0 = it.hi0 - it.lo0;
    it.n_blk1 = it.hi1 > 0 ? it.hi1 - it.lo1 : 0;
    it.jlo = it.lo0;
    it.nb = max(it.hi0, it.hi1) - it.jlo;
    return it;
}

// MASK: kMaskNone; kMaskWindow, a causal sliding window of p.window keys (only
// with CAUSAL); kMaskBlocks, the block mask p.blocks (bf16 O only).  PERSIST:
// one CTA per SM walks a list of (batch*head, pair) items (two tiles, bf16 O,
// no block mask).
template <int D, bool CAUSAL, bool O32, int MASK, int TILES, bool PERSIST = false>
__global__ void __launch_bounds__(threads_for(TILES), TILES == 2 ? 1 : 2)
fa_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
              const FwdParams p) {
    using L = FwdLayout<D, TILES>;
    constexpr int kProducerWarp = 4 * TILES, kMmaWarp = 4 * TILES + 1;
    constexpr bool LOCAL = MASK == kMaskWindow;
    constexpr bool SPARSE = MASK == kMaskBlocks;
    // d = 64 without a mask: P has its own tensor-memory columns, so S of block
    // j + 1 is issued as soon as the softmax has read S of block j, and the
    // softmax runs from block to block without waiting for P V and the next S
    constexpr bool PIPE = D == 64 && MASK == kMaskNone;
    static_assert(!PERSIST || (TILES == 2 && !O32 && !SPARSE && (D == 128 || PIPE)),
                  "persistent: two-tile pairs with a bf16 O, no block mask");
    // the row sums as paired fp32 adds (bitwise the same sums): measured faster
    // with a bf16 O at d = 128 (the sliding-window kernel too: 5% faster, and its
    // spills are gone) and in the d = 64 pipelined kernels (two-tile: 2-3%)
    constexpr bool PAIRED_SUMS = (PIPE && !O32) || (D == 128 && MASK != kMaskBlocks && !O32);
    // P is converted and stored in chunks of kPC packed columns: 16 at d = 128, which
    // frees the registers the paired sums need there, 32 at d = 64 and for the fp32
    // O (measured faster, and without spills, there)
    constexpr int kPC = (D == 128 && !O32) ? 16 : 32;
    extern __shared__ uint8_t smem_raw[];
    __shared__ FwdShared sh;
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t pad = ((raw + 1023u) & ~1023u) - raw;
    uint8_t* smem = smem_raw + pad;
    const uint32_t sbase = raw + pad;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int N = p.N;
    const int n_kv = (N + kBN - 1) / kBN;
    const int window = (CAUSAL && LOCAL) ? p.window : 0;
    // Work items in launch order (x, the batch*head, fastest; the pair index y
    // from the heaviest pair down): i = y BH + x.  Without PERSIST a CTA has one
    // item, its launch position.  With PERSIST, CTA c of G takes items c,
    // 2G - 1 - c, 2G + c, ... (a snake that balances heavy and light pairs
    // without a shared counter).
    auto item_of = [&](long long i) {
        const int y = static_cast<int>(i / p.BH);
        return fwd_item<CAUSAL, TILES>(static_cast<int>(i - static_cast<long long>(y) * p.BH),
                                       p.n_pairs - 1 - y, N, n_kv, window);
    };
    FwdItem it0 = PERSIST ? item_of(blockIdx.x)
                          : fwd_item<CAUSAL, TILES>(blockIdx.x, p.n_pairs - 1 - static_cast<int>(blockIdx.y),
                                                    N, n_kv, window);
    const int bh = it0.bh;
    const int q_start0 = it0.q_start0, q_start1 = it0.q_start1;
    [[maybe_unused]] const int hi0 = it0.hi0, hi1 = it0.hi1, lo0 = it0.lo0, lo1 = it0.lo1, jlo = it0.jlo;
    int n_blk0 = it0.n_blk0, n_blk1 = it0.n_blk1;
    int nb = it0.nb;  // key blocks loaded (with a block mask: counted below)
    // work item k of this CTA into it, or false past the last
    auto item_at = [&](int k, FwdItem& it) -> bool {
        if constexpr (PERSIST) {
            const int G = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
            const long long i = static_cast<long long>(k) * G + ((k & 1) ? G - 1 - c : c);
            if (i >= p.items) return false;
            it = item_of(i);
            return true;
        }
        if (k > 0) return false;
        it = it0;
        return true;
    };

    const uint32_t bar_q = smem_addr(&sh.q_full);
    const uint32_t bar_qe = smem_addr(&sh.q_empty);
    const uint32_t bar_of = smem_addr(&sh.o_free[0]);
    const uint32_t bar_kv_full = smem_addr(&sh.kv_full[0]);
    const uint32_t bar_kv_empty = smem_addr(&sh.kv_empty[0]);
    const uint32_t bar_s = smem_addr(&sh.s_full[0]);
    const uint32_t bar_sf = smem_addr(&sh.s_free[0]);
    const uint32_t bar_p = smem_addr(&sh.p_ready[0]);
    const uint32_t bar_o = smem_addr(&sh.o_done[0]);

    if (threadIdx.x == 0) {
        sh.abort_flag = 0;
        mbar_init(bar_q, 1);
        for (int s = 0; s < L::kStages; ++s) {
            mbar_init(bar_kv_full + 8 * s, 1);
            mbar_init(bar_kv_empty + 8 * s, 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(bar_s + 8 * t, 1);
            mbar_init(bar_sf + 8 * t, 128);
            mbar_init(bar_p + 8 * t, 128);
            mbar_init(bar_o + 8 * t, 1);
            mbar_init(bar_of + 8 * t, 128);
        }
        mbar_init(bar_qe, 1);
        mbar_init_fence();
        if constexpr (SPARSE && TILES == 1) {
            // the query tile is needed unless its mask row is empty: load it now, so
            // that its latency overlaps the mask read below
            mbar_arrive_expect_tx(bar_q, L::kTileBytes);
            for (int b = 0; b < L::kBoxes; ++b)
                tma_load_3d(sbase + L::kQ0 + b * L::kBoxBytes, &tmQ, bar_q, b * 64, q_start0, bh);
        }
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_addr(&sh.tmem_base), L::kTmemCols);
        tmem_relinquish();
    }
    if (warp == kProducerWarp && lane == 0) {
        tma_prefetch_map(&tmQ);
        tma_prefetch_map(&tmK);
        tma_prefetch_map(&tmV);
        if (!O32) tma_prefetch_map(&tmO);
    }
    if constexpr (SPARSE) {
        if (warp == kProducerWarp) {
            // bit j of use[t]: tile t's mask row has key block j set (and j is at or
            // below the diagonal when causal); one ballot per 32 blocks
            const uint8_t* m = p.blocks + bh * p.blocks_head_stride;
            const int qb[2] = {q_start0 / kBN, q_start1 / kBN};
            // eight 32-block words at a time: all their loads are in flight before
            // the first ballot
            for (int w0 = 0; w0 * 32 < n_kv; w0 += 8) {
                bool u[8][2];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int j = (w0 + i) * 32 + lane;
#pragma unroll
                    for (int t = 0; t < 2; ++t) {
                        u[i][t] = false;
                        if ((t == 0 || q_start1 < N) && j < n_kv && (!CAUSAL || j <= qb[t]))
                            u[i][t] = m[static_cast<long long>(qb[t]) * n_kv + j] != 0;
                    }
                }
#pragma unroll
                for (int i = 0; i < 8; ++i) {
#pragma unroll
                    for (int t = 0; t < 2; ++t) {
                        const uint32_t bits = __ballot_sync(0xffffffffu, u[i][t]);
                        if (lane == 0 && (w0 + i) * 32 < n_kv) sh.use[t][w0 + i] = bits;
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // a kernel launched after this one as its programmatic dependent (the
    // backward's D kernel) may be scheduled; it waits for this grid to finish
    griddep_launch_dependents();
    const uint32_t tmem = sh.tmem_base;
    const Watchdog wd{p.err, &sh.abort_flag, p.wait_limit_ns};
    if constexpr (SPARSE) {
        int c0 = 0, c1 = 0, cu = 0;
        for (int w = 0; w * 32 < n_kv; ++w) {
            c0 += __popc(sh.use[0][w]);
            c1 += __popc(sh.use[1][w]);
            cu += __popc(sh.use[0][w] | sh.use[1][w]);
        }
        n_blk0 = c0;
        n_blk1 = c1;
        nb = cu;
        it0.n_blk0 = c0;
        it0.n_blk1 = c1;
        it0.nb = cu;
    }

    if (warp >= kProducerWarp) {
        if (warp == kProducerWarp) {
            // ------------------------------------------------------- producer --
            // with a block mask, a tile that visits no key block loads no Q, and a
            // pair that visits none loads nothing.  Ring loads are numbered across
            // the items (g): the slot and the barrier phases follow g.
            if (lane == 0) {
                bool pok = true;
                int g0 = 0;  // ring loads of the earlier items
                FwdItem it;
                for (int k = 0; (PERSIST || k == 0) && pok && item_at(k, it); ++k) {
                    if (SPARSE && it.nb == 0) break;
                    // the Q buffers take this item's tiles once the previous item's MMAs are done
                    if (PERSIST && k > 0 && !mbar_wait(bar_qe, (k - 1) & 1, wd, kSiteProdQ)) break;
                    if (!(SPARSE && TILES == 1)) {  // (the one-tile block-mask kernel loaded Q at the start)
                        const bool q0 = !SPARSE || it.n_blk0 > 0;
                        uint32_t qbytes = L::kTileBytes * (q0 + (it.n_blk1 > 0));
                        mbar_arrive_expect_tx(bar_q, qbytes);
                        for (int b = 0; b < L::kBoxes; ++b) {
                            if (q0)
                                tma_load_3d(sbase + L::kQ0 + b * L::kBoxBytes, &tmQ, bar_q, b * 64, it.q_start0,
                                            it.bh);
                            if (it.n_blk1 > 0)
                                tma_load_3d(sbase + L::kQ1 + b * L::kBoxBytes, &tmQ, bar_q, b * 64, it.q_start1,
                                            it.bh);
                        }
                    }
                    int jb = -1;  // block mask: the block being loaded
                    for (int ld = 0; ld < 2 * it.nb; ++ld) {
                        const int g = g0 + ld;
                        const int slot = g % L::kStages;
                        if (g >= L::kStages &&
                            !mbar_wait(bar_kv_empty + 8 * slot, ((g / L::kStages) - 1) & 1, wd, kSiteProdEmpty)) {
                            pok = false;
                            break;
                        }
                        bool is_k = (ld & 1) == 0;
                        int blk = it.jlo + (ld >> 1);
                        if constexpr (PIPE) {
                            // the MMA warp's order: K0 K1 V0 K2 V1 ... K(nb-1) V(nb-2) V(nb-1)
                            is_k = ld == 0 || ((ld & 1) && ld < 2 * it.nb - 1);
                            blk = is_k ? (ld + 1) / 2 : (ld == 2 * it.nb - 1 ? it.nb - 1 : ld / 2 - 1);
                        }
                        const CUtensorMap* map = is_k ? &tmK : &tmV;
                        const uint32_t dst = sbase + L::kRing + slot * L::kTileBytes;
                        if constexpr (SPARSE) {
                            if ((ld & 1) == 0) jb = next_set_bit(sh.use[0], sh.use[1], jb + 1, n_kv);
                            blk = jb;
                        }
                        mbar_arrive_expect_tx(bar_kv_full + 8 * slot, L::kTileBytes);
                        for (int b = 0; b < L::kBoxes; ++b)
                            tma_load_3d(dst + b * L::kBoxBytes, map, bar_kv_full + 8 * slot, b * 64,
                                        blk * kBN, it.bh);
                    }
                    g0 += 2 * it.nb;
                }
            }
        } else if (warp == kMmaWarp) {
            // ------------------------------------------------------------ MMA --
            // The whole warp runs this loop; each MMA and commit is issued by one
            // elected lane (see mma_ss_warp).
            {
                const uint32_t tS[2] = {tmem + L::kTmemS0, tmem + L::kTmemS1};
                const uint32_t tO[2] = {tmem + L::kTmemO0, tmem + L::kTmemO1};
                const uint32_t qlo[2] = {sw128_desc_lo(sbase + L::kQ0, 16), sw128_desc_lo(sbase + L::kQ1, 16)};
                const uint32_t klo0 = sw128_desc_lo(sbase + L::kRing, 16);          // K: K-major
                const uint32_t vlo0 = sw128_desc_lo(sbase + L::kRing, 128 * 128);   // V: MN-major
                constexpr uint32_t kSlot = L::kTileBytes >> 4;
                if constexpr (SPARSE) {
                    // walk the union of the two tiles' key blocks; tile t takes the
                    // blocks whose bit is set in use[t]
                    auto uses = [&](int t, int j) { return ((sh.use[t][j >> 5] >> (j & 31)) & 1u) != 0; };
                    if (nb > 0) {
                        bool ok = __all_sync(0xffffffffu, mbar_wait(bar_q, 0, wd, kSiteMmaQ) &&
                                                              mbar_wait(bar_kv_full, 0, wd, kSiteMmaKV));
                        int j = next_set_bit(sh.use[0], sh.use[1], 0, n_kv);
                        if (ok) {
                            tc_fence_after();
#pragma unroll
                            for (int t = 0; t < 2; ++t) {
                                if (uses(t, j)) {
                                    issue_s<D>(tS[t], qlo[t], klo0);
                                    mma_commit_warp(bar_s + 8 * t);
                                }
                            }
                            mma_commit_warp(bar_kv_empty);
                        }
                        int cnt[2] = {0, 0};  // P.V products issued per tile
                        for (int u = 0; ok && u < nb; ++u) {
                            const int jn = next_set_bit(sh.use[0], sh.use[1], j + 1, n_kv);
                            const int lv = 2 * u + 1, lk = 2 * u + 2;
                            const int sv = lv % L::kStages, sk = lk % L::kStages;
                            if (!__all_sync(0xffffffffu,
                                            mbar_wait(bar_kv_full + 8 * sv, (lv / L::kStages) & 1, wd, kSiteMmaKV))) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                            bool k_ready = false;
#pragma unroll
                            for (int t = 0; t < 2; ++t) {
                                if (ok && uses(t, j)) {
                                    ok = __all_sync(0xffffffffu,
                                                    mbar_wait(bar_p + 8 * t, cnt[t] & 1, wd, kSiteMmaP));
                                    if (ok) {
                                        tc_fence_after();
                                        issue_pv<D>(tO[t], tS[t], vlo0 + sv * kSlot, cnt[t] > 0);
                                        mma_commit_warp(bar_o + 8 * t);
                                    }
                                    ++cnt[t];
                                }
                                if (ok && jn < n_kv && uses(t, jn)) {
                                    if (!k_ready) {
                                        ok = __all_sync(0xffffffffu,
                                                        mbar_wait(bar_kv_full + 8 * sk, (lk / L::kStages) & 1,
                                                                  wd, kSiteMmaKV));
                                        if (ok) tc_fence_after();
                                        k_ready = true;
                                    }
                                    if (ok) {
                                        issue_s<D>(tS[t], qlo[t], klo0 + sk * kSlot);
                                        mma_commit_warp(bar_s + 8 * t);
                                    }
                                }
                            }
                            if (!ok) break;
                            mma_commit_warp(bar_kv_empty + 8 * sv);
                            if (k_ready) mma_commit_warp(bar_kv_empty + 8 * sk);
                            j = jn;
                        }
                    }
                } else if constexpr (PIPE) {
                    // iteration j issues S(j) of both tiles (each once the softmax has read
                    // the tile's previous S), then P(j - 1) V(j - 1) of both tiles.  Ring
                    // loads (g0), each tile's blocks (cb) and Q fills (k) are counted
                    // across the items; the barrier phases follow them.
                    const uint32_t tP[2] = {tmem + L::kTmemP0, tmem + L::kTmemP1};
                    bool ok = true;
                    int g0 = 0;            // ring loads of the earlier items
                    int cb0 = 0, cb1 = 0;  // blocks of tile 0 / 1 in the earlier items
                    FwdItem it;
                    for (int k = 0; (PERSIST || k == 0) && ok && item_at(k, it); ++k) {
                        const int hi[2] = {it.hi0, it.n_blk1 > 0 ? it.hi1 : 0};
                        const int cb[2] = {cb0, cb1};
                        const int nbk = it.nb;
                        ok = __all_sync(0xffffffffu, mbar_wait(bar_q, k & 1, wd, kSiteMmaQ));
                        for (int j = 0; ok && j <= nbk; ++j) {
                            if (j < nbk) {
                                const int lk = g0 + (j == 0 ? 0 : 2 * j - 1), sk = lk % L::kStages;  // K_j
                                if (!__all_sync(0xffffffffu, mbar_wait(bar_kv_full + 8 * sk,
                                                                       (lk / L::kStages) & 1, wd, kSiteMmaKV))) {
                                    ok = false;
                                    break;
                                }
#pragma unroll
                                for (int t = 0; t < TILES; ++t) {
                                    if (ok && j < hi[t]) {
                                        // the tile's previous S (at j = 0 the previous item's last)
                                        if (cb[t] + j > 0)
                                            ok = __all_sync(0xffffffffu, mbar_wait(bar_sf + 8 * t, (cb[t] + j - 1) & 1,
                                                                                   wd, kSiteMmaP));
                                        if (ok) {
                                            tc_fence_after();
                                            issue_s<D>(tS[t], qlo[t], klo0 + sk * kSlot);
                                            mma_commit_warp(bar_s + 8 * t);
                                        }
                                    }
                                }
                                if (!ok) break;
                                mma_commit_warp(bar_kv_empty + 8 * sk);
                            }
                            if (j > 0) {
                                const int lv = g0 + min(2 * j, 2 * nbk - 1), sv = lv % L::kStages;  // V_(j-1)
                                if (!__all_sync(0xffffffffu, mbar_wait(bar_kv_full + 8 * sv,
                                                                       (lv / L::kStages) & 1, wd, kSiteMmaKV))) {
                                    ok = false;
                                    break;
                                }
#pragma unroll
                                for (int t = 0; t < TILES; ++t) {
                                    if (ok && j - 1 < hi[t]) {
                                        // the item's first P V overwrites O: the softmax warps must
                                        // have read the previous item's O out
                                        if (PERSIST && j == 1 && k > 0) {
                                            ok = __all_sync(0xffffffffu,
                                                            mbar_wait(bar_of + 8 * t, (k - 1) & 1, wd, kSiteMmaOF));
                                        }
                                        if (ok)
                                            ok = __all_sync(0xffffffffu, mbar_wait(bar_p + 8 * t, (cb[t] + j - 1) & 1,
                                                                                   wd, kSiteMmaP));
                                        if (ok) {
                                            tc_fence_after();
                                            issue_pv<D>(tO[t], tP[t], vlo0 + sv * kSlot, j > 1);
                                            mma_commit_warp(bar_o + 8 * t);
                                        }
                                    }
                                }
                                if (!ok) break;
                                mma_commit_warp(bar_kv_empty + 8 * sv);
                            }
                        }
                        // the Q tiles take the next item's once this item's MMAs are done
                        if (PERSIST && ok) mma_commit_warp(bar_qe);
                        g0 += 2 * nbk;
                        cb0 += it.n_blk0;
                        cb1 += it.n_blk1;
                    }
                } else {
                    // Ring loads (g), S_t / P_t / P_t V products (cb[t]) and Q fills
                    // (k) are counted across the items; the barrier phases follow them.
                    bool ok = true;
                    int g0 = 0;            // ring loads of the earlier items
                    int cb0 = 0, cb1 = 0;  // blocks of tile 0 / 1 in the earlier items
                    FwdItem it;
                    for (int k = 0; (PERSIST || k == 0) && ok && item_at(k, it); ++k) {
                        const int lo[2] = {it.lo0, it.lo1};
                        const int hi[2] = {it.hi0, it.n_blk1 > 0 ? it.hi1 : 0};
                        const int cb[2] = {cb0, cb1};
                        const int s0 = g0 % L::kStages;
                        ok = __all_sync(0xffffffffu, mbar_wait(bar_q, k & 1, wd, kSiteMmaQ) &&
                                                         mbar_wait(bar_kv_full + 8 * s0, (g0 / L::kStages) & 1, wd,
                                                                   kSiteMmaKV));
                        if (ok) {
                            tc_fence_after();
                            for (int t = 0; t < 2; ++t) {
                                if (lo[t] == it.jlo && hi[t] > it.jlo) {
                                    issue_s<D>(tS[t], qlo[t], klo0 + s0 * kSlot);
                                    mma_commit_warp(bar_s + 8 * t);
                                }
                            }
                            mma_commit_warp(bar_kv_empty + 8 * s0);
                        }
                        // before tile t's first P V of an item (accumulate = 0), the softmax
                        // warps must have read the previous item's O_t out
                        auto o_free_wait = [&](int t) -> bool {
                            if (!PERSIST || k == 0) return true;
                            const bool w = __all_sync(0xffffffffu,
                                                      mbar_wait(bar_of + 8 * t, (k - 1) & 1, wd, kSiteMmaOF));
                            if (w) tc_fence_after();
                            return w;
                        };
                        if constexpr (!LOCAL) {
                            // every tile starts at key block 0: tile t takes blocks [0, hi[t]).
                            // Both tiles' O must be free before the first P V (tile 1's
                            // epilogue ends about a block after tile 0's, while tile 0 runs
                            // its first softmax): the block loop stays that of one item.
                            if (ok) ok = o_free_wait(0) && (hi[1] == 0 || o_free_wait(1));
                            for (int j = 0; ok && j < it.nb; ++j) {
                                const int lv = g0 + 2 * j + 1, lk = g0 + 2 * j + 2;
                                const int sv = lv % L::kStages, sk = lk % L::kStages;
                                if (!__all_sync(0xffffffffu, mbar_wait(bar_kv_full + 8 * sv, (lv / L::kStages) & 1,
                                                                       wd, kSiteMmaKV))) {
                                    ok = false;
                                    break;
                                }
                                tc_fence_after();
                                bool k_ready = false;
                                for (int t = 0; t < 2 && ok; ++t) {
                                    if (j >= hi[t]) continue;
                                    if (!__all_sync(0xffffffffu,
                                                    mbar_wait(bar_p + 8 * t, (cb[t] + j) & 1, wd, kSiteMmaP))) {
                                        ok = false;
                                        break;
                                    }
                                    tc_fence_after();
                                    issue_pv<D>(tO[t], tS[t], vlo0 + sv * kSlot, j > 0);
                                    mma_commit_warp(bar_o + 8 * t);
                                    if (j + 1 < hi[t]) {
                                        if (!k_ready) {
                                            if (!__all_sync(0xffffffffu,
                                                            mbar_wait(bar_kv_full + 8 * sk, (lk / L::kStages) & 1,
                                                                      wd, kSiteMmaKV))) {
                                                ok = false;
                                                break;
                                            }
                                            tc_fence_after();
                                            k_ready = true;
                                        }
                                        issue_s<D>(tS[t], qlo[t], klo0 + sk * kSlot);
                                        mma_commit_warp(bar_s + 8 * t);
                                    }
                                }
                                if (!ok) break;
                                mma_commit_warp(bar_kv_empty + 8 * sv);
                                if (k_ready) mma_commit_warp(bar_kv_empty + 8 * sk);
                            }
                        } else {
                            // tile t takes blocks [lo[t], hi[t]); S of a tile's first block may
                            // be issued while the other tile is still in its leading blocks
                            for (int u = 0; ok && u < it.nb; ++u) {
                                const int j = it.jlo + u;  // key block
                                const int lv = g0 + 2 * u + 1, lk = g0 + 2 * u + 2;
                                const int sv = lv % L::kStages, sk = lk % L::kStages;
                                if (!__all_sync(0xffffffffu, mbar_wait(bar_kv_full + 8 * sv, (lv / L::kStages) & 1,
                                                                       wd, kSiteMmaKV))) {
                                    ok = false;
                                    break;
                                }
                                tc_fence_after();
                                bool k_ready = false;
                                // fully unrolled over the two tiles so the per-tile arrays stay in registers
#pragma unroll
                                for (int t = 0; t < 2; ++t) {
                                    if (ok && j >= lo[t] && j < hi[t]) {
                                        if (j == lo[t]) ok = o_free_wait(t);
                                        if (ok)
                                            ok = __all_sync(0xffffffffu,
                                                            mbar_wait(bar_p + 8 * t, (cb[t] + j - lo[t]) & 1, wd,
                                                                      kSiteMmaP));
                                        if (ok) {
                                            tc_fence_after();
                                            issue_pv<D>(tO[t], tS[t], vlo0 + sv * kSlot, j > lo[t]);
                                            mma_commit_warp(bar_o + 8 * t);
                                        }
                                    }
                                    if (ok && j + 1 >= lo[t] && j + 1 < hi[t]) {
                                        if (!k_ready) {
                                            ok = __all_sync(0xffffffffu,
                                                            mbar_wait(bar_kv_full + 8 * sk, (lk / L::kStages) & 1,
                                                                      wd, kSiteMmaKV));
                                            if (ok) tc_fence_after();
                                            k_ready = true;
                                        }
                                        if (ok) {
                                            issue_s<D>(tS[t], qlo[t], klo0 + sk * kSlot);
                                            mma_commit_warp(bar_s + 8 * t);
                                        }
                                    }
                                }
                                if (!ok) break;
                                mma_commit_warp(bar_kv_empty + 8 * sv);
                                if (k_ready) mma_commit_warp(bar_kv_empty + 8 * sk);
                            }
                        }
                        // the Q tiles take the next item's once this item's MMAs are done
                        // (committing right after the last S measured slower)
                        if (PERSIST && ok) mma_commit_warp(bar_qe);
                        g0 += 2 * it.nb;
                        cb0 += it.n_blk0;
                        cb1 += it.n_blk1;
                    }
                }
            }
            __syncwarp();
        }
    } else {
        // -------------------------------------------------------- softmax --
        const int t = warp >> 2;
        const int r = threadIdx.x & 127;
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + lane_off + (t ? L::kTmemS1 : L::kTmemS0);
        const uint32_t tO = tmem + lane_off + (t ? L::kTmemO1 : L::kTmemO0);
        // P: over S, or (PIPE) in its own columns
        const uint32_t tP = PIPE ? tmem + lane_off + (t ? L::kTmemP1 : L::kTmemP0) : tS;
        const uint32_t my_s = bar_s + 8 * t, my_p = bar_p + 8 * t, my_o = bar_o + 8 * t;
        const uint32_t my_sf = bar_sf + 8 * t;
        const float sl2 = p.scale_log2;
        bool ok = true;
        int cbt = 0;  // this tile's blocks in the earlier items (barrier phases)
        FwdItem it;
        for (int k = 0; (k == 0 || (PERSIST && ok)) && item_at(k, it); ++k) {
            const int ibh = it.bh;
            const int q_start = t ? it.q_start1 : it.q_start0;
            const int nbt = t ? it.n_blk1 : it.n_blk0;
            const int lot = t ? it.lo1 : it.lo0;
            const int row = q_start + r;
            float m_used = -INFINITY;
            float l = 0.f, l_mma = 0.f;
            int jsp = -1;  // block mask: the last key block visited
            for (int jj = 0; jj < nbt; ++jj) {
                int j = lot + jj;  // key block
                if constexpr (SPARSE) {
                    jsp = next_set_bit(sh.use[t], nullptr, jsp + 1, n_kv);
                    j = jsp;
                }
                // wait results are made warp-uniform: tcgen05.ld/st are warp-collective
                if (!__all_sync(0xffffffffu, mbar_wait(my_s, (cbt + jj) & 1, wd, kSiteSoftS))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t s[4][32];
                tmem_ld32(tS + 0, s[0]);
                tmem_ld32(tS + 32, s[1]);
                tmem_ld32(tS + 64, s[2]);
                tmem_ld32(tS + 96, s[3]);
                tmem_ld_wait(s[0]);
                tmem_ld_wait(s[1]);
                tmem_ld_wait(s[2]);
                tmem_ld_wait(s[3]);
                if constexpr (PIPE) {
                    tc_fence_before();
                    mbar_arrive(my_sf);  // S's columns may take the next block's scores now
                }

                const int kbase = j * kBN;
                const bool need_mask = (CAUSAL && kbase + kBN - 1 > q_start) || (kbase + kBN > N) ||
                                       (window > 0 && kbase <= q_start + kBM - 1 - window);
                if (need_mask) {
                    const int last = CAUSAL ? min(row, N - 1) : N - 1;  // last visible key
                    if constexpr (LOCAL) {
                        const int first = row - window + 1;  // first visible key
                        // a block is masked from above (diagonal, ragged end), from below (the
                        // window's lower edge) or, with a short window, both: one compare per
                        // score unless both
                        const bool upper = (kbase + kBN - 1 > q_start) || (kbase + kBN > N);
                        const bool lower = kbase <= q_start + kBM - 1 - window;
                        if (upper && lower) {
#pragma unroll
                            for (int c = 0; c < 128; ++c)
                                if (kbase + c > last || kbase + c < first) s[c >> 5][c & 31] = f2u(-INFINITY);
                        } else if (lower) {
#pragma unroll
                            for (int c = 0; c < 128; ++c)
                                if (kbase + c < first) s[c >> 5][c & 31] = f2u(-INFINITY);
                        } else {
#pragma unroll
                            for (int c = 0; c < 128; ++c)
                                if (kbase + c > last) s[c >> 5][c & 31] = f2u(-INFINITY);
                        }
                    } else {
#pragma unroll
                        for (int c = 0; c < 128; ++c)
                            if (kbase + c > last) s[c >> 5][c & 31] = f2u(-INFINITY);
                    }
                }
                float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
                for (int c = 0; c < 32; c += 2) {
                    mx0 = fmax3(mx0, u2f(s[0][c]), u2f(s[0][c + 1]));
                    mx1 = fmax3(mx1, u2f(s[1][c]), u2f(s[1][c + 1]));
                    mx2 = fmax3(mx2, u2f(s[2][c]), u2f(s[2][c + 1]));
                    mx3 = fmax3(mx3, u2f(s[3][c]), u2f(s[3][c + 1]));
                }
                const float m_cand = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * sl2;
                const bool grow = m_cand > m_used + kRescaleThreshold;
                float alpha = 1.f;
                if (grow) {
                    alpha = ex2(m_used - m_cand);  // 0 on the first block (m_used = -inf)
                    m_used = m_cand;
                }
                // unmasked kernels round the row sums' rescale and update separately (no
                // FMA contraction), so they and the persistent short forward give the
                // same LSE bits
                if constexpr (MASK == kMaskNone) {
                    l = __fmul_rn(l, alpha);
                    l_mma = __fmul_rn(l_mma, alpha);
                } else {
                    l *= alpha;
                    l_mma *= alpha;
                }
                const float neg_m = (m_used == -INFINITY) ? 0.f : -m_used;
                // Two row sums: l_mma over the bf16 P values the P.V MMA consumes (it
                // normalises O, so the weights actually applied sum to one) and l over
                // the fp32 values (it gives LSE).
                // the scale-and-subtract runs as one paired fp32 FMA per two scores
                const uint64_t c2 = f2_pack(sl2, sl2), nm2 = f2_pack(neg_m, neg_m);
                float ls0 = 0.f, ls1 = 0.f, lr0 = 0.f, lr1 = 0.f;
                uint64_t ls2 = 0;  // PAIRED_SUMS: ls0 and ls1 as one pair (bitwise the same sums)
#pragma unroll
                for (int h = 0; h < 64 / kPC; ++h) {
                    uint32_t pk[kPC];
#pragma unroll
                    for (int i = 0; i < kPC; ++i) {
                        const int c = h * 2 * kPC + 2 * i;
                        const float2 x = f2_unpack(ffma2(
                            f2_pack(u2f(s[c >> 5][c & 31]), u2f(s[c >> 5][(c & 31) + 1])), c2, nm2));
                        const float p0 = ex2(x.x), p1 = ex2(x.y);
                        pk[i] = pack_bf16(p0, p1);
                        if constexpr (PAIRED_SUMS) {
                            ls2 = fadd2(ls2, f2_pack(p0, p1));
                        } else {
                            ls0 += p0;
                            ls1 += p1;
                        }
                        // the bf16 values straight from the packed pair (16k causal:
                        // 0.725 -> 0.700 ms against unpacking them for fp32 adds)
                        add_bf16x2_f32(pk[i], lr0, lr1);
                    }
                    if (PIPE && h == 0 && jj > 0) {
                        // P's columns are free once the previous P V has read them
                        if (!__all_sync(0xffffffffu, mbar_wait(my_o, (cbt + jj - 1) & 1, wd, kSiteSoftO))) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                    }
                    if constexpr (kPC == 16) tmem_st16(tP + h * 16, pk);
                    else tmem_st32(tP + h * 32, pk);
                }
                if (!ok) break;
                if constexpr (PAIRED_SUMS) {
                    const float2 a2 = f2_unpack(ls2);
                    ls0 = a2.x;
                    ls1 = a2.y;
                }
                if constexpr (MASK == kMaskNone) {
                    l = __fadd_rn(l, __fadd_rn(ls0, ls1));
                    l_mma = __fadd_rn(l_mma, __fadd_rn(lr0, lr1));
                } else {
                    l += ls0 + ls1;
                    l_mma += lr0 + lr1;
                }
                if (jj > 0 && __any_sync(0xffffffffu, grow)) {
                    // rescale this warp's 32 rows of O once P_{j-1} V_{j-1} has landed (done after
                    // P_j is written so the S registers are dead; P_j V_j waits for p_ready)
                    if (!__all_sync(0xffffffffu, mbar_wait(my_o, (cbt + jj - 1) & 1, wd, kSiteSoftO))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int c0 = 0; c0 < D; c0 += 32) {
                        uint32_t o[32];
                        tmem_ld32(tO + c0, o);
                        tmem_ld_wait(o);
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = f2u(u2f(o[i]) * alpha);
                        tmem_st32(tO + c0, o);
                    }
                }
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(my_p);
            }

            // --------------------------------------------------------- epilogue --
            bool epi = ok && nbt > 0;
            if (epi) epi = __all_sync(0xffffffffu, mbar_wait(my_o, (cbt + nbt - 1) & 1, wd, kSiteEpi));
            cbt += nbt;
            if constexpr (PERSIST) {
                // O / l in bf16, 64 columns (one TMA box) at a time, through this tile's
                // staging area to a TMA store; O's columns go to the next item's P V
                // once both halves are read (one o_free phase per item, also for an
                // empty tile).  Thread 0 of the warpgroup issues the stores and waits
                // for a store's read of the area before the area is written again.
                const float inv_l = epi ? 1.f / l_mma : 0.f;
                uint8_t* stage = smem + L::kBytes + (t ? L::kBoxBytes : 0);
                if (epi) tc_fence_after();
#pragma unroll
                for (int h = 0; h < D / 64; ++h) {
                    if (r == 0) bulk_wait_read<0>();  // the area's previous store has read it
                    named_bar_sync(1 + t, 128);
                    if (epi) {
#pragma unroll
                        for (int c = 0; c < 2; ++c) {
                            uint32_t o[32];
                            tmem_ld32(tO + 64 * h + 32 * c, o);
                            tmem_ld_wait(o);
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                uint4 v;
                                v.x = pack_bf16(u2f(o[8 * q + 0]) * inv_l, u2f(o[8 * q + 1]) * inv_l);
                                v.y = pack_bf16(u2f(o[8 * q + 2]) * inv_l, u2f(o[8 * q + 3]) * inv_l);
                                v.z = pack_bf16(u2f(o[8 * q + 4]) * inv_l, u2f(o[8 * q + 5]) * inv_l);
                                v.w = pack_bf16(u2f(o[8 * q + 6]) * inv_l, u2f(o[8 * q + 7]) * inv_l);
                                const int chunk = 4 * c + q;
                                *reinterpret_cast<uint4*>(stage + r * 128 + ((chunk ^ (r & 7)) << 4)) = v;
                            }
                        }
                        fence_async_shared();
                    }
                    if (h == D / 64 - 1) {
                        if (epi) tc_fence_before();
                        mbar_arrive(bar_of + 8 * t);
                    }
                    named_bar_sync(1 + t, 128);
                    if (r == 0 && epi) {
                        tma_store_3d(&tmO, smem_addr(stage), 64 * h, q_start, ibh);
                        bulk_commit();
                    }
                }
                if (epi && row < N) p.LSE[static_cast<int64_t>(ibh) * N + row] = (m_used + __log2f(l)) * kLn2;
                continue;
            }
            if (epi) {
                tc_fence_after();
                const float inv_l = 1.f / l_mma;
                const int64_t bh_row = static_cast<int64_t>(ibh) * N + row;
                if (O32) {
                    float* dst = p.O32 + bh_row * D;
#pragma unroll
                    for (int c0 = 0; c0 < D; c0 += 32) {
                        uint32_t o[32];
                        tmem_ld32(tO + c0, o);
                        tmem_ld_wait(o);
                        if (row < N) {
#pragma unroll
                            for (int i = 0; i < 32; i += 4)
                                *reinterpret_cast<float4*>(dst + c0 + i) =
                                    make_float4(u2f(o[i]) * inv_l, u2f(o[i + 1]) * inv_l,
                                                u2f(o[i + 2]) * inv_l, u2f(o[i + 3]) * inv_l);
                        }
                    }
                } else {
                    uint8_t* stage = smem + (t ? L::kQ1 : L::kQ0);
#pragma unroll
                    for (int c0 = 0; c0 < D; c0 += 32) {
                        uint32_t o[32];
                        tmem_ld32(tO + c0, o);
                        tmem_ld_wait(o);
                        const int box = c0 / 64;
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const int chunk = (c0 % 64) / 8 + q;
                            uint4 v;
                            v.x = pack_bf16(u2f(o[8 * q + 0]) * inv_l, u2f(o[8 * q + 1]) * inv_l);
                            v.y = pack_bf16(u2f(o[8 * q + 2]) * inv_l, u2f(o[8 * q + 3]) * inv_l);
                            v.z = pack_bf16(u2f(o[8 * q + 4]) * inv_l, u2f(o[8 * q + 5]) * inv_l);
                            v.w = pack_bf16(u2f(o[8 * q + 6]) * inv_l, u2f(o[8 * q + 7]) * inv_l);
                            *reinterpret_cast<uint4*>(stage + box * L::kBoxBytes + r * 128 +
                                                      ((chunk ^ (r & 7)) << 4)) = v;
                        }
                    }
                    fence_async_shared();
                }
                if (row < N) p.LSE[bh_row] = (m_used + __log2f(l)) * kLn2;
            }
            bool empty_tile = false;
            if constexpr (SPARSE) {
                // a tile whose mask row visits no key block: every row is the empty
                // sum, O = 0 and LSE = -inf, staged as zeros over its Q buffer (the one-tile
                // kernel loaded Q all the same: that copy must land first)
                empty_tile = nbt == 0 && q_start < N;
                if (empty_tile) {
                    bool q_in = true;
                    if constexpr (TILES == 1) q_in = __all_sync(0xffffffffu, mbar_wait(bar_q, 0, wd, kSiteEpi));
                    if (q_in) {
                        uint8_t* stage = smem + (t ? L::kQ1 : L::kQ0);
#pragma unroll
                        for (int b = 0; b < L::kBoxes; ++b)
#pragma unroll
                            for (int c = 0; c < 8; ++c)
                                *reinterpret_cast<uint4*>(stage + b * L::kBoxBytes + r * 128 + c * 16) =
                                    make_uint4(0u, 0u, 0u, 0u);
                        fence_async_shared();
                        if (row < N) p.LSE[static_cast<int64_t>(ibh) * N + row] = -INFINITY;
                    }
                    epi = q_in;
                }
            }
            if (!O32 && (nbt > 0 || empty_tile)) {
                // every thread of the warpgroup reaches this barrier, even after an abort
                named_bar_sync(1 + t, 128);
                if (r == 0 && epi) {
                    const uint32_t src = sbase + (t ? L::kQ1 : L::kQ0);
                    for (int b = 0; b < L::kBoxes; ++b)
                        tma_store_3d(&tmO, src + b * L::kBoxBytes, b * 64, q_start, ibh);
                    bulk_commit();
                    bulk_wait_read<0>();
                }
            }
        }
    }

    // ------------------------------------------------------------ teardown --
    if (PERSIST && warp < 4 * TILES && (threadIdx.x & 127) == 0) bulk_wait_read<0>();
    if (sh.abort_flag) drain_after_abort();
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, L::kTmemCols);
    }
}

template <int D, bool CAUSAL, bool O32, int MASK = kMaskNone, int TILES = 2>
cudaError_t launch_fwd_t(const FwdArgs& a, cudaStream_t stream) {
    using L = FwdLayout<D, TILES>;
    CUtensorMap tq, tk, tv, to;
    if (!make_tile_map(&tq, a.Q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, a.N, a.BH, 64, kBM) ||
        !make_tile_map(&tk, a.K, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, a.N, a.BH, 64, kBN) ||
        !make_tile_map(&tv, a.V, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, a.N, a.BH, 64, kBN))
        return cudaErrorInvalidValue;
    if (O32) {
        to = tq;
    } else if (!make_tile_map(&to, a.O, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, a.N, a.BH, 64, kBM)) {
        return cudaErrorInvalidValue;
    }
    // Pairs with a bf16 O and more pairs than SMs: the persistent kernel, so that
    // one item's epilogue and the next item's first loads overlap the work of the
    // SM's other tile.  Measured against one CTA per pair: d = 64 3-6% faster from
    // 3k to 32k tokens (up to 2k tokens the one-tile persistent kernel of
    // fa_fwd_short.cu is faster still); d = 128 sliding windows 3% faster; d = 128
    // without a mask 1-7% faster up to 4096 tokens, where the items are short, but
    // 1-3% slower from 8192 up, where the hardware's dynamic CTA scheduling
    // balances long causal pairs better than a static list.
    constexpr bool kCanPersist = TILES == 2 && !O32 && MASK != kMaskBlocks && (D == 128 || MASK == kMaskNone);
    const int n_pairs = (a.N + TILES * kBM - 1) / (TILES * kBM);
    const long long items = static_cast<long long>(a.BH) * n_pairs;
    int sms = 0;
    if (kCanPersist) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return cudaGetLastError();
    }
    if (items > (1ll << 30)) return cudaErrorInvalidValue;
    // d = 128 without a mask: only up to 4096 tokens (below)
    const bool persist = kCanPersist && items > sms && (D != 128 || MASK != kMaskNone || a.N <= kPersistMaxN128);
    constexpr auto kern = &fa_fwd_kernel<D, CAUSAL, O32, MASK, TILES>;
    constexpr auto kern_p = &fa_fwd_kernel<D, CAUSAL, O32, MASK, TILES, kCanPersist>;
    cudaError_t e = persist ? set_max_dyn_smem_once<kern_p>(L::kDynSmemPersist)
                            : set_max_dyn_smem_once<kern>(L::kDynSmem);
    if (e != cudaSuccess) return e;
    FwdParams p;
    p.LSE = a.LSE;
    p.O32 = O32 ? static_cast<float*>(a.O) : nullptr;
    p.O16 = O32 ? nullptr : static_cast<__nv_bfloat16*>(a.O);
    p.BH = a.BH;
    p.items = static_cast<int>(items);
    p.N = a.N;
    p.window = (a.window > 0 && a.window < a.N) ? a.window : 0;
    p.blocks = a.blocks;
    p.blocks_head_stride = a.blocks_head_stride;
    p.n_pairs = n_pairs;
    p.scale_log2 = a.tau * kLog2e;
    p.err = a.err;
    p.wait_limit_ns = a.wait_limit_ns;
    dim3 grid(static_cast<unsigned>(a.BH), static_cast<unsigned>(p.n_pairs));
    if (persist) grid = dim3(static_cast<unsigned>(sms));
    if (a.ev_start) cudaEventRecord(a.ev_start, stream);
    if (persist) kern_p<<<grid, threads_for(TILES), L::kDynSmemPersist, stream>>>(tq, tk, tv, to, p);
    else kern<<<grid, threads_for(TILES), L::kDynSmem, stream>>>(tq, tk, tv, to, p);
    e = cudaGetLastError();
    if (e == cudaSuccess && a.ev_stop) e = cudaEventRecord(a.ev_stop, stream);
    return e;
}

}  // namespace

cudaError_t launch_fwd(const FwdArgs& a, cudaStream_t stream) {
    if (a.blocks) {  // a block mask leaves each query tile little work: one tile per CTA or item
        if (a.o32) return cudaErrorInvalidValue;
        if (a.d == 64)
            return a.causal ? launch_fwd_t<64, true, false, kMaskBlocks, 1>(a, stream)
                            : launch_fwd_t<64, false, false, kMaskBlocks, 1>(a, stream);
        return launch_fwd_sparse(a, stream);  // persistent, fa_fwd_sparse.cu
    }
    if (a.causal && !a.o32 && a.window > 0 && a.window < a.N)
        return a.d == 64 ? launch_fwd_t<64, true, false, kMaskWindow>(a, stream)
                         : launch_fwd_t<128, true, false, kMaskWindow>(a, stream);
    if (a.d == 64) {
        if (!a.o32 && a.N <= kSingleTileMaxN) return launch_fwd_short(a, stream);
        if (a.causal) return a.o32 ? launch_fwd_t<64, true, true>(a, stream) : launch_fwd_t<64, true, false>(a, stream);
        return a.o32 ? launch_fwd_t<64, false, true>(a, stream) : launch_fwd_t<64, false, false>(a, stream);
    }
    if (a.causal) return a.o32 ? launch_fwd_t<128, true, true>(a, stream) : launch_fwd_t<128, true, false>(a, stream);
    return a.o32 ? launch_fwd_t<128, false, true>(a, stream) : launch_fwd_t<128, false, false>(a, stream);
}

}  // namespace fa
