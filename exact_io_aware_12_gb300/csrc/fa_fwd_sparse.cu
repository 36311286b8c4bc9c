// Persistent block-sparse forward, d = 128 (bf16 O).
//
// The method is the forward of fa_fwd.cu ("Atencao eficiente - FlashAttention,
// sparse e hibrida", "Insight 1 - Tiling", "Insight 2 - Online softmax" and
// "Sparse e hibrida"; tonho.wtf "flash attention", "como funciona"): one
// 128-row query tile walks the key blocks its mask row selects with the online
// softmax; O / l and LSE = m + ln l are written at the end.  What changes is
// the scheduling.  With a local + global mask a query tile has ~6 key blocks,
// and a CTA that owns one tile spent ~26% of its life outside its main loop
// (measured: mask read and set-up ~1.1 us, ~1.9 us to the first S, ~1.6 us of
// epilogue, against ~13.9 us of blocks).  Here each CTA (two per SM) walks a
// list of query tiles and keeps its barriers and tensor memory:
//   - the loader warp turns the next tile's mask row into a block list (in one
//     of two shared-memory slots) and loads its Q as soon as the last S of the
//     current tile has read the single Q buffer;
//   - the K/V ring streams from one tile into the next;
//   - O and LSE go from registers to global memory, so Q never holds O.
//
// Work item i of BH * n_q is query tile (n_q - 1 - i / BH) of head (i % BH).
// CTA c of G takes items c, 2G - 1 - c, 2G + c, ... (a snake).
//
// Per tile the pipeline and the arithmetic are those of the d = 128 two-tile
// kernel of fa_fwd.cu, one tile wide: P is written over S's first 64 columns,
// so S of block j + 1 is issued after P V of block j; the row sums run as
// paired fp32 adds, rounded separately, in the same order, so an all-ones mask
// gives the dense kernel's bits.
#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>

#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int kBM = 128, kBN = 128, kD = 128;
constexpr int kThreads = 192;                  // softmax warps 0-3, loader 4, MMA 5
constexpr int kLoaderWarp = 4, kMmaWarp = 5;
constexpr int kStages = 2;                     // K/V ring slots
constexpr int kTile = kBM * kD * 2;            // one [128 x 128] bf16 tile (two TMA boxes)
constexpr int kBox = 128 * 128;                // one [128 rows x 64 cols] bf16 box
constexpr int kQ = 0;
constexpr int kRing = kTile;
constexpr int kBytes = kRing + kStages * kTile;
constexpr int kDynSmem = kBytes + 1024;        // + alignment slack
constexpr uint32_t kTmS = 0, kTmO = 128, kTmCols = 256;
constexpr int kPC = 16;                        // P packed columns per tensor-memory store
constexpr int kWords = kMaxMaskBlocks / 32;
constexpr float kLn2 = 0.69314718055994531f;
constexpr float kLog2e = 1.44269504088896341f;
constexpr float kRescaleThreshold = 8.0f;      // log2 units: P stays <= 2^8

struct SparseParams {
    __nv_bfloat16* O;
    float* LSE;
    const uint8_t* blocks;          // [heads][n_kv][n_kv]
    long long blocks_head_stride;   // bytes between heads' masks (0: one mask)
    int N, BH, n_q, n_kv, items;
    float scale_log2;
    unsigned int* err;
    unsigned long long wait_limit_ns;
};

struct SparseShared {
    uint64_t q_full, q_empty;
    uint64_t item_ready[2], item_done[2];
    uint64_t kv_full[kStages], kv_empty[kStages];
    uint64_t s_full, p_ready, o_done, o_free;
    uint32_t use[2][kWords];  // slot b: bit j = the tile visits key block j
    int n_blk[2];             // slot b: the number of such blocks
    uint32_t tmem_base;
    int abort_flag;
};

enum : uint32_t {
    kSiteItemDone = 61, kSiteQEmpty = 62, kSiteKvEmpty = 63, kSiteItem = 64, kSiteMmaQ = 65,
    kSiteMmaKV = 66, kSiteMmaP = 67, kSiteMmaOF = 68, kSiteSoftS = 69, kSiteSoftO = 70, kSiteEpi = 71
};

__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }
__device__ __forceinline__ uint32_t f2u(float x) { return __float_as_uint(x); }

constexpr uint32_t kDescHi = sw128_desc_hi(1024);

// The k-th work item of this CTA (snake order), or -1 past the end.
__device__ __forceinline__ int item_of(int k, int c, int G, int items) {
    const long long idx = static_cast<long long>(k) * G + ((k & 1) ? G - 1 - c : c);
    return idx < items ? static_cast<int>(idx) : -1;
}

// The first set bit of `bits` at or after j (bit j of word j / 32), or n.
__device__ __forceinline__ int next_block(const uint32_t* bits, int j, int n) {
    while (j < n) {
        const uint32_t w = bits[j >> 5] >> (j & 31);
        if (w) return min(n, j + __ffs(w) - 1);
        j = (j | 31) + 1;
    }
    return n;
}

// S = Q K^T: both K-major [128 rows x 128], two 64-column boxes.
__device__ __forceinline__ void issue_s(uint32_t tmem_d, uint32_t q_lo, uint32_t k_lo) {
    constexpr uint32_t id = idesc_bf16(128, 128, false, false);
#pragma unroll
    for (int k = 0; k < kD / 16; ++k) {
        const uint32_t off = ((k / 4) * kBox + (k % 4) * 32) >> 4;
        if (k == 0) mma_ss_warp<0>(tmem_d, q_lo + off, k_lo + off, kDescHi, id);
        else mma_ss_warp<1>(tmem_d, q_lo + off, k_lo + off, kDescHi, id);
    }
}

// O += P V: P (bf16) packed over S's first 64 columns, V an MN-major [128 keys x 128] tile.
__device__ __forceinline__ void issue_pv(uint32_t tmem_o, uint32_t tmem_p, uint32_t v_lo, bool accumulate) {
    constexpr uint32_t id = idesc_bf16(128, kD, false, true);
    if (accumulate) mma_ts_warp<1>(tmem_o, tmem_p, v_lo, kDescHi, id);
    else mma_ts_warp<0>(tmem_o, tmem_p, v_lo, kDescHi, id);
#pragma unroll
    for (int k = 1; k < kBN / 16; ++k)
        mma_ts_warp<1>(tmem_o, tmem_p + k * 8, v_lo + ((k * 2048) >> 4), kDescHi, id);
}

template <bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 2)
fa_fwd_sparse_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const SparseParams p) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ SparseShared sh;
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t pad = ((raw + 1023u) & ~1023u) - raw;
    const uint32_t sbase = raw + pad;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int N = p.N, n_kv = p.n_kv;
    const int G = gridDim.x, c = blockIdx.x;

    const uint32_t bar_qf = smem_addr(&sh.q_full);
    const uint32_t bar_qe = smem_addr(&sh.q_empty);
    const uint32_t bar_ir = smem_addr(&sh.item_ready[0]);
    const uint32_t bar_id = smem_addr(&sh.item_done[0]);
    const uint32_t bar_kvf = smem_addr(&sh.kv_full[0]);
    const uint32_t bar_kve = smem_addr(&sh.kv_empty[0]);
    const uint32_t bar_s = smem_addr(&sh.s_full);
    const uint32_t bar_p = smem_addr(&sh.p_ready);
    const uint32_t bar_o = smem_addr(&sh.o_done);
    const uint32_t bar_of = smem_addr(&sh.o_free);

    if (threadIdx.x == 0) {
        sh.abort_flag = 0;
        mbar_init(bar_qf, 1);
        mbar_init(bar_qe, 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar_ir + 8 * b, 1);
            mbar_init(bar_id + 8 * b, 129);  // the MMA warp's lane 0 and the 128 softmax threads
        }
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar_kvf + 8 * s, 1);
            mbar_init(bar_kve + 8 * s, 1);
        }
        mbar_init(bar_s, 1);
        mbar_init(bar_p, 128);
        mbar_init(bar_o, 1);
        mbar_init(bar_of, 128);
        mbar_init_fence();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_addr(&sh.tmem_base), kTmCols);
        tmem_relinquish();
    }
    if (warp == kLoaderWarp && lane == 0) {
        tma_prefetch_map(&tmQ);
        tma_prefetch_map(&tmK);
        tma_prefetch_map(&tmV);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    griddep_launch_dependents();
    const uint32_t tmem = sh.tmem_base;
    const Watchdog wd{p.err, &sh.abort_flag, p.wait_limit_ns};

    if (warp == kLoaderWarp) {
        // -------------------------------------------------------------- loader --
        // Per item: the block list (all lanes), then Q and the K/V blocks (lane 0).
        int g = 0;  // K/V loads issued for earlier items
        bool ok = true;
        for (int k = 0; ok; ++k) {
            const int idx = item_of(k, c, G, p.items);
            if (idx < 0) break;
            const int qt = p.n_q - 1 - idx / p.BH, bh = idx % p.BH;
            const int b = k & 1;
            // slot b held item k - 2's list until both readers were done with it
            if (k >= 2 && !__all_sync(0xffffffffu, mbar_wait(bar_id + 8 * b, ((k >> 1) - 1) & 1, wd, kSiteItemDone)))
                break;
            const uint8_t* m = p.blocks + bh * p.blocks_head_stride + static_cast<long long>(qt) * n_kv;
            int cnt = 0;
            // eight 32-block words at a time: their loads are in flight before the ballots
            for (int w0 = 0; w0 * 32 < n_kv; w0 += 8) {
                bool u[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int j = (w0 + i) * 32 + lane;
                    u[i] = j < n_kv && (!CAUSAL || j <= qt) && m[j] != 0;
                }
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const uint32_t bits = __ballot_sync(0xffffffffu, u[i]);
                    cnt += __popc(bits);
                    if (lane == 0 && (w0 + i) * 32 < n_kv) sh.use[b][w0 + i] = bits;
                }
            }
            if (lane == 0) sh.n_blk[b] = cnt;
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_ir + 8 * b);
            if (lane == 0) {
                // the single Q buffer: free once the last S of item k - 1 has read it
                if (k >= 1 && !mbar_wait(bar_qe, (k - 1) & 1, wd, kSiteQEmpty)) ok = false;
                if (ok) {
                    mbar_arrive_expect_tx(bar_qf, kTile);
                    for (int x = 0; x < 2; ++x)
                        tma_load_3d(sbase + kQ + x * kBox, &tmQ, bar_qf, x * 64, qt * kBM, bh);
                }
                int jb = -1;
                for (int ld = 0; ok && ld < 2 * cnt; ++ld, ++g) {
                    const int slot = g % kStages;
                    if (g >= kStages && !mbar_wait(bar_kve + 8 * slot, ((g / kStages) - 1) & 1, wd, kSiteKvEmpty)) {
                        ok = false;
                        break;
                    }
                    const bool is_k = (ld & 1) == 0;  // K0 V0 K1 V1 ...
                    if (is_k) jb = next_block(sh.use[b], jb + 1, n_kv);
                    mbar_arrive_expect_tx(bar_kvf + 8 * slot, kTile);
                    for (int x = 0; x < 2; ++x)
                        tma_load_3d(sbase + kRing + slot * kTile + x * kBox, is_k ? &tmK : &tmV,
                                    bar_kvf + 8 * slot, x * 64, jb * kBN, bh);
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        // ----------------------------------------------------------------- MMA --
        const uint32_t tS = tmem + kTmS, tO = tmem + kTmO;
        const uint32_t qlo = sw128_desc_lo(sbase + kQ, 16);
        const uint32_t klo0 = sw128_desc_lo(sbase + kRing, 16);          // K: K-major
        const uint32_t vlo0 = sw128_desc_lo(sbase + kRing, 128 * 128);   // V: MN-major
        constexpr uint32_t kSlot = kTile >> 4;
        int g = 0, gblk = 0;
        bool ok = true;
        for (int k = 0; ok; ++k) {
            const int idx = item_of(k, c, G, p.items);
            if (idx < 0) break;
            const int b = k & 1;
            ok = __all_sync(0xffffffffu, mbar_wait(bar_ir + 8 * b, (k >> 1) & 1, wd, kSiteItem) &&
                                             mbar_wait(bar_qf, k & 1, wd, kSiteMmaQ));
            if (!ok) break;
            const int nb = sh.n_blk[b];
            if (nb == 0) {
                mma_commit_warp(bar_qe);  // nothing reads this Q
            } else {
                // S(0): K_0 in slot g
                {
                    const int sk = g % kStages;
                    ok = __all_sync(0xffffffffu, mbar_wait(bar_kvf + 8 * sk, (g / kStages) & 1, wd, kSiteMmaKV));
                    if (!ok) break;
                    tc_fence_after();
                    issue_s(tS, qlo, klo0 + sk * kSlot);
                    mma_commit_warp(bar_s);
                    mma_commit_warp(bar_kve + 8 * sk);
                    if (nb == 1) mma_commit_warp(bar_qe);
                }
                for (int j = 0; j < nb; ++j) {
                    const int gv = g + 2 * j + 1, sv = gv % kStages;  // V_j
                    // the first P V of an item overwrites O: the previous item's
                    // epilogue must have read it out
                    ok = __all_sync(0xffffffffu,
                                    mbar_wait(bar_kvf + 8 * sv, (gv / kStages) & 1, wd, kSiteMmaKV) &&
                                        mbar_wait(bar_p, (gblk + j) & 1, wd, kSiteMmaP) &&
                                        (j > 0 || k == 0 || mbar_wait(bar_of, (k - 1) & 1, wd, kSiteMmaOF)));
                    if (!ok) break;
                    tc_fence_after();
                    issue_pv(tO, tS, vlo0 + sv * kSlot, j > 0);
                    mma_commit_warp(bar_o);
                    mma_commit_warp(bar_kve + 8 * sv);
                    if (j + 1 < nb) {
                        const int gk = g + 2 * j + 2, sk = gk % kStages;  // K_(j+1)
                        ok = __all_sync(0xffffffffu, mbar_wait(bar_kvf + 8 * sk, (gk / kStages) & 1, wd, kSiteMmaKV));
                        if (!ok) break;
                        tc_fence_after();
                        issue_s(tS, qlo, klo0 + sk * kSlot);  // over P(j), which P V(j) has read
                        mma_commit_warp(bar_s);
                        mma_commit_warp(bar_kve + 8 * sk);
                        if (j + 2 == nb) mma_commit_warp(bar_qe);  // the item's last S
                    }
                }
                if (!ok) break;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_id + 8 * b);  // done with the list
            g += 2 * nb;
            gblk += nb;
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------- softmax --
        const int r = threadIdx.x & 127;
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + lane_off + kTmS, tO = tmem + lane_off + kTmO;
        const float sl2 = p.scale_log2;
        bool ok = true;
        int gblk = 0;
        for (int k = 0; ok; ++k) {
            const int idx = item_of(k, c, G, p.items);
            if (idx < 0) break;
            const int qt = p.n_q - 1 - idx / p.BH, bh = idx % p.BH;
            const int b = k & 1;
            const int q_start = qt * kBM, row = q_start + r;
            if (!__all_sync(0xffffffffu, mbar_wait(bar_ir + 8 * b, (k >> 1) & 1, wd, kSiteItem))) break;
            const int nb = sh.n_blk[b];
            float m_used = -INFINITY;
            float l = 0.f, l_mma = 0.f;
            int j = -1;  // key block
            for (int jj = 0; jj < nb; ++jj) {
                j = next_block(sh.use[b], j + 1, n_kv);
                const int gb = gblk + jj;
                if (!__all_sync(0xffffffffu, mbar_wait(bar_s, gb & 1, wd, kSiteSoftS))) {
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
                const int kbase = j * kBN;
                if ((CAUSAL && kbase + kBN - 1 > q_start) || (kbase + kBN > N)) {
                    const int last = CAUSAL ? min(row, N - 1) : N - 1;  // last visible key
#pragma unroll
                    for (int cc = 0; cc < 128; ++cc)
                        if (kbase + cc > last) s[cc >> 5][cc & 31] = f2u(-INFINITY);
                }
                float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
                for (int cc = 0; cc < 32; cc += 2) {
                    mx0 = fmax3(mx0, u2f(s[0][cc]), u2f(s[0][cc + 1]));
                    mx1 = fmax3(mx1, u2f(s[1][cc]), u2f(s[1][cc + 1]));
                    mx2 = fmax3(mx2, u2f(s[2][cc]), u2f(s[2][cc + 1]));
                    mx3 = fmax3(mx3, u2f(s[3][cc]), u2f(s[3][cc + 1]));
                }
                const float m_cand = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * sl2;
                const bool grow = m_cand > m_used + kRescaleThreshold;
                float alpha = 1.f;
                if (grow) {
                    alpha = ex2(m_used - m_cand);  // 0 on the item's first block (m_used = -inf)
                    m_used = m_cand;
                }
                // the row sums' rescale and update are rounded separately (no FMA
                // contraction), as in the dense kernel
                l = __fmul_rn(l, alpha);
                l_mma = __fmul_rn(l_mma, alpha);
                const float neg_m = (m_used == -INFINITY) ? 0.f : -m_used;
                // l_mma sums the bf16 P values the P V MMA consumes (it normalises
                // O), l the fp32 values (it gives LSE); paired fp32 adds
                const uint64_t c2 = f2_pack(sl2, sl2), nm2 = f2_pack(neg_m, neg_m);
                uint64_t ls2 = 0;
                float lr0 = 0.f, lr1 = 0.f;  // the bf16 sums, added straight from the packed pairs
#pragma unroll
                for (int h = 0; h < 64 / kPC; ++h) {
                    uint32_t pk[kPC];
#pragma unroll
                    for (int i = 0; i < kPC; ++i) {
                        const int cc = h * 2 * kPC + 2 * i;
                        const float2 x = f2_unpack(ffma2(
                            f2_pack(u2f(s[cc >> 5][cc & 31]), u2f(s[cc >> 5][(cc & 31) + 1])), c2, nm2));
                        const float p0 = ex2(x.x), p1 = ex2(x.y);
                        pk[i] = pack_bf16(p0, p1);
                        ls2 = fadd2(ls2, f2_pack(p0, p1));
                        add_bf16x2_f32(pk[i], lr0, lr1);
                    }
                    tmem_st16(tS + h * 16, pk);
                }
                const float2 a2 = f2_unpack(ls2);
                l = __fadd_rn(l, __fadd_rn(a2.x, a2.y));
                l_mma = __fadd_rn(l_mma, __fadd_rn(lr0, lr1));
                if (jj > 0 && __any_sync(0xffffffffu, grow)) {
                    // rescale this warp's rows of O once the previous P V has landed (after
                    // P is written, so the S registers are dead; this P V waits for p_ready)
                    if (!__all_sync(0xffffffffu, mbar_wait(bar_o, (gb - 1) & 1, wd, kSiteSoftO))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int c0 = 0; c0 < kD; c0 += 32) {
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
                mbar_arrive(bar_p);
            }
            if (!ok) break;
            mbar_arrive(bar_id + 8 * b);  // done with the list
            // ------------------------------------------------------- epilogue --
            // O / l_mma -> bf16 straight to global memory, LSE per row; a tile that
            // visits no key block writes the empty sum (O = 0, LSE = -inf)
            const int64_t bh_row = static_cast<int64_t>(bh) * N + row;
            if (nb > 0) {
                if (!__all_sync(0xffffffffu, mbar_wait(bar_o, (gblk + nb - 1) & 1, wd, kSiteEpi))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t o[4][32];
#pragma unroll
                for (int x = 0; x < 4; ++x) tmem_ld32(tO + 32 * x, o[x]);
#pragma unroll
                for (int x = 0; x < 4; ++x) tmem_ld_wait(o[x]);
                tc_fence_before();
                mbar_arrive(bar_of);  // O's columns may take the next item's first P V
                if (row < N) {
                    const float inv_l = 1.f / l_mma;
                    uint4* dst = reinterpret_cast<uint4*>(p.O + bh_row * kD);
#pragma unroll
                    for (int x = 0; x < 4; ++x)
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            uint4 v;
                            v.x = pack_bf16(u2f(o[x][8 * q + 0]) * inv_l, u2f(o[x][8 * q + 1]) * inv_l);
                            v.y = pack_bf16(u2f(o[x][8 * q + 2]) * inv_l, u2f(o[x][8 * q + 3]) * inv_l);
                            v.z = pack_bf16(u2f(o[x][8 * q + 4]) * inv_l, u2f(o[x][8 * q + 5]) * inv_l);
                            v.w = pack_bf16(u2f(o[x][8 * q + 6]) * inv_l, u2f(o[x][8 * q + 7]) * inv_l);
                            dst[4 * x + q] = v;
                        }
                    p.LSE[bh_row] = (m_used + __log2f(l)) * kLn2;
                }
            } else {
                mbar_arrive(bar_of);
                if (row < N) {
                    uint4* dst = reinterpret_cast<uint4*>(p.O + bh_row * kD);
#pragma unroll
                    for (int x = 0; x < 16; ++x) dst[x] = make_uint4(0u, 0u, 0u, 0u);
                    p.LSE[bh_row] = -INFINITY;
                }
            }
            gblk += nb;
        }
    }

    // -------------------------------------------------------------- teardown --
    if (sh.abort_flag) drain_after_abort();
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmCols);
    }
}

template <bool CAUSAL>
cudaError_t launch_sparse_t(const FwdArgs& a, cudaStream_t stream) {
    CUtensorMap tq, tk, tv;
    const auto BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    if (!make_tile_map(&tq, a.Q, BF, 2, kD, a.N, a.BH, 64, kBM) ||
        !make_tile_map(&tk, a.K, BF, 2, kD, a.N, a.BH, 64, kBN) ||
        !make_tile_map(&tv, a.V, BF, 2, kD, a.N, a.BH, 64, kBN))
        return cudaErrorInvalidValue;
    constexpr auto kern = &fa_fwd_sparse_kernel<CAUSAL>;
    cudaError_t e = set_max_dyn_smem_once<kern>(kDynSmem);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return cudaGetLastError();
    SparseParams p;
    p.O = static_cast<__nv_bfloat16*>(a.O);
    p.LSE = a.LSE;
    p.blocks = a.blocks;
    p.blocks_head_stride = a.blocks_head_stride;
    p.N = a.N;
    p.BH = a.BH;
    p.n_q = (a.N + kBM - 1) / kBM;
    p.n_kv = (a.N + kBN - 1) / kBN;
    const long long items = static_cast<long long>(a.BH) * p.n_q;
    if (items > (1ll << 30) || p.n_kv > kMaxMaskBlocks) return cudaErrorInvalidValue;
    p.items = static_cast<int>(items);
    p.scale_log2 = a.tau * kLog2e;
    p.err = a.err;
    p.wait_limit_ns = a.wait_limit_ns;
    const int grid = static_cast<int>(std::min<long long>(items, 2ll * sms));
    if (a.ev_start) cudaEventRecord(a.ev_start, stream);
    fa_fwd_sparse_kernel<CAUSAL><<<grid, kThreads, kDynSmem, stream>>>(tq, tk, tv, p);
    e = cudaGetLastError();
    if (e == cudaSuccess && a.ev_stop) e = cudaEventRecord(a.ev_stop, stream);
    return e;
}

}  // namespace

cudaError_t launch_fwd_sparse(const FwdArgs& a, cudaStream_t stream) {
    return a.causal ? launch_sparse_t<true>(a, stream) : launch_sparse_t<false>(a, stream);
}

}  // namespace fa
