// Persistent forward for short d = 64 problems (N <= 2048, GPT-2-sized).
//
// The method is the forward of fa_fwd.cu ("Atencao eficiente - FlashAttention,
// sparse e hibrida", "Insight 1 - Tiling" and "Insight 2 - Online softmax";
// tonho.wtf "flash attention", "como funciona"): one 128-row query tile walks
// the key blocks with the online softmax, O / l and LSE = m + ln l are
// written at the end.  What changes is the scheduling.  On these shapes a
// query tile has only 1 to 16 key blocks, and a CTA that owns one tile spends
// about 40% of its life waiting for its first Q and K tiles and storing O
// (measured: ~2 us to the first S, ~1.1 us epilogue, ~5.4 us of main loop).
// Here each CTA (two per SM) walks a list of query tiles and keeps its barriers
// and tensor memory: Q is double-buffered, so the next tile's Q and first K/V
// blocks load while the current tile runs, and the K/V ring streams from one
// tile into the next without a gap.
//
// Work item i of BH * n_q is query tile (n_q - 1 - i / BH) of head (i % BH):
// the heaviest causal tiles first.  CTA c of G takes items in "snake" order,
// c, 2G - 1 - c, 2G + c, 4G - 1 - c, ..., which balances heavy and light tiles
// without a shared counter.
//
// Per tile the pipeline is the one-tile d = 64 forward of fa_fwd.cu: P has
// its own tensor-memory columns, so S of block j + 1 is issued as soon as the
// softmax has read S of block j; the producer loads K0 K1 V0 K2 V1 ... in that
// order; O is rescaled only when a row's max grows by more than 2^8.
#include <cuda_bf16.h>

#include <cmath>

#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int kBM = 128, kBN = 128, kD = 64;
constexpr int kThreads = 192;                 // softmax warps 0-3, producer 4, MMA 5
constexpr int kProducerWarp = 4, kMmaWarp = 5;
constexpr int kStages = 4;                    // K/V ring slots
constexpr int kTile = kBM * kD * 2;           // one [128 x 64] bf16 tile = one TMA box
constexpr int kQ = 0;                         // Q buffers 0 and 1 (O is staged over them)
constexpr int kRing = 2 * kTile;
constexpr int kBytes = kRing + kStages * kTile;
constexpr int kDynSmem = kBytes + 1024;       // + alignment slack
constexpr uint32_t kTmS = 0, kTmO = 128, kTmP = 192, kTmCols = 256;
constexpr int kPC = 32;                       // P packed columns per tensor-memory store
constexpr float kLn2 = 0.69314718055994531f;
constexpr float kLog2e = 1.44269504088896341f;
constexpr float kRescaleThreshold = 8.0f;     // log2 units: P stays <= 2^8

struct ShortParams {
    float* LSE;
    int N, BH, n_q, items;
    float scale_log2;
    unsigned int* err;
    unsigned long long wait_limit_ns;
};

struct ShortShared {
    uint64_t q_full[2];
    uint64_t q_free[2];   // the O staged over Q buffer b has been stored
    uint64_t kv_full[kStages];
    uint64_t kv_empty[kStages];
    uint64_t s_full, s_free, p_ready, o_done, o_free;
    uint32_t tmem_base;
    int abort_flag;
};

enum : uint32_t {
    kSiteQFree = 41, kSiteKvEmpty = 42, kSiteMmaQ = 43, kSiteMmaKV = 44, kSiteMmaSF = 45,
    kSiteMmaP = 46, kSiteMmaOF = 47, kSiteSoftS = 48, kSiteSoftO = 49, kSiteEpi = 50
};

__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }
__device__ __forceinline__ uint32_t f2u(float x) { return __float_as_uint(x); }

constexpr uint32_t kDescHi = sw128_desc_hi(1024);

// The k-th work item of this CTA (snake order), or -1 past the end.
__device__ __forceinline__ int item_of(int k, int c, int G, int items) {
    const int idx = k * G + ((k & 1) ? G - 1 - c : c);
    return idx < items ? idx : -1;
}

template <bool CAUSAL>
__device__ __forceinline__ int blocks_of(int qt, int n_kv) {
    return CAUSAL ? min(n_kv, qt + 1) : n_kv;
}

template <bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 2)
fa_fwd_short_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                    const ShortParams p) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ ShortShared sh;
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t pad = ((raw + 1023u) & ~1023u) - raw;
    uint8_t* smem = smem_raw + pad;
    const uint32_t sbase = raw + pad;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int N = p.N;
    const int n_kv = (N + kBN - 1) / kBN;
    const int G = gridDim.x, c = blockIdx.x;

    const uint32_t bar_qf = smem_addr(&sh.q_full[0]);
    const uint32_t bar_qe = smem_addr(&sh.q_free[0]);
    const uint32_t bar_kvf = smem_addr(&sh.kv_full[0]);
    const uint32_t bar_kve = smem_addr(&sh.kv_empty[0]);
    const uint32_t bar_s = smem_addr(&sh.s_full);
    const uint32_t bar_sf = smem_addr(&sh.s_free);
    const uint32_t bar_p = smem_addr(&sh.p_ready);
    const uint32_t bar_o = smem_addr(&sh.o_done);
    const uint32_t bar_of = smem_addr(&sh.o_free);

    if (threadIdx.x == 0) {
        sh.abort_flag = 0;
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar_qf + 8 * b, 1);
            mbar_init(bar_qe + 8 * b, 1);
        }
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar_kvf + 8 * s, 1);
            mbar_init(bar_kve + 8 * s, 1);
        }
        mbar_init(bar_s, 1);
        mbar_init(bar_sf, 128);
        mbar_init(bar_p, 128);
        mbar_init(bar_o, 1);
        mbar_init(bar_of, 128);
        mbar_init_fence();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_addr(&sh.tmem_base), kTmCols);
        tmem_relinquish();
    }
    if (warp == kProducerWarp && lane == 0) {
        tma_prefetch_map(&tmQ);
        tma_prefetch_map(&tmK);
        tma_prefetch_map(&tmV);
        tma_prefetch_map(&tmO);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    griddep_launch_dependents();
    const uint32_t tmem = sh.tmem_base;
    const Watchdog wd{p.err, &sh.abort_flag, p.wait_limit_ns};

    if (warp == kProducerWarp) {
        // ------------------------------------------------------------ producer --
        if (lane == 0) {
            int lbase = 0;  // loads issued for earlier items
            for (int k = 0;; ++k) {
                const int idx = item_of(k, c, G, p.items);
                if (idx < 0) break;
                const int qt = p.n_q - 1 - idx / p.BH, bh = idx % p.BH;
                const int nb = blocks_of<CAUSAL>(qt, n_kv);
                const int qb = k & 1;
                // Q buffer qb held item k - 2's staged O until its store read it
                if (k >= 2 && !mbar_wait(bar_qe + 8 * qb, ((k >> 1) - 1) & 1, wd, kSiteQFree)) break;
                mbar_arrive_expect_tx(bar_qf + 8 * qb, kTile);
                tma_load_3d(sbase + kQ + qb * kTile, &tmQ, bar_qf + 8 * qb, 0, qt * kBM, bh);
                bool ok = true;
                for (int ld = 0; ld < 2 * nb; ++ld) {
                    const int g = lbase + ld, slot = g % kStages;
                    if (g >= kStages && !mbar_wait(bar_kve + 8 * slot, ((g / kStages) - 1) & 1, wd, kSiteKvEmpty)) {
                        ok = false;
                        break;
                    }
                    // the MMA warp's order: K0 K1 V0 K2 V1 ... K(nb-1) V(nb-2) V(nb-1)
                    const bool is_k = ld == 0 || ((ld & 1) && ld < 2 * nb - 1);
                    const int blk = is_k ? (ld + 1) / 2 : (ld == 2 * nb - 1 ? nb - 1 : ld / 2 - 1);
                    mbar_arrive_expect_tx(bar_kvf + 8 * slot, kTile);
                    tma_load_3d(sbase + kRing + slot * kTile, is_k ? &tmK : &tmV, bar_kvf + 8 * slot, 0,
                                blk * kBN, bh);
                }
                if (!ok) break;
                lbase += 2 * nb;
            }
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        // ----------------------------------------------------------------- MMA --
        const uint32_t tS = tmem + kTmS, tO = tmem + kTmO, tP = tmem + kTmP;
        const uint32_t klo0 = sw128_desc_lo(sbase + kRing, 16);          // K: K-major
        const uint32_t vlo0 = sw128_desc_lo(sbase + kRing, 128 * 128);   // V: MN-major
        constexpr uint32_t kSlot = kTile >> 4;
        constexpr uint32_t id_s = idesc_bf16(128, 128, false, false);
        constexpr uint32_t id_pv = idesc_bf16(128, kD, false, true);
        int lbase = 0, gblk = 0;
        bool ok = true;
        for (int k = 0; ok; ++k) {
            const int idx = item_of(k, c, G, p.items);
            if (idx < 0) break;
            const int qt = p.n_q - 1 - idx / p.BH;
            const int nb = blocks_of<CAUSAL>(qt, n_kv);
            const int qb = k & 1;
            const uint32_t qlo = sw128_desc_lo(sbase + kQ + qb * kTile, 16);
            if (!__all_sync(0xffffffffu, mbar_wait(bar_qf + 8 * qb, (k >> 1) & 1, wd, kSiteMmaQ))) break;
            for (int j = 0; j <= nb; ++j) {
                if (j < nb) {
                    const int g = lbase + (j == 0 ? 0 : 2 * j - 1), sk = g % kStages;  // K_j
                    // S's columns are free once the softmax has read the previous S
                    ok = __all_sync(0xffffffffu,
                                    mbar_wait(bar_kvf + 8 * sk, (g / kStages) & 1, wd, kSiteMmaKV) &&
                                        (gblk + j == 0 ||
                                         mbar_wait(bar_sf, (gblk + j - 1) & 1, wd, kSiteMmaSF)));
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < kD / 16; ++kk) {
                        const uint32_t off = (kk * 32) >> 4;
                        if (kk == 0) mma_ss_warp<0>(tS, qlo + off, klo0 + sk * kSlot + off, kDescHi, id_s);
                        else mma_ss_warp<1>(tS, qlo + off, klo0 + sk * kSlot + off, kDescHi, id_s);
                    }
                    mma_commit_warp(bar_s);
                    mma_commit_warp(bar_kve + 8 * sk);
                }
                if (j > 0) {
                    const int g = lbase + min(2 * j, 2 * nb - 1), sv = g % kStages;  // V_(j-1)
                    // the first P V of a tile overwrites O: the previous tile's
                    // epilogue must have read it out
                    ok = __all_sync(0xffffffffu,
                                    mbar_wait(bar_kvf + 8 * sv, (g / kStages) & 1, wd, kSiteMmaKV) &&
                                        mbar_wait(bar_p, (gblk + j - 1) & 1, wd, kSiteMmaP) &&
                                        (j > 1 || k == 0 || mbar_wait(bar_of, (k - 1) & 1, wd, kSiteMmaOF)));
                    if (!ok) break;
                    tc_fence_after();
                    if (j > 1) mma_ts_warp<1>(tO, tP, vlo0 + sv * kSlot, kDescHi, id_pv);
                    else mma_ts_warp<0>(tO, tP, vlo0 + sv * kSlot, kDescHi, id_pv);
#pragma unroll
                    for (int kk = 1; kk < kBN / 16; ++kk)
                        mma_ts_warp<1>(tO, tP + kk * 8, vlo0 + sv * kSlot + ((kk * 2048) >> 4), kDescHi, id_pv);
                    mma_commit_warp(bar_o);
                    mma_commit_warp(bar_kve + 8 * sv);
                }
            }
            lbase += 2 * nb;
            gblk += nb;
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------- softmax --
        const int r = threadIdx.x & 127;
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + lane_off + kTmS, tO = tmem + lane_off + kTmO;
        const uint32_t tP = tmem + lane_off + kTmP;
        const float sl2 = p.scale_log2;
        bool ok = true;
        int gblk = 0;
        for (int k = 0; ok; ++k) {
            const int idx = item_of(k, c, G, p.items);
            if (idx < 0) break;
            const int qt = p.n_q - 1 - idx / p.BH, bh = idx % p.BH;
            const int nb = blocks_of<CAUSAL>(qt, n_kv);
            const int qb = k & 1;
            const int q_start = qt * kBM, row = q_start + r;
            float m_used = -INFINITY;
            float l = 0.f, l_mma = 0.f;
            for (int jj = 0; jj < nb; ++jj) {
                const int g = gblk + jj;
                if (!__all_sync(0xffffffffu, mbar_wait(bar_s, g & 1, wd, kSiteSoftS))) {
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
                tc_fence_before();
                mbar_arrive(bar_sf);  // S's columns may take the next block's scores now

                const int kbase = jj * kBN;
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
                    alpha = ex2(m_used - m_cand);  // 0 on the tile's first block (m_used = -inf)
                    m_used = m_cand;
                }
                // the row sums' rescale and update are rounded separately (no FMA
                // contraction), so every forward kernel gives the same LSE bits
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
                    if (h == 0 && g > 0) {
                        // P's columns are free once the previous P V (of this or the
                        // previous tile) has read them
                        if (!__all_sync(0xffffffffu, mbar_wait(bar_o, (g - 1) & 1, wd, kSiteSoftO))) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                    }
                    tmem_st32(tP + h * 32, pk);
                }
                if (!ok) break;
                const float2 a2 = f2_unpack(ls2);
                l = __fadd_rn(l, __fadd_rn(a2.x, a2.y));
                l_mma = __fadd_rn(l_mma, __fadd_rn(lr0, lr1));
                if (jj > 0 && __any_sync(0xffffffffu, grow)) {
                    // rescale this warp's rows of O once the previous P V has landed
                    if (!__all_sync(0xffffffffu, mbar_wait(bar_o, (g - 1) & 1, wd, kSiteSoftO))) {
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
            // ------------------------------------------------------- epilogue --
            // O / l_mma -> bf16, staged over this tile's Q buffer (every S MMA of the
            // tile has read Q by now), one TMA store; LSE per row
            bool epi = ok;
            if (epi) epi = __all_sync(0xffffffffu, mbar_wait(bar_o, (gblk + nb - 1) & 1, wd, kSiteEpi));
            if (epi) {
                tc_fence_after();
                uint32_t o[2][32];
                tmem_ld32(tO, o[0]);
                tmem_ld32(tO + 32, o[1]);
                tmem_ld_wait(o[0]);
                tmem_ld_wait(o[1]);
                tc_fence_before();
                mbar_arrive(bar_of);  // O's columns may take the next tile's first P V
                const float inv_l = 1.f / l_mma;
                uint8_t* stage = smem + kQ + qb * kTile;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int chunk = 4 * h + q;
                        uint4 v;
                        v.x = pack_bf16(u2f(o[h][8 * q + 0]) * inv_l, u2f(o[h][8 * q + 1]) * inv_l);
                        v.y = pack_bf16(u2f(o[h][8 * q + 2]) * inv_l, u2f(o[h][8 * q + 3]) * inv_l);
                        v.z = pack_bf16(u2f(o[h][8 * q + 4]) * inv_l, u2f(o[h][8 * q + 5]) * inv_l);
                        v.w = pack_bf16(u2f(o[h][8 * q + 6]) * inv_l, u2f(o[h][8 * q + 7]) * inv_l);
                        *reinterpret_cast<uint4*>(stage + r * 128 + ((chunk ^ (r & 7)) << 4)) = v;
                    }
                }
                fence_async_shared();
                if (row < N) p.LSE[static_cast<int64_t>(bh) * N + row] = (m_used + __log2f(l)) * kLn2;
            }
            // all four warps reach this barrier once per tile, even after a failed
            // wait, and agree whether every one of them staged its rows
            if (named_bar_or(1, 128, !epi)) {
                ok = false;
                break;
            }
            if (r == 0) {
                tma_store_3d(&tmO, sbase + kQ + qb * kTile, 0, q_start, bh);
                bulk_commit();
                bulk_wait_read<0>();
                mbar_arrive(bar_qe + 8 * qb);  // the Q buffer may take item k + 2's Q
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
cudaError_t launch_short_t(const FwdArgs& a, cudaStream_t stream) {
    CUtensorMap tq, tk, tv, to;
    const auto BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    if (!make_tile_map(&tq, a.Q, BF, 2, kD, a.N, a.BH, 64, kBM) ||
        !make_tile_map(&tk, a.K, BF, 2, kD, a.N, a.BH, 64, kBN) ||
        !make_tile_map(&tv, a.V, BF, 2, kD, a.N, a.BH, 64, kBN) ||
        !make_tile_map(&to, a.O, BF, 2, kD, a.N, a.BH, 64, kBM))
        return cudaErrorInvalidValue;
    constexpr auto kern = &fa_fwd_short_kernel<CAUSAL>;
    cudaError_t e = set_max_dyn_smem_once<kern>(kDynSmem);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return cudaGetLastError();
    ShortParams p;
    p.LSE = a.LSE;
    p.N = a.N;
    p.BH = a.BH;
    p.n_q = (a.N + kBM - 1) / kBM;
    const long long items = static_cast<long long>(a.BH) * p.n_q;
    if (items > (1ll << 30)) return cudaErrorInvalidValue;
    p.items = static_cast<int>(items);
    p.scale_log2 = a.tau * kLog2e;
    p.err = a.err;
    p.wait_limit_ns = a.wait_limit_ns;
    const int grid = static_cast<int>(std::min<long long>(items, 2ll * sms));
    if (a.ev_start) cudaEventRecord(a.ev_start, stream);
    fa_fwd_short_kernel<CAUSAL><<<grid, kThreads, kDynSmem, stream>>>(tq, tk, tv, to, p);
    e = cudaGetLastError();
    if (e == cudaSuccess && a.ev_stop) e = cudaEventRecord(a.ev_stop, stream);
    return e;
}

}  // namespace

cudaError_t launch_fwd_short(const FwdArgs& a, cudaStream_t stream) {
    return a.causal ? launch_short_t<true>(a, stream) : launch_short_t<false>(a, stream);
}

}  // namespace fa
