// FP8 (e4m3) forward of exact IO-aware attention for sm_103a, d = 128.
//
// Method: the same tiled forward with online softmax as fa_fwd.cu ("Atencao
// eficiente - FlashAttention, sparse e hibrida", "Insight 1 - Tiling",
// "Insight 2 - Online softmax"), with the 8-bit inputs that the same page's
// FlashAttention-4 note credits to FlashAttention-3 ("FP8 para Hopper").
// Q, K, V arrive as e4m3 with one scale per tensor (value = byte * scale), so
//   S = tau sq sk (Q8 K8^T),   O = sv (P8 V8) / l,
// where P8 is the softmax numerator rounded to e4m3 for the second product.
//
// GB300 design (the bf16 kernel's pipeline, on kind::f8f6f4):
//   - both products run on tcgen05.mma kind::f8f6f4 (K = 32 per instruction,
//     twice the bf16 rate); Q, K and V tiles are [128 x 128 bytes], one
//     128-byte-swizzled TMA box each, so a K or V slot is 16 KB and the ring
//     holds 8 of them;
//   - an MMA takes both operands of one type, so P goes back to tensor memory
//     as e4m3, not bf16: each softmax thread converts its row of P
//     (cvt.rn.satfinite.e4m3x2), packs four keys per 32-bit column and writes
//     the 32 columns over its tile's S, where the P V product reads it as the
//     A operand (A from tensor memory, V from shared memory).  A version with
//     P staged in shared memory ran at the same speed; this one moves 64 KB
//     less through shared memory per key block and needs no proxy fences;
//   - P = 2^(x - m + 6) with the row max m rescaled only when it grows by more
//     than 2^2: P stays <= 2^8 (e4m3 saturates at 448) and the smallest
//     weights sit 2^6 further above e4m3's subnormal range than with P <= 1;
//     l sums the same (unrounded) P in fp32, so the shift cancels in O / l and
//     LSE = m - 6 + log2 l (in log2 units, converted at the store);
//   - warps 0-3 / 4-7: softmax of query tile 0 / 1; warp 8: TMA; warp 9: MMA.
#include <cuda_bf16.h>

#include <cmath>

#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int kBM = 128;  // query rows per tile
constexpr int kBN = 128;  // keys per block
constexpr int kD = 128;   // head dimension (bytes per fp8 row)
constexpr int kThreads = 320;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kTile = kBM * kD;  // one fp8 [128 x 128] tile
constexpr int kStages = 8;
// shared memory: [Q0][pad][Q1][pad] (each Q tile followed by 16 KB, so the bf16
// O tile of 32 KB can be staged over it at the end), then the ring of K and V
// slots
constexpr int kQ0 = 0, kQ1 = 2 * kTile, kRing = 4 * kTile;
constexpr int kBytes = kRing + kStages * kTile;
constexpr int kDynSmem = kBytes + 1024;  // + alignment slack
constexpr int kOutBox = 128 * 128;       // one bf16 [128 rows x 64 cols] TMA box of O
constexpr uint32_t kTmemS0 = 0, kTmemS1 = 128, kTmemO0 = 256, kTmemO1 = 384;
constexpr float kShift = 6.0f;    // log2 of the factor P carries
constexpr float kRescale = 2.0f;  // log2 growth of the max that triggers a rescale
constexpr float kLn2 = 0.69314718055994531f;
constexpr float kLog2e = 1.44269504088896341f;

struct Fp8Params {
    float* LSE;
    int N;
    int n_pairs;
    float scale_log2;  // tau * sq * sk * log2(e)
    float v_scale;     // sv
    unsigned int* err;
    unsigned long long wait_limit_ns;
};

struct Fp8Shared {
    uint64_t q_full;
    uint64_t kv_full[kStages];
    uint64_t kv_empty[kStages];
    uint64_t s_full[2];
    uint64_t p_ready[2];
    uint64_t o_done[2];
    uint32_t tmem_base;
    int abort_flag;
};

enum : uint32_t {
    kSiteProdEmpty = 51, kSiteMmaQ = 52, kSiteMmaKV = 53, kSiteMmaP = 54,
    kSiteSoftS = 55, kSiteSoftO = 56, kSiteEpi = 57
};

__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }
__device__ __forceinline__ uint32_t f2u(float x) { return __float_as_uint(x); }

constexpr uint32_t kDescHi = sw128_desc_hi(1024);  // 8-row groups 1 KB apart

// S = Q K^T: both K-major [128 rows x 128 bytes]; four K-steps of 32.
__device__ __forceinline__ void issue_s(uint32_t tmem_d, uint32_t q_lo, uint32_t k_lo) {
    constexpr uint32_t id = idesc_e4m3(128, 128, false, false);
    mma_ss_f8_warp<0>(tmem_d, q_lo, k_lo, kDescHi, id);
#pragma unroll
    for (int k = 1; k < kD / 32; ++k) mma_ss_f8_warp<1>(tmem_d, q_lo + 2 * k, k_lo + 2 * k, kDescHi, id);
}

// O += P V: P [128 rows x 128 keys] e4m3 in tensor memory (four keys per
// column), V MN-major [128 keys x 128 dims]; a K-step of 32 keys is 8 columns
// of P and 32 rows of V (4 KB).
__device__ __forceinline__ void issue_pv(uint32_t tmem_o, uint32_t tmem_p, uint32_t v_lo,
                                         bool accumulate) {
    constexpr uint32_t id = idesc_e4m3(128, 128, false, true);
    if (accumulate) mma_ts_f8_warp<1>(tmem_o, tmem_p, v_lo, kDescHi, id);
    else mma_ts_f8_warp<0>(tmem_o, tmem_p, v_lo, kDescHi, id);
#pragma unroll
    for (int k = 1; k < kBN / 32; ++k)
        mma_ts_f8_warp<1>(tmem_o, tmem_p + 8 * k, v_lo + ((k * 32 * 128) >> 4), kDescHi, id);
}

template <bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
fa_fwd_fp8_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                  const Fp8Params p) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ Fp8Shared sh;
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t pad = ((raw + 1023u) & ~1023u) - raw;
    uint8_t* smem = smem_raw + pad;
    const uint32_t sbase = raw + pad;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int bh = blockIdx.x;
    const int pair = p.n_pairs - 1 - static_cast<int>(blockIdx.y);  // heaviest pairs first
    const int N = p.N;
    const int n_kv = (N + kBN - 1) / kBN;
    const int q_start0 = pair * 2 * kBM;
    const int q_start1 = q_start0 + kBM;
    const int n_blk0 = CAUSAL ? min(n_kv, q_start0 / kBN + 1) : n_kv;
    const int n_blk1 = q_start1 < N ? (CAUSAL ? min(n_kv, q_start1 / kBN + 1) : n_kv) : 0;
    const int nb = max(n_blk0, n_blk1);

    const uint32_t bar_q = smem_addr(&sh.q_full);
    const uint32_t bar_kv_full = smem_addr(&sh.kv_full[0]);
    const uint32_t bar_kv_empty = smem_addr(&sh.kv_empty[0]);
    const uint32_t bar_s = smem_addr(&sh.s_full[0]);
    const uint32_t bar_p = smem_addr(&sh.p_ready[0]);
    const uint32_t bar_o = smem_addr(&sh.o_done[0]);

    if (threadIdx.x == 0) {
        sh.abort_flag = 0;
        mbar_init(bar_q, 1);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar_kv_full + 8 * s, 1);
            mbar_init(bar_kv_empty + 8 * s, 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(bar_s + 8 * t, 1);
            mbar_init(bar_p + 8 * t, 128);
            mbar_init(bar_o + 8 * t, 1);
        }
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
        tma_prefetch_map(&tmO);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sh.tmem_base;
    const Watchdog wd{p.err, &sh.abort_flag, p.wait_limit_ns};

    if (warp == kProducerWarp) {
        // ----------------------------------------------------------- producer --
        if (lane == 0) {
            mbar_arrive_expect_tx(bar_q, kTile * (1 + (n_blk1 > 0)));
            tma_load_3d(sbase + kQ0, &tmQ, bar_q, 0, q_start0, bh);
            if (n_blk1 > 0) tma_load_3d(sbase + kQ1, &tmQ, bar_q, 0, q_start1, bh);
            for (int ld = 0; ld < 2 * nb; ++ld) {
                const int slot = ld % kStages;
                if (ld >= kStages &&
                    !mbar_wait(bar_kv_empty + 8 * slot, ((ld / kStages) - 1) & 1, wd, kSiteProdEmpty))
                    break;
                mbar_arrive_expect_tx(bar_kv_full + 8 * slot, kTile);
                tma_load_3d(sbase + kRing + slot * kTile, (ld & 1) ? &tmV : &tmK,
                            bar_kv_full + 8 * slot, 0, (ld >> 1) * kBN, bh);
            }
        }
    } else if (warp == kMmaWarp) {
        // ---------------------------------------------------------------- MMA --
        const uint32_t tS[2] = {tmem + kTmemS0, tmem + kTmemS1};
        const uint32_t tO[2] = {tmem + kTmemO0, tmem + kTmemO1};
        const uint32_t qlo[2] = {sw128_desc_lo(sbase + kQ0, 16), sw128_desc_lo(sbase + kQ1, 16)};
        const uint32_t klo0 = sw128_desc_lo(sbase + kRing, 16);         // K: K-major
        const uint32_t vlo0 = sw128_desc_lo(sbase + kRing, 128 * 128);  // V: MN-major
        constexpr uint32_t kSlot = kTile >> 4;
        const int nblk[2] = {n_blk0, n_blk1};
        bool ok = __all_sync(0xffffffffu, mbar_wait(bar_q, 0, wd, kSiteMmaQ) &&
                                              mbar_wait(bar_kv_full, 0, wd, kSiteMmaKV));
        if (ok) {
            tc_fence_after();
            for (int t = 0; t < 2; ++t) {
                if (nblk[t] > 0) {
                    issue_s(tS[t], qlo[t], klo0);
                    mma_commit_warp(bar_s + 8 * t);
                }
            }
            mma_commit_warp(bar_kv_empty);
        }
        for (int j = 0; ok && j < nb; ++j) {
            const int lv = 2 * j + 1, lk = 2 * j + 2;
            const int sv = lv % kStages, sk = lk % kStages;
            if (!__all_sync(0xffffffffu,
                            mbar_wait(bar_kv_full + 8 * sv, (lv / kStages) & 1, wd, kSiteMmaKV))) {
                ok = false;
                break;
            }
            tc_fence_after();
            bool k_ready = false;
            for (int t = 0; t < 2 && ok; ++t) {
                if (j >= nblk[t]) continue;
                if (!__all_sync(0xffffffffu, mbar_wait(bar_p + 8 * t, j & 1, wd, kSiteMmaP))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                issue_pv(tO[t], tS[t], vlo0 + sv * kSlot, j > 0);
                mma_commit_warp(bar_o + 8 * t);
                if (j + 1 < nblk[t]) {
                    if (!k_ready) {
                        if (!__all_sync(0xffffffffu,
                                        mbar_wait(bar_kv_full + 8 * sk, (lk / kStages) & 1, wd,
                                                  kSiteMmaKV))) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        k_ready = true;
                    }
                    issue_s(tS[t], qlo[t], klo0 + sk * kSlot);
                    mma_commit_warp(bar_s + 8 * t);
                }
            }
            if (!ok) break;
            mma_commit_warp(bar_kv_empty + 8 * sv);
            if (k_ready) mma_commit_warp(bar_kv_empty + 8 * sk);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax --
        const int t = warp >> 2;
        const int r = threadIdx.x & 127;
        const int q_start = t ? q_start1 : q_start0;
        const int nbt = t ? n_blk1 : n_blk0;
        const int row = q_start + r;
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + lane_off + (t ? kTmemS1 : kTmemS0);
        const uint32_t tO = tmem + lane_off + (t ? kTmemO1 : kTmemO0);
        const uint32_t my_s = bar_s + 8 * t, my_p = bar_p + 8 * t, my_o = bar_o + 8 * t;
        const float sl2 = p.scale_log2;
        float m_used = -INFINITY;
        float l = 0.f;
        bool ok = true;
        for (int j = 0; j < nbt; ++j) {
            if (!__all_sync(0xffffffffu, mbar_wait(my_s, j & 1, wd, kSiteSoftS))) {
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
                for (int c = 0; c < 128; ++c)
                    if (kbase + c > last) s[c >> 5][c & 31] = f2u(-INFINITY);
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
            const bool grow = m_cand > m_used + kRescale;
            float alpha = 1.f;
            if (grow) {
                alpha = ex2(m_used - m_cand);  // 0 on the first block (m_used = -inf)
                m_used = m_cand;
            }
            l *= alpha;
            const float off = (m_used == -INFINITY) ? 0.f : kShift - m_used;
            const uint64_t c2 = f2_pack(sl2, sl2), o2 = f2_pack(off, off);
            uint64_t ls2 = 0;  // paired partial sums
            // P (e4m3), keys [4i, 4i + 4) in column i of this row, over S: the P V
            // of the previous block, which read these columns, finished before S
            // of this block (issued after it) did
            uint32_t w[32];
#pragma unroll
            for (int c = 0; c < 8; ++c) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int k0 = 16 * c + 4 * q;
                    const float2 a = f2_unpack(ffma2(
                        f2_pack(u2f(s[k0 >> 5][k0 & 31]), u2f(s[k0 >> 5][(k0 & 31) + 1])), c2, o2));
                    const float2 b = f2_unpack(ffma2(
                        f2_pack(u2f(s[k0 >> 5][(k0 & 31) + 2]), u2f(s[k0 >> 5][(k0 & 31) + 3])), c2, o2));
                    const float p0 = ex2(a.x), p1 = ex2(a.y), p2 = ex2(b.x), p3 = ex2(b.y);
                    ls2 = fadd2(ls2, f2_pack(p0, p1));
                    ls2 = fadd2(ls2, f2_pack(p2, p3));
                    w[4 * c + q] = pack_e4m3x4(p0, p1, p2, p3);
                }
            }
            tmem_st32(tS, w);
            const float2 ls = f2_unpack(ls2);
            l += ls.x + ls.y;
            if (j > 0 && __any_sync(0xffffffffu, grow)) {
                // rescale this warp's rows of O once the previous P V has landed
                if (!__all_sync(0xffffffffu, mbar_wait(my_o, (j - 1) & 1, wd, kSiteSoftO))) {
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
            mbar_arrive(my_p);
        }

        // ---------------------------------------------------------- epilogue --
        bool epi = ok && nbt > 0;
        if (epi) epi = __all_sync(0xffffffffu, mbar_wait(my_o, (nbt - 1) & 1, wd, kSiteEpi));
        if (epi) {
            tc_fence_after();
            const float scale = p.v_scale / l;
            // bf16 O staged over this tile's Q and P (32 KB, two [128 x 64] boxes)
            uint8_t* stage = smem + (t ? kQ1 : kQ0);
#pragma unroll
            for (int c0 = 0; c0 < kD; c0 += 32) {
                uint32_t o[32];
                tmem_ld32(tO + c0, o);
                tmem_ld_wait(o);
                const int box = c0 / 64;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int chunk = (c0 % 64) / 8 + q;
                    uint4 v;
                    v.x = pack_bf16(u2f(o[8 * q + 0]) * scale, u2f(o[8 * q + 1]) * scale);
                    v.y = pack_bf16(u2f(o[8 * q + 2]) * scale, u2f(o[8 * q + 3]) * scale);
                    v.z = pack_bf16(u2f(o[8 * q + 4]) * scale, u2f(o[8 * q + 5]) * scale);
                    v.w = pack_bf16(u2f(o[8 * q + 6]) * scale, u2f(o[8 * q + 7]) * scale);
                    *reinterpret_cast<uint4*>(stage + box * kOutBox + r * 128 +
                                              ((chunk ^ (r & 7)) << 4)) = v;
                }
            }
            fence_async_shared();
            if (row < N)
                p.LSE[static_cast<int64_t>(bh) * N + row] = (m_used - kShift + __log2f(l)) * kLn2;
        }
        if (nbt > 0) {
            named_bar_sync(1 + t, 128);  // every thread of the warpgroup gets here
            if (r == 0 && epi) {
                const uint32_t src = sbase + (t ? kQ1 : kQ0);
                for (int b = 0; b < kD / 64; ++b) tma_store_3d(&tmO, src + b * kOutBox, b * 64, q_start, bh);
                bulk_commit();
                bulk_wait_read<0>();
            }
        }
    }

    // ------------------------------------------------------------- teardown --
    if (sh.abort_flag) drain_after_abort();
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <bool CAUSAL>
cudaError_t launch_fp8_t(const Fp8Args& a, cudaStream_t stream) {
    CUtensorMap tq, tk, tv, to;
    const auto U8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
    if (!make_tile_map(&tq, a.Q, U8, 1, kD, a.N, a.BH, kD, kBM) ||
        !make_tile_map(&tk, a.K, U8, 1, kD, a.N, a.BH, kD, kBN) ||
        !make_tile_map(&tv, a.V, U8, 1, kD, a.N, a.BH, kD, kBN) ||
        !make_tile_map(&to, a.O, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, kD, a.N, a.BH, 64, kBM))
        return cudaErrorInvalidValue;
    constexpr auto kern = &fa_fwd_fp8_kernel<CAUSAL>;
    cudaError_t e = set_max_dyn_smem_once<kern>(kDynSmem);
    if (e != cudaSuccess) return e;
    Fp8Params p;
    p.LSE = a.LSE;
    p.N = a.N;
    p.n_pairs = (a.N + 2 * kBM - 1) / (2 * kBM);
    p.scale_log2 = a.tau * a.q_scale * a.k_scale * kLog2e;
    p.v_scale = a.v_scale;
    p.err = a.err;
    p.wait_limit_ns = a.wait_limit_ns;
    dim3 grid(static_cast<unsigned>(a.BH), static_cast<unsigned>(p.n_pairs));
    if (a.ev_start) cudaEventRecord(a.ev_start, stream);
    kern<<<grid, kThreads, kDynSmem, stream>>>(tq, tk, tv, to, p);
    e = cudaGetLastError();
    if (e == cudaSuccess && a.ev_stop) e = cudaEventRecord(a.ev_stop, stream);
    return e;
}

}  // namespace

cudaError_t launch_fwd_fp8(const Fp8Args& a, cudaStream_t stream) {
    return a.causal ? launch_fp8_t<true>(a, stream) : launch_fp8_t<false>(a, stream);
}

}  // namespace fa
