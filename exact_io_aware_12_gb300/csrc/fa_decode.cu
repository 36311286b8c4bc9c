// Decode forward of exact attention for sm_103a: a few new query rows against
// a long KV cache.
//
// Method ("Atencao eficiente - FlashAttention, sparse e hibrida", box
// "FlashAttention nao acelera o decode token a token"): a decode step brings
// one new query row (here 1..8 rows: the last Nq positions of the sequence)
// that must read the whole KV cache from HBM, so the step is bound by memory
// bandwidth, not by the tensor cores.  The arithmetic is the forward's online
// softmax ("Insight 2 - Online softmax"): per query row a running max m and
// sum l, merged block by block, and O = sum_j e^(s_j - m) V_j / l.
//
// GB300 design:
//   - split KV: the cache of each (batch, head) is cut into S chunks of whole
//     64-key tiles and every (head, chunk) is one CTA, two CTAs per SM, so
//     B*H*S CTAs cover the 152 SMs for a few waves even for one sequence;
//   - each CTA streams its K and V tiles with 1-D bulk copies (one per 64-key
//     tile of K and of V: the rows are contiguous) through a 3-slot ring of
//     shared memory with mbarriers, keeping two tiles in flight while one is
//     consumed;
//   - scores on CUDA cores (1..8 query rows are far below a tensor-core tile):
//     d/8 threads per key, each 8 products of a 16-byte K chunk with the query
//     rows held in registers, reduced with shuffles;
//   - one warp per query row runs the online softmax of the tile; then each
//     thread accumulates two output columns over its share of the tile's keys;
//   - with S > 1 each CTA writes its unnormalised O with m and l (log2 units)
//     and fa_decode_combine_kernel merges a row's S partials:
//     M = max_s m_s, O = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s;
//     with S = 1 the CTA writes O and LSE itself.
#include <cuda_bf16.h>

#include <cmath>

#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int kThreads = 256;
constexpr int kTileKeys = 64;
constexpr int kStages = 3;
constexpr float kLn2 = 0.69314718055994531f;
constexpr float kLog2e = 1.44269504088896341f;

template <int D, int NQ>
struct DecLayout {
    static constexpr int kTileBytes = kTileKeys * D * 2;     // one K or V tile (bf16)
    static constexpr int kSlotBytes = 2 * kTileBytes;        // K tile, then V tile
    static constexpr int kRing = 0;
    static constexpr int kP = kStages * kSlotBytes;          // float [NQ][64]: scores, then P
    static constexpr int kAlpha = kP + NQ * kTileKeys * 4;   // float [NQ]: this tile's rescale
    static constexpr int kStat = kAlpha + 8 * 4;             // float m[NQ], l[NQ] at the end
    static constexpr int kBars = kStat + 16 * 4;             // uint64 full[kStages], int abort
    static constexpr int kBytes = kBars + 64;
    static constexpr int kGroups = kThreads / (D / 2);       // P.V key groups
    static_assert(kGroups * NQ * D * 4 <= kStages * kSlotBytes, "reduction buffer fits the ring");
};

struct DecParams {
    const __nv_bfloat16* Q;
    const __nv_bfloat16* K;
    const __nv_bfloat16* V;
    __nv_bfloat16* O;   // S == 1: final outputs
    float* LSE;
    float* Opart;       // S > 1: [S][BH * Nq][D], unnormalised
    float* Mpart;       // [S][BH * Nq], log2 units of the scaled scores
    float* Lpart;       // [S][BH * Nq]
    int BH, Nq, Nk, chunk, splits, causal;
    float scale_log2;   // tau * log2(e)
    unsigned int* err;
    unsigned long long wait_limit_ns;
};

enum : uint32_t { kSiteDecLoad = 41 };

__device__ __forceinline__ float bf_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf_hi(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }

template <int D, int NQ>
__global__ void __launch_bounds__(kThreads, 2) fa_decode_split_kernel(const DecParams p) {
    using L = DecLayout<D, NQ>;
    extern __shared__ __align__(128) uint8_t smem[];
    const uint32_t sbase = smem_addr(smem);
    float* sc = reinterpret_cast<float*>(smem + L::kP);
    float* alpha_s = reinterpret_cast<float*>(smem + L::kAlpha);
    float* stat = reinterpret_cast<float*>(smem + L::kStat);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kBars + 8 * kStages);
    const uint32_t bar_full = sbase + L::kBars;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int bh = blockIdx.x, split = blockIdx.y;
    const int Nq = p.Nq, Nk = p.Nk;
    const int k0 = split * p.chunk;
    const int k1 = min(Nk, k0 + p.chunk);
    const int n_tiles = (k1 - k0 + kTileKeys - 1) / kTileKeys;
    const int64_t kv_row0 = static_cast<int64_t>(bh) * Nk;

    if (tid == 0) {
        *abort_flag = 0;
        for (int s = 0; s < kStages; ++s) mbar_init(bar_full + 8 * s, 1);
        mbar_init_fence();
    }
    __syncthreads();
    const Watchdog wd{p.err, abort_flag, p.wait_limit_ns};

    auto issue = [&](int t) {  // tile t of this chunk into slot t % kStages (one thread)
        const int slot = t % kStages;
        const int key0 = k0 + t * kTileKeys;
        const uint32_t bytes = static_cast<uint32_t>(min(kTileKeys, k1 - key0)) * D * 2;
        const uint32_t dst = sbase + L::kRing + slot * L::kSlotBytes;
        fence_async_shared();  // order this slot's earlier reads before the copy overwrites it
        mbar_arrive_expect_tx(bar_full + 8 * slot, 2 * bytes);
        bulk_load_1d(dst, p.K + (kv_row0 + key0) * D, bytes, bar_full + 8 * slot);
        bulk_load_1d(dst + L::kTileBytes, p.V + (kv_row0 + key0) * D, bytes, bar_full + 8 * slot);
    };
    if (tid == 0)
        for (int t = 0; t < min(kStages, n_tiles); ++t) issue(t);

    // Scores: TPK threads per key, thread `sub` owns columns [8 sub, 8 sub + 8)
    constexpr int TPK = D / 8;
    constexpr int kKeysPerPass = kThreads / TPK;
    const int sub = tid % TPK, kin = tid / TPK;
    float qr[NQ][8];
#pragma unroll
    for (int qi = 0; qi < NQ; ++qi) {
        if (qi < Nq) {
            const uint4 w = *reinterpret_cast<const uint4*>(
                p.Q + (static_cast<int64_t>(bh) * Nq + qi) * D + sub * 8);
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                qr[qi][2 * e] = bf_lo(ws[e]);
                qr[qi][2 * e + 1] = bf_hi(ws[e]);
            }
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) qr[qi][e] = 0.f;
        }
    }
    // P.V: thread owns column pair cp of key group grp
    constexpr int CP = D / 2;
    constexpr int kKeysPerGroup = kTileKeys / L::kGroups;
    const int cp = tid % CP, grp = tid / CP;
    float acc[NQ][2];
#pragma unroll
    for (int qi = 0; qi < NQ; ++qi) acc[qi][0] = acc[qi][1] = 0.f;
    // online-softmax state of query row `warp` (warps < Nq), lane-uniform
    float m_run = -INFINITY, l_run = 0.f;
    const float c = p.scale_log2;

    bool ok = n_tiles == 0 || mbar_wait(bar_full, 0, wd, kSiteDecLoad);
    ok = __syncthreads_and(ok);
    for (int t = 0; ok && t < n_tiles; ++t) {
        const int slot = t % kStages;
        const uint8_t* kt = smem + L::kRing + slot * L::kSlotBytes;
        const uint8_t* vt = kt + L::kTileBytes;
        const int key0 = k0 + t * kTileKeys;
        const int n_valid = min(kTileKeys, k1 - key0);

        // 1. scores s[qi][key] (rows past n_valid hold stale data; masked below)
#pragma unroll
        for (int pass = 0; pass < kTileKeys / kKeysPerPass; ++pass) {
            const int kk = pass * kKeysPerPass + kin;
            const uint4 w = *reinterpret_cast<const uint4*>(kt + kk * D * 2 + sub * 16);
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
            float s[NQ];
#pragma unroll
            for (int qi = 0; qi < NQ; ++qi) {
                float a = 0.f;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    a = fmaf(qr[qi][2 * e], bf_lo(ws[e]), a);
                    a = fmaf(qr[qi][2 * e + 1], bf_hi(ws[e]), a);
                }
                s[qi] = a;
            }
#pragma unroll
            for (int off = TPK / 2; off > 0; off >>= 1)
#pragma unroll
                for (int qi = 0; qi < NQ; ++qi) s[qi] += __shfl_xor_sync(0xffffffffu, s[qi], off);
            if (sub == 0)
#pragma unroll
                for (int qi = 0; qi < NQ; ++qi) sc[qi * kTileKeys + kk] = s[qi];
        }
        __syncthreads();

        // 2. online softmax of row `warp` over this tile (masked: past the chunk,
        //    and with causal past key warp + Nk - Nq)
        if (warp < Nq) {
            const int last = p.causal ? min(k1 - 1, warp + Nk - Nq) : k1 - 1;
            const bool v0 = key0 + lane <= last, v1 = key0 + lane + 32 <= last;
            const float x0 = v0 ? sc[warp * kTileKeys + lane] * c : -INFINITY;
            const float x1 = v1 ? sc[warp * kTileKeys + lane + 32] * c : -INFINITY;
            float mt = fmaxf(x0, x1);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, off));
            const float m_new = fmaxf(m_run, mt);
            const float alpha = (m_new == -INFINITY) ? 1.f : ex2(m_run - m_new);
            const float p0 = v0 ? ex2(x0 - m_new) : 0.f;
            const float p1 = v1 ? ex2(x1 - m_new) : 0.f;
            float ps = p0 + p1;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
            l_run = l_run * alpha + ps;
            m_run = m_new;
            sc[warp * kTileKeys + lane] = p0;
            sc[warp * kTileKeys + lane + 32] = p1;
            if (lane == 0) alpha_s[warp] = alpha;
        }
        __syncthreads();

        // 3. acc = alpha acc + P V over this thread's keys and column pair
#pragma unroll
        for (int qi = 0; qi < NQ; ++qi) {
            const float a = qi < Nq ? alpha_s[qi] : 1.f;
            acc[qi][0] *= a;
            acc[qi][1] *= a;
        }
#pragma unroll 4
        for (int jj = 0; jj < kKeysPerGroup; ++jj) {
            const int j = grp * kKeysPerGroup + jj;
            if (j < n_valid) {
                const uint32_t w = *reinterpret_cast<const uint32_t*>(vt + j * D * 2 + cp * 4);
                const float v0 = bf_lo(w), v1 = bf_hi(w);
#pragma unroll
                for (int qi = 0; qi < NQ; ++qi) {
                    const float pj = sc[qi * kTileKeys + j];
                    acc[qi][0] = fmaf(pj, v0, acc[qi][0]);
                    acc[qi][1] = fmaf(pj, v1, acc[qi][1]);
                }
            }
        }

        // 4. wait for the next tile; the barrier also frees this slot and sc
        bool ok_next = true;
        if (t + 1 < n_tiles)
            ok_next = mbar_wait(bar_full + 8 * ((t + 1) % kStages), ((t + 1) / kStages) & 1, wd,
                                kSiteDecLoad);
        ok = __syncthreads_and(ok_next);
        if (ok && tid == 0 && t + kStages < n_tiles) issue(t + kStages);
    }
    if (!ok) {
        drain_after_abort();  // copies already issued may still land in the ring
        return;
    }

    // Reduce the key groups' partial sums through shared memory (the ring is idle)
    if (warp < Nq && lane == 0) {
        stat[warp] = m_run;
        stat[8 + warp] = l_run;
    }
    float* red = reinterpret_cast<float*>(smem + L::kRing);  // [groups][NQ][D]
#pragma unroll
    for (int qi = 0; qi < NQ; ++qi) {
        red[(grp * NQ + qi) * D + 2 * cp] = acc[qi][0];
        red[(grp * NQ + qi) * D + 2 * cp + 1] = acc[qi][1];
    }
    __syncthreads();
    const int rows = p.BH * Nq;
    for (int e = tid; e < Nq * D; e += kThreads) {
        const int qi = e / D, col = e % D;
        float s = 0.f;
#pragma unroll
        for (int g = 0; g < L::kGroups; ++g) s += red[(g * NQ + qi) * D + col];
        const int row = bh * Nq + qi;
        if (p.splits == 1) {
            p.O[static_cast<int64_t>(row) * D + col] = __float2bfloat16_rn(s / stat[8 + qi]);
        } else {
            p.Opart[(static_cast<int64_t>(split) * rows + row) * D + col] = s;
        }
    }
    if (tid < Nq) {
        const int row = bh * Nq + tid;
        const float m = stat[tid], l = stat[8 + tid];
        if (p.splits == 1) {
            p.LSE[row] = (m + __log2f(l)) * kLn2;
        } else {
            p.Mpart[static_cast<int64_t>(split) * rows + row] = m;
            p.Lpart[static_cast<int64_t>(split) * rows + row] = l;
        }
    }
}

// Merge the S partials of each (head, query row): one warp per row, D/32
// columns per lane.
template <int D>
__global__ void __launch_bounds__(256) fa_decode_combine_kernel(const float* __restrict__ Opart,
                                                                const float* __restrict__ Mpart,
                                                                const float* __restrict__ Lpart,
                                                                __nv_bfloat16* __restrict__ O,
                                                                float* __restrict__ LSE, int rows,
                                                                int splits) {
    constexpr int PER = D / 32;
    const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    float M = -INFINITY;
    for (int s = 0; s < splits; ++s) M = fmaxf(M, Mpart[static_cast<int64_t>(s) * rows + row]);
    float lsum = 0.f, acc[PER];
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] = 0.f;
    for (int s = 0; s < splits; ++s) {
        const int64_t r = static_cast<int64_t>(s) * rows + row;
        const float m = Mpart[r];
        const float w = (m == -INFINITY) ? 0.f : ex2(m - M);  // a chunk the row sees nothing of
        lsum = fmaf(w, Lpart[r], lsum);
        const float* src = Opart + r * D + lane * PER;
#pragma unroll
        for (int e = 0; e < PER; ++e) acc[e] = fmaf(w, src[e], acc[e]);
    }
    const float inv = 1.f / lsum;
#pragma unroll
    for (int e = 0; e < PER; ++e)
        O[static_cast<int64_t>(row) * D + lane * PER + e] = __float2bfloat16_rn(acc[e] * inv);
    if (lane == 0) LSE[row] = (M + __log2f(lsum)) * kLn2;
}

template <int D, int NQ>
cudaError_t launch_decode_t(const DecArgs& a, cudaStream_t stream) {
    using L = DecLayout<D, NQ>;
    constexpr auto kern = &fa_decode_split_kernel<D, NQ>;
    cudaError_t e = set_max_dyn_smem_once<kern>(L::kBytes);
    if (e != cudaSuccess) return e;
    DecParams p;
    p.Q = static_cast<const __nv_bfloat16*>(a.Q);
    p.K = static_cast<const __nv_bfloat16*>(a.K);
    p.V = static_cast<const __nv_bfloat16*>(a.V);
    p.O = static_cast<__nv_bfloat16*>(a.O);
    p.LSE = a.LSE;
    const size_t rows = static_cast<size_t>(a.BH) * a.Nq;
    p.Opart = a.workspace;
    p.Mpart = a.workspace ? a.workspace + static_cast<size_t>(a.splits) * rows * D : nullptr;
    p.Lpart = a.workspace ? p.Mpart + static_cast<size_t>(a.splits) * rows : nullptr;
    p.BH = a.BH;
    p.Nq = a.Nq;
    p.Nk = a.Nk;
    p.chunk = a.chunk;
    p.splits = a.splits;
    p.causal = a.causal ? 1 : 0;
    p.scale_log2 = a.tau * kLog2e;
    p.err = a.err;
    p.wait_limit_ns = a.wait_limit_ns;
    if (a.ev_start) cudaEventRecord(a.ev_start, stream);
    kern<<<dim3(static_cast<unsigned>(a.BH), static_cast<unsigned>(a.splits)), kThreads, L::kBytes,
           stream>>>(p);
    e = cudaGetLastError();
    if (e == cudaSuccess && a.splits > 1) {
        const unsigned blocks = static_cast<unsigned>((rows + 7) / 8);
        fa_decode_combine_kernel<D><<<blocks, 256, 0, stream>>>(
            p.Opart, p.Mpart, p.Lpart, p.O, p.LSE, static_cast<int>(rows), a.splits);
        e = cudaGetLastError();
    }
    if (e == cudaSuccess && a.ev_stop) e = cudaEventRecord(a.ev_stop, stream);
    return e;
}

}  // namespace

void decode_plan(int BH, int Nk, int* splits, int* chunk) {
    // about eight waves of two CTAs on each of 152 SMs, chunks of at least
    // 512 keys, whole 64-key tiles
    const long long want = (8LL * 2 * 152 + BH - 1) / BH;
    const long long most = (static_cast<long long>(Nk) + 511) / 512;
    long long s = want < most ? want : most;
    if (s < 1) s = 1;
    long long c = (static_cast<long long>(Nk) + s - 1) / s;
    c = (c + kTileKeys - 1) / kTileKeys * kTileKeys;
    *chunk = static_cast<int>(c);
    *splits = static_cast<int>((Nk + c - 1) / c);
}

cudaError_t launch_decode(const DecArgs& a, cudaStream_t stream) {
    const int nq = a.Nq <= 1 ? 1 : a.Nq <= 2 ? 2 : a.Nq <= 4 ? 4 : 8;
    if (a.d == 64) {
        switch (nq) {
            case 1: return launch_decode_t<64, 1>(a, stream);
            case 2: return launch_decode_t<64, 2>(a, stream);
            case 4: return launch_decode_t<64, 4>(a, stream);
            default: return launch_decode_t<64, 8>(a, stream);
        }
    }
    switch (nq) {
        case 1: return launch_decode_t<128, 1>(a, stream);
        case 2: return launch_decode_t<128, 2>(a, stream);
        case 4: return launch_decode_t<128, 4>(a, stream);
        default: return launch_decode_t<128, 8>(a, stream);
    }
}

}  // namespace fa
