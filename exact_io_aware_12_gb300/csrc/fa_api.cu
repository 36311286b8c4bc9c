// The C ABI of the library (declared in include/fa.h): argument checks, TMA
// descriptor encoding, the per-device error word and the kernel launches.
#include <atomic>
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <unordered_map>

#include "../../include/fa.h"
#include "fa_internal.h"
#include "ptx.cuh"

// One error word per device (each device holds its own copy of this
// variable; host code must look its address up per device).
__device__ unsigned int g_fa_error_word;

namespace fa {
namespace {

constexpr unsigned long long kDefaultWaitLimitNs = 2000000000ull;
std::atomic<unsigned long long> g_wait_limit_ns{kDefaultWaitLimitNs};
thread_local cudaEvent_t t_ev_start = nullptr;  // fa_set_timing_events
thread_local cudaEvent_t t_ev_stop = nullptr;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

constexpr int kMaxDevices = 64;
struct DeviceInfo {
    std::once_flag once;
    bool supported = false;
    unsigned int* err_word = nullptr;  // device address of g_fa_error_word
};
DeviceInfo g_dev[kMaxDevices];

// Checks the current device once: it must be sm_103 and the error word's
// device address must resolve.  Returns nullptr if the device is unusable.
DeviceInfo* current_device(fa_status* why) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        *why = FA_ERR_CUDA;
        return nullptr;
    }
    DeviceInfo& di = g_dev[dev];
    std::call_once(di.once, [&di, dev] {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
            cudaGetLastError();
            return;
        }
        if (major != 10 || minor != 3) return;
        void* addr = nullptr;
        if (cudaGetSymbolAddress(&addr, g_fa_error_word) != cudaSuccess) {
            cudaGetLastError();
            return;
        }
        di.err_word = static_cast<unsigned int*>(addr);
        di.supported = true;
    });
    if (!di.supported) {
        *why = FA_ERR_UNSUPPORTED;
        return nullptr;
    }
    return &di;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

// Shape checks common to every call.  Returns FA_OK and sets *empty when the
// problem has no rows.
fa_status check_shape(int B, int H, int N, int d, float tau, int causal, bool* empty) {
    if (B < 0 || H < 0 || N < 0 || d < 0) return FA_ERR_INVALID_ARG;
    if (!(std::isfinite(tau) && tau > 0.f)) return FA_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
    *empty = (B == 0 || H == 0 || N == 0);
    if (d != 64 && d != 128) return *empty ? FA_OK : FA_ERR_UNSUPPORTED;
    if (*empty) return FA_OK;
    const long long bh = static_cast<long long>(B) * H;
    if (bh > INT_MAX) return FA_ERR_UNSUPPORTED;
    // grid.y holds 256-row query-tile pairs (forward) and 128-row key tiles (backward)
    if ((static_cast<long long>(N) + 127) / 128 > 65535) return FA_ERR_UNSUPPORTED;
    return FA_OK;
}

fa_status map_cuda(cudaError_t e) { return e == cudaSuccess ? FA_OK : FA_ERR_CUDA; }

// Block-mask checks: mask_heads is 1 or B*H and the mask fits the kernels'
// per-tile bit sets.  Sets *bytes (the mask's size) and *head_stride.
fa_status check_blocks(const uint8_t* blocks, int mask_heads, int B, int H, int N, size_t* bytes,
                       long long* head_stride) {
    if (blocks == nullptr) return FA_ERR_INVALID_ARG;
    const long long bh = static_cast<long long>(B) * H;
    if (mask_heads != 1 && mask_heads != bh) return FA_ERR_INVALID_ARG;
    const long long nb = (static_cast<long long>(N) + kMaskBlockEdge - 1) / kMaskBlockEdge;
    if (nb > kMaxMaskBlocks) return FA_ERR_UNSUPPORTED;
    *bytes = static_cast<size_t>(mask_heads) * static_cast<size_t>(nb * nb);
    *head_stride = mask_heads == 1 ? 0 : nb * nb;
    return FA_OK;
}

fa_status fwd_common(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H,
                     int N, int d, float tau, int causal, void* stream, bool o32, int window = 0,
                     const uint8_t* blocks = nullptr, int mask_heads = 0) {
    bool empty = false;
    fa_status s = check_shape(B, H, N, d, tau, causal, &empty);
    if (s != FA_OK || empty) return s;
    size_t mask_bytes = 0;
    long long mask_stride = 0;
    if (mask_heads != 0) {
        s = check_blocks(blocks, mask_heads, B, H, N, &mask_bytes, &mask_stride);
        if (s != FA_OK) return s;
    }
    const void* ptrs[] = {Q, K, V, O, LSE};
    for (const void* p : ptrs)
        if (p == nullptr || !aligned16(p)) return FA_ERR_INVALID_ARG;
    const size_t rows = static_cast<size_t>(B) * H * N;
    const size_t in_bytes = rows * d * 2, o_bytes = rows * d * (o32 ? 4 : 2), l_bytes = rows * 4;
    const void* ins[] = {Q, K, V};
    for (const void* in : ins)
        if (overlaps(O, o_bytes, in, in_bytes) || overlaps(LSE, l_bytes, in, in_bytes))
            return FA_ERR_INVALID_ARG;
    if (overlaps(O, o_bytes, LSE, l_bytes)) return FA_ERR_INVALID_ARG;
    if (blocks && (overlaps(O, o_bytes, blocks, mask_bytes) || overlaps(LSE, l_bytes, blocks, mask_bytes)))
        return FA_ERR_INVALID_ARG;
    DeviceInfo* di = current_device(&s);
    if (!di) return s;
    FwdArgs a;
    a.Q = Q;
    a.K = K;
    a.V = V;
    a.O = O;
    a.LSE = LSE;
    a.BH = B * H;
    a.N = N;
    a.d = d;
    a.tau = tau;
    a.causal = causal != 0;
    a.window = window;
    a.blocks = blocks;
    a.blocks_head_stride = mask_stride;
    a.o32 = o32;
    a.err = di->err_word;
    a.wait_limit_ns = g_wait_limit_ns.load();
    a.ev_start = t_ev_start;
    a.ev_stop = t_ev_stop;
    return map_cuda(launch_fwd(a, static_cast<cudaStream_t>(stream)));
}

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

__global__ void watchdog_selftest_kernel(unsigned int* err, unsigned long long limit_ns) {
    __shared__ uint64_t never;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(smem_addr(&never), 1);
        mbar_init_fence();
    }
    __syncthreads();
    const Watchdog wd{err, &abort_flag, limit_ns};
    // Nothing ever arrives on `never`: the wait must give up after limit_ns.
    mbar_wait(smem_addr(&never), 0, wd, 0xEE);
    __syncthreads();
}

}  // namespace

namespace {
// Encoded maps, keyed by every argument of the encode: a map only describes an
// address, a shape and a box, so a hit is the same 128 bytes the driver would
// produce again.  Bounded: cleared when full.
struct MapKey {
    uintptr_t base;
    int dtype, esize, cols, rows, planes, box_cols, box_rows;
    bool operator==(const MapKey& o) const {
        return base == o.base && dtype == o.dtype && esize == o.esize && cols == o.cols &&
               rows == o.rows && planes == o.planes && box_cols == o.box_cols && box_rows == o.box_rows;
    }
};
struct MapKeyHash {
    size_t operator()(const MapKey& k) const {
        uint64_t h = k.base * 0x9E3779B97F4A7C15ull;
        const int f[] = {k.dtype, k.esize, k.cols, k.rows, k.planes, k.box_cols, k.box_rows};
        for (int x : f) h = (h ^ static_cast<uint64_t>(x)) * 0x100000001B3ull;
        return static_cast<size_t>(h);
    }
};
constexpr size_t kMapCacheMax = 4096;
std::mutex g_map_mutex;
std::unordered_map<MapKey, CUtensorMap, MapKeyHash>& map_cache() {
    static std::unordered_map<MapKey, CUtensorMap, MapKeyHash> cache;
    return cache;
}
}  // namespace

bool make_tile_map(CUtensorMap* map, const void* base, CUtensorMapDataType dtype, int esize,
                   int cols, int rows, int planes, int box_cols, int box_rows) {
    const MapKey key{reinterpret_cast<uintptr_t>(base), static_cast<int>(dtype), esize, cols, rows,
                     planes, box_cols, box_rows};
    {
        std::lock_guard<std::mutex> lock(g_map_mutex);
        auto it = map_cache().find(key);
        if (it != map_cache().end()) {
            *map = it->second;
            return true;
        }
    }
    if (!encode_tile_map(map, base, dtype, esize, cols, rows, planes, box_cols, box_rows)) return false;
    std::lock_guard<std::mutex> lock(g_map_mutex);
    if (map_cache().size() >= kMapCacheMax) map_cache().clear();
    map_cache().emplace(key, *map);
    return true;
}

bool encode_tile_map(CUtensorMap* map, const void* base, CUtensorMapDataType dtype, int esize,
                     int cols, int rows, int planes, int box_cols, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows),
                                static_cast<cuuint64_t>(planes)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols) * esize,
                                   static_cast<cuuint64_t>(cols) * rows * esize};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows), 1};
    const cuuint32_t estride[3] = {1, 1, 1};
    return fn(map, dtype, 3, const_cast<void*>(base), dims, strides, box, estride,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_watchdog_selftest(unsigned int* err, unsigned long long limit_ns,
                                     cudaStream_t stream) {
    watchdog_selftest_kernel<<<1, 32, 0, stream>>>(err, limit_ns);
    return cudaGetLastError();
}

}  // namespace fa

using namespace fa;

extern "C" {

fa_status fa_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H,
                 int N, int d, float tau, int causal, void* stream) {
    return fwd_common(Q, K, V, O, LSE, B, H, N, d, tau, causal, stream, false);
}

fa_status fa_fwd_o32(const void* Q, const void* K, const void* V, float* O, float* LSE, int B,
                     int H, int N, int d, float tau, int causal, void* stream) {
    return fwd_common(Q, K, V, O, LSE, B, H, N, d, tau, causal, stream, true);
}

size_t fa_bwd_workspace_size(int B, int H, int N, int d) {
    if (B <= 0 || H <= 0 || N <= 0 || (d != 64 && d != 128)) return 0;
    const size_t rows = static_cast<size_t>(B) * H * N;
    return round256(rows * sizeof(float)) + round256(rows * d * sizeof(float));
}

static fa_status bwd_common(const void* Q, const void* K, const void* V, const void* O,
                            const void* dO, const float* LSE, void* dQ, void* dK, void* dV,
                            void* workspace, size_t workspace_bytes, int B, int H, int N, int d,
                            float tau, int causal, int window, void* stream,
                            const uint8_t* blocks = nullptr, int mask_heads = 0) {
    bool empty = false;
    fa_status s = check_shape(B, H, N, d, tau, causal, &empty);
    if (s != FA_OK || empty) return s;
    size_t mask_bytes = 0;
    long long mask_stride = 0;
    if (mask_heads != 0) {
        s = check_blocks(blocks, mask_heads, B, H, N, &mask_bytes, &mask_stride);
        if (s != FA_OK) return s;
    }
    const void* ptrs[] = {Q, K, V, O, dO, LSE, dQ, dK, dV};
    for (const void* p : ptrs)
        if (p == nullptr || !aligned16(p)) return FA_ERR_INVALID_ARG;
    if (workspace != nullptr && !aligned16(workspace)) return FA_ERR_INVALID_ARG;
    const size_t rows = static_cast<size_t>(B) * H * N;
    const size_t tb = rows * d * 2;
    const void* ins[] = {Q, K, V, O, dO};
    void* outs[] = {dQ, dK, dV};
    for (void* o : outs) {
        for (const void* in : ins)
            if (overlaps(o, tb, in, tb)) return FA_ERR_INVALID_ARG;
        if (overlaps(o, tb, LSE, rows * 4)) return FA_ERR_INVALID_ARG;
    }
    if (overlaps(dQ, tb, dK, tb) || overlaps(dQ, tb, dV, tb) || overlaps(dK, tb, dV, tb))
        return FA_ERR_INVALID_ARG;
    if (blocks)
        for (void* o : outs)
            if (overlaps(o, tb, blocks, mask_bytes)) return FA_ERR_INVALID_ARG;
    const size_t need = fa_bwd_workspace_size(B, H, N, d);
    if (workspace != nullptr) {
        if (workspace_bytes < need) return FA_ERR_WORKSPACE;
        const void* all[] = {Q, K, V, O, dO, dQ, dK, dV};
        for (const void* p : all)
            if (overlaps(workspace, need, p, tb)) return FA_ERR_INVALID_ARG;
        if (overlaps(workspace, need, LSE, rows * 4)) return FA_ERR_INVALID_ARG;
        if (blocks && overlaps(workspace, need, blocks, mask_bytes)) return FA_ERR_INVALID_ARG;
    }
    DeviceInfo* di = current_device(&s);
    if (!di) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    void* ws = workspace;
    if (ws == nullptr && cudaMallocAsync(&ws, need, st) != cudaSuccess) {
        cudaGetLastError();
        return FA_ERR_CUDA;
    }
    BwdArgs a;
    a.Q = Q;
    a.K = K;
    a.V = V;
    a.O = O;
    a.dO = dO;
    a.LSE = LSE;
    a.dQ = dQ;
    a.dK = dK;
    a.dV = dV;
    a.D = static_cast<float*>(ws);
    a.dQacc = reinterpret_cast<float*>(static_cast<char*>(ws) + round256(rows * sizeof(float)));
    a.BH = B * H;
    a.N = N;
    a.d = d;
    a.tau = tau;
    a.causal = causal != 0;
    a.window = window;
    a.blocks = blocks;
    a.blocks_head_stride = mask_stride;
    a.err = di->err_word;
    a.wait_limit_ns = g_wait_limit_ns.load();
    a.ev_start = t_ev_start;
    a.ev_stop = t_ev_stop;
    const cudaError_t e = launch_bwd(a, st);
    if (workspace == nullptr) cudaFreeAsync(ws, st);
    return map_cuda(e);
}

fa_status fa_bwd(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                 const float* LSE, void* dQ, void* dK, void* dV, void* workspace,
                 size_t workspace_bytes, int B, int H, int N, int d, float tau, int causal,
                 void* stream) {
    return bwd_common(Q, K, V, O, dO, LSE, dQ, dK, dV, workspace, workspace_bytes, B, H, N, d, tau,
                      causal, 0, stream);
}

fa_status fa_fwd_window(const void* Q, const void* K, const void* V, void* O, float* LSE, int B,
                        int H, int N, int d, float tau, int window, void* stream) {
    if (window < 1) return FA_ERR_INVALID_ARG;
    return fwd_common(Q, K, V, O, LSE, B, H, N, d, tau, 1, stream, false, window);
}

fa_status fa_bwd_window(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                        const float* LSE, void* dQ, void* dK, void* dV, void* workspace,
                        size_t workspace_bytes, int B, int H, int N, int d, float tau, int window,
                        void* stream) {
    if (window < 1) return FA_ERR_INVALID_ARG;
    return bwd_common(Q, K, V, O, dO, LSE, dQ, dK, dV, workspace, workspace_bytes, B, H, N, d, tau,
                      1, window, stream);
}

fa_status fa_fwd_blocks(const void* Q, const void* K, const void* V, void* O, float* LSE, int B,
                        int H, int N, int d, float tau, int causal, const unsigned char* block_mask,
                        int mask_heads, void* stream) {
    if (mask_heads == 0) return FA_ERR_INVALID_ARG;
    return fwd_common(Q, K, V, O, LSE, B, H, N, d, tau, causal, stream, false, 0, block_mask,
                      mask_heads);
}

fa_status fa_bwd_blocks(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                        const float* LSE, void* dQ, void* dK, void* dV, void* workspace,
                        size_t workspace_bytes, int B, int H, int N, int d, float tau, int causal,
                        const unsigned char* block_mask, int mask_heads, void* stream) {
    if (mask_heads == 0) return FA_ERR_INVALID_ARG;
    return bwd_common(Q, K, V, O, dO, LSE, dQ, dK, dV, workspace, workspace_bytes, B, H, N, d, tau,
                      causal, 0, stream, block_mask, mask_heads);
}

size_t fa_decode_workspace_size(int B, int H, int Nq, int Nk, int d) {
    if (B <= 0 || H <= 0 || Nq <= 0 || Nq > 8 || Nk <= 0 || (d != 64 && d != 128)) return 0;
    const long long bh = static_cast<long long>(B) * H;
    if (bh > INT_MAX) return 0;
    int splits = 1, chunk = 0;
    decode_plan(static_cast<int>(bh), Nk, &splits, &chunk);
    if (splits <= 1) return 0;
    const size_t rows = static_cast<size_t>(bh) * Nq;
    return round256(static_cast<size_t>(splits) * rows * (d + 2) * sizeof(float));
}

fa_status fa_fwd_decode(const void* Q, const void* K, const void* V, void* O, float* LSE, int B,
                        int H, int Nq, int Nk, int d, float tau, int causal, void* workspace,
                        size_t workspace_bytes, void* stream) {
    if (B < 0 || H < 0 || Nq < 0 || Nk < 0 || d < 0) return FA_ERR_INVALID_ARG;
    if (!(std::isfinite(tau) && tau > 0.f)) return FA_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
    if (B == 0 || H == 0 || Nq == 0) return FA_OK;
    if (Nk == 0 || (causal && Nq > Nk)) return FA_ERR_INVALID_ARG;
    if ((d != 64 && d != 128) || Nq > 8) return FA_ERR_UNSUPPORTED;
    const long long bh = static_cast<long long>(B) * H;
    if (bh > INT_MAX) return FA_ERR_UNSUPPORTED;
    int splits = 1, chunk = 0;
    decode_plan(static_cast<int>(bh), Nk, &splits, &chunk);
    if (splits > 65535) return FA_ERR_UNSUPPORTED;
    const void* ptrs[] = {Q, K, V, O, LSE};
    for (const void* p : ptrs)
        if (p == nullptr || !aligned16(p)) return FA_ERR_INVALID_ARG;
    if (workspace != nullptr && !aligned16(workspace)) return FA_ERR_INVALID_ARG;
    const size_t qb = static_cast<size_t>(bh) * Nq * d * 2, kb = static_cast<size_t>(bh) * Nk * d * 2;
    const size_t lb = static_cast<size_t>(bh) * Nq * 4;
    const void* ins[] = {Q, K, V};
    const size_t in_bytes[] = {qb, kb, kb};
    for (int i = 0; i < 3; ++i)
        if (overlaps(O, qb, ins[i], in_bytes[i]) || overlaps(LSE, lb, ins[i], in_bytes[i]))
            return FA_ERR_INVALID_ARG;
    if (overlaps(O, qb, LSE, lb)) return FA_ERR_INVALID_ARG;
    const size_t need = fa_decode_workspace_size(B, H, Nq, Nk, d);
    if (workspace != nullptr && need > 0) {
        if (workspace_bytes < need) return FA_ERR_WORKSPACE;
        const void* all[] = {Q, K, V, O, LSE};
        const size_t all_bytes[] = {qb, kb, kb, qb, lb};
        for (int i = 0; i < 5; ++i)
            if (overlaps(workspace, need, all[i], all_bytes[i])) return FA_ERR_INVALID_ARG;
    }
    fa_status s = FA_OK;
    DeviceInfo* di = current_device(&s);
    if (!di) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    void* ws = need > 0 ? workspace : nullptr;
    const bool own = need > 0 && workspace == nullptr;
    if (own && cudaMallocAsync(&ws, need, st) != cudaSuccess) {
        cudaGetLastError();
        return FA_ERR_CUDA;
    }
    DecArgs a;
    a.Q = Q;
    a.K = K;
    a.V = V;
    a.O = O;
    a.LSE = LSE;
    a.workspace = static_cast<float*>(ws);
    a.BH = static_cast<int>(bh);
    a.Nq = Nq;
    a.Nk = Nk;
    a.d = d;
    a.tau = tau;
    a.causal = causal != 0;
    a.splits = splits;
    a.chunk = chunk;
    a.err = di->err_word;
    a.wait_limit_ns = g_wait_limit_ns.load();
    a.ev_start = t_ev_start;
    a.ev_stop = t_ev_stop;
    const cudaError_t e = launch_decode(a, st);
    if (own) cudaFreeAsync(ws, st);
    return map_cuda(e);
}

fa_status fa_fwd_fp8(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H,
                     int N, int d, float tau, int causal, float q_scale, float k_scale,
                     float v_scale, void* stream) {
    bool empty = false;
    fa_status s = check_shape(B, H, N, d, tau, causal, &empty);
    if (s != FA_OK || empty) return s;
    if (d != 128) return FA_ERR_UNSUPPORTED;
    const float scales[] = {q_scale, k_scale, v_scale};
    for (float sc : scales)
        if (!(std::isfinite(sc) && sc > 0.f)) return FA_ERR_INVALID_ARG;
    const void* ptrs[] = {Q, K, V, O, LSE};
    for (const void* p : ptrs)
        if (p == nullptr || !aligned16(p)) return FA_ERR_INVALID_ARG;
    const size_t rows = static_cast<size_t>(B) * H * N;
    const size_t in_bytes = rows * d, o_bytes = rows * d * 2, l_bytes = rows * 4;
    const void* ins[] = {Q, K, V};
    for (const void* in : ins)
        if (overlaps(O, o_bytes, in, in_bytes) || overlaps(LSE, l_bytes, in, in_bytes))
            return FA_ERR_INVALID_ARG;
    if (overlaps(O, o_bytes, LSE, l_bytes)) return FA_ERR_INVALID_ARG;
    DeviceInfo* di = current_device(&s);
    if (!di) return s;
    Fp8Args a;
    a.Q = Q;
    a.K = K;
    a.V = V;
    a.O = O;
    a.LSE = LSE;
    a.BH = B * H;
    a.N = N;
    a.tau = tau;
    a.q_scale = q_scale;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    a.causal = causal != 0;
    a.err = di->err_word;
    a.wait_limit_ns = g_wait_limit_ns.load();
    a.ev_start = t_ev_start;
    a.ev_stop = t_ev_stop;
    return map_cuda(launch_fwd_fp8(a, static_cast<cudaStream_t>(stream)));
}

const char* fa_status_string(fa_status s) {
    switch (s) {
        case FA_OK: return "FA_OK";
        case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG: invalid argument";
        case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED: unsupported head dim, size or device";
        case FA_ERR_WORKSPACE: return "FA_ERR_WORKSPACE: workspace too small";
        case FA_ERR_CUDA: return "FA_ERR_CUDA: CUDA runtime or launch error";
        case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT: a kernel pipeline wait timed out";
    }
    return "unknown fa_status";
}

fa_status fa_last_device_error(void* stream) {
    fa_status s;
    DeviceInfo* di = current_device(&s);
    if (!di) return s;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return FA_ERR_CUDA;
    }
    unsigned int word = 0;
    if (cudaMemcpy(&word, di->err_word, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) {
        cudaGetLastError();
        return FA_ERR_CUDA;
    }
    if (word != 0) {
        const unsigned int zero = 0;
        if (cudaMemcpy(di->err_word, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) {
            cudaGetLastError();
            return FA_ERR_CUDA;
        }
        return FA_ERR_TIMEOUT;
    }
    return FA_OK;
}

fa_status fa_set_wait_limit_ns(unsigned long long ns) {
    g_wait_limit_ns.store(ns == 0 ? kDefaultWaitLimitNs : ns);
    return FA_OK;
}

fa_status fa_set_timing_events(void* start, void* stop) {
    if ((start == nullptr) != (stop == nullptr)) return FA_ERR_INVALID_ARG;
    t_ev_start = static_cast<cudaEvent_t>(start);
    t_ev_stop = static_cast<cudaEvent_t>(stop);
    return FA_OK;
}

fa_status fa_watchdog_selftest(unsigned long long limit_ns, void* stream) {
    if (limit_ns == 0 || limit_ns > 10000000000ull) return FA_ERR_INVALID_ARG;
    fa_status s;
    DeviceInfo* di = current_device(&s);
    if (!di) return s;
    return map_cuda(launch_watchdog_selftest(di->err_word, limit_ns,
                                             static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free backward (fa_bwd_noalloc).  The scratch is a fixed array in
// the device image.  In host code `g_fa_noalloc_scratch` only names a host-side
// stand-in, so its device address is looked up per device with
// cudaGetSymbolAddress before it is handed to the kernels.
static __device__ __align__(256) unsigned char g_fa_noalloc_scratch[FA_NOALLOC_SCRATCH_BYTES];

namespace {
// The scratch array's device address, per device; null until a lookup succeeds.
// A failed lookup (for instance a first call made while the stream is being
// captured) is not remembered: the next call tries again.
std::atomic<void*> g_noalloc_ptr[fa::kMaxDevices];

// Looks the array's address up on the current device (the caller's).
void* noalloc_scratch_for_current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= fa::kMaxDevices) {
        cudaGetLastError();
        return nullptr;
    }
    void* p = g_noalloc_ptr[dev].load(std::memory_order_acquire);
    if (p != nullptr) return p;
    if (cudaGetSymbolAddress(&p, g_fa_noalloc_scratch) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    g_noalloc_ptr[dev].store(p, std::memory_order_release);
    return p;
}
}  // namespace

extern "C" fa_status fa_bwd_noalloc(const void* Q, const void* K, const void* V, const void* O,
                                    const void* dO, const float* LSE, void* dQ, void* dK,
                                    void* dV, int B, int H, int N, int d, float tau, int causal,
                                    void* stream) {
    bool empty = false;
    const fa_status s = fa::check_shape(B, H, N, d, tau, causal, &empty);
    if (s != FA_OK || empty) return s;
    // the one limit of this entry point: the problem's scratch must fit the array
    if (fa_bwd_workspace_size(B, H, N, d) > FA_NOALLOC_SCRATCH_BYTES) return FA_ERR_WORKSPACE;
    // an unsupported device gets the same answer as from every other entry point
    fa_status why = FA_OK;
    if (fa::current_device(&why) == nullptr) return why;
    void* scratch = noalloc_scratch_for_current_device();
    if (scratch == nullptr) return FA_ERR_CUDA;
    // fa_bwd with a caller-provided workspace allocates nothing
    return fa_bwd(Q, K, V, O, dO, LSE, dQ, dK, dV, scratch, FA_NOALLOC_SCRATCH_BYTES, B, H, N, d,
                  tau, causal, stream);
}

