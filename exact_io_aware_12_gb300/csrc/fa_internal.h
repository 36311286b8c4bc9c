// Host-side declarations shared by the library's translation units.
#pragma once

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <utility>
#include <cuda.h>
#include <cuda_runtime.h>

namespace fa {

// Block masks (block-sparse attention): one byte per [128 query x 128 key] block,
// at most kMaxMaskBlocks blocks per row (so N <= 131072).
constexpr int kMaskBlockEdge = 128;
constexpr int kMaxMaskBlocks = 1024;

// Arguments of one forward launch (device pointers, validated by the caller).
struct FwdArgs {
    const void* Q;
    const void* K;
    const void* V;
    void* O;          // bf16 or fp32 (o32)
    float* LSE;
    int BH, N, d;
    float tau;
    bool causal;
    int window;       // causal sliding window in keys (0 = none)
    const uint8_t* blocks = nullptr;  // block mask [heads][nb][nb] (device) or null
    long long blocks_head_stride = 0;  // bytes between heads' masks (0: one mask)
    bool o32;
    unsigned int* err;
    unsigned long long wait_limit_ns;
    cudaEvent_t ev_start;  // optional: recorded around the kernel
    cudaEvent_t ev_stop;
};

// Arguments of one backward launch sequence.
struct BwdArgs {
    const void* Q;
    const void* K;
    const void* V;
    const void* O;
    const void* dO;
    const float* LSE;
    void* dQ;
    void* dK;
    void* dV;
    float* D;       // workspace: fp32 [BH*N]
    float* dQacc;   // workspace: fp32 [BH*N*d]
    int BH, N, d;
    float tau;
    bool causal;
    int window;     // causal sliding window in keys (0 = none)
    const uint8_t* blocks = nullptr;  // block mask [heads][nb][nb] (device) or null
    long long blocks_head_stride = 0;  // bytes between heads' masks (0: one mask)
    unsigned int* err;
    unsigned long long wait_limit_ns;
    cudaEvent_t ev_start;  // optional: recorded around the main kernel
    cudaEvent_t ev_stop;
};

// Arguments of one FP8 (e4m3) forward: Q, K, V are e4m3 bytes [BH][N][128]
// with one scale per tensor (value = byte * scale); O bf16, LSE fp32.
struct Fp8Args {
    const void* Q;
    const void* K;
    const void* V;
    void* O;
    float* LSE;
    int BH, N;
    float tau, q_scale, k_scale, v_scale;
    bool causal;
    unsigned int* err;
    unsigned long long wait_limit_ns;
    cudaEvent_t ev_start;  // optional: recorded around the kernel
    cudaEvent_t ev_stop;
};

// Arguments of one decode forward (split kernel + combine kernel).
struct DecArgs {
    const void* Q;    // bf16 [BH][Nq][d]
    const void* K;    // bf16 [BH][Nk][d]
    const void* V;
    void* O;          // bf16 [BH][Nq][d]
    float* LSE;       // fp32 [BH][Nq]
    float* workspace; // splits > 1: partials (decode_workspace_bytes)
    int BH, Nq, Nk, d;
    float tau;
    bool causal;
    int splits, chunk;  // from decode_plan
    unsigned int* err;
    unsigned long long wait_limit_ns;
    cudaEvent_t ev_start;  // optional: recorded around the two kernels
    cudaEvent_t ev_stop;
};

// How the decode forward cuts the KV cache: `splits` chunks of `chunk` keys
// (a multiple of 64).  Depends only on its arguments.
void decode_plan(int BH, int Nk, int* splits, int* chunk);

// Encodes a 3-D tiled tensor map over a contiguous [BH][N][cols] tensor with
// a {box_cols, box_rows, 1} box and the 128-byte swizzle (box_cols * esize
// must be 128).  Returns false if the driver rejects it.  make_tile_map keeps
// the maps it has encoded and returns a kept one for the same arguments.
bool make_tile_map(CUtensorMap* map, const void* base, CUtensorMapDataType dtype, int esize,
                   int cols, int rows, int planes, int box_cols, int box_rows);
bool encode_tile_map(CUtensorMap* map, const void* base, CUtensorMapDataType dtype, int esize,
                     int cols, int rows, int planes, int box_cols, int box_rows);

// Raises a kernel's dynamic shared-memory limit to `bytes`, once per device
// (the attribute stays set; later calls only check a flag).
template <auto Kern>
cudaError_t set_max_dyn_smem_once(int bytes) {
    static std::atomic<int> done[64] = {};
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaGetLastError();
    const bool cacheable = dev >= 0 && dev < 64;
    if (cacheable && done[dev].load(std::memory_order_acquire) == bytes) return cudaSuccess;
    const cudaError_t e = cudaFuncSetAttribute(Kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && cacheable) done[dev].store(bytes, std::memory_order_release);
    return e;
}

// Launches `kern` as a programmatic dependent of the previous kernel on the
// stream: it may be scheduled before that kernel has finished, and must call
// griddepcontrol.wait before touching anything that kernel writes.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t stream, Args&&... args) {
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
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

cudaError_t launch_fwd(const FwdArgs& a, cudaStream_t stream);
// d = 64, N <= 2048, bf16 O, no window or block mask: the persistent forward
cudaError_t launch_fwd_short(const FwdArgs& a, cudaStream_t stream);
// d = 128 with a block mask, bf16 O: the persistent block-sparse forward
cudaError_t launch_fwd_sparse(const FwdArgs& a, cudaStream_t stream);
cudaError_t launch_bwd(const BwdArgs& a, cudaStream_t stream);
cudaError_t launch_decode(const DecArgs& a, cudaStream_t stream);
cudaError_t launch_fwd_fp8(const Fp8Args& a, cudaStream_t stream);
cudaError_t launch_watchdog_selftest(unsigned int* err, unsigned long long limit_ns,
                                     cudaStream_t stream);

}  // namespace fa
