// Host-buffer pipeline (fa_host_pipeline_*): forward + backward steps whose
// inputs and outputs live in host memory.
//
// Each step copies Q, K, V, dO in, runs fa_fwd and fa_bwd on one of `depth`
// device buffer sets, and copies O, LSE, dQ, dK, dV out.  Copies in run on one
// stream, copies out on another and the kernels on the caller's stream;
// events order each buffer set's reuse:
//   - a set's inputs are refilled once its previous step's kernels are done
//     (the copy out reads only the outputs);
//   - its kernels rewrite the outputs once the previous copy out has read them.
// So with depth >= 2 the copies of neighbouring steps overlap the kernels.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <new>

#include "../../include/fa.h"

namespace {

constexpr int kMaxDepth = 8;

struct BufferSet {
    void* q = nullptr;
    void* k = nullptr;
    void* v = nullptr;
    void* dout = nullptr;
    void* o = nullptr;
    void* dq = nullptr;
    void* dk = nullptr;
    void* dv = nullptr;
    float* lse = nullptr;
    void* ws = nullptr;
    cudaEvent_t loaded = nullptr;  // inputs copied in
    cudaEvent_t done = nullptr;    // kernels finished: the inputs may be refilled
    cudaEvent_t freed = nullptr;   // outputs copied out: they may be rewritten
};

}  // namespace

struct fa_host_pipeline {
    int B = 0, H = 0, N = 0, d = 0, causal = 0, depth = 0;
    float tau = 0.f;
    int device = -1;
    size_t tensor_bytes = 0, lse_bytes = 0, ws_bytes = 0;
    cudaStream_t compute = nullptr;  // the caller's stream
    cudaStream_t h2d = nullptr, d2h = nullptr;
    long long steps = 0;
    BufferSet set[kMaxDepth];
};

namespace {

fa_status cuda_ok(cudaError_t e) {
    if (e == cudaSuccess) return FA_OK;
    cudaGetLastError();
    return FA_ERR_CUDA;
}

void release(fa_host_pipeline* p) {
    if (p->device >= 0) cudaSetDevice(p->device);
    for (int i = 0; i < kMaxDepth; ++i) {
        BufferSet& b = p->set[i];
        void* bufs[] = {b.q, b.k, b.v, b.dout, b.o, b.dq, b.dk, b.dv, b.lse, b.ws};
        for (void* x : bufs)
            if (x) cudaFree(x);
        cudaEvent_t evs[] = {b.loaded, b.done, b.freed};
        for (cudaEvent_t e : evs)
            if (e) cudaEventDestroy(e);
    }
    if (p->h2d) cudaStreamDestroy(p->h2d);
    if (p->d2h) cudaStreamDestroy(p->d2h);
    cudaGetLastError();
    delete p;
}

}  // namespace

extern "C" {

fa_status fa_host_pipeline_create(int B, int H, int N, int d, float tau, int causal, int depth,
                                  void* stream, fa_host_pipeline** out) {
    if (out == nullptr) return FA_ERR_INVALID_ARG;
    *out = nullptr;
    if (B < 1 || H < 1 || N < 1 || depth < 1 || depth > kMaxDepth) return FA_ERR_INVALID_ARG;
    if (!(std::isfinite(tau) && tau > 0.f) || (causal != 0 && causal != 1)) return FA_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    fa_host_pipeline* p = new (std::nothrow) fa_host_pipeline;
    if (p == nullptr) return FA_ERR_CUDA;
    p->B = B;
    p->H = H;
    p->N = N;
    p->d = d;
    p->tau = tau;
    p->causal = causal;
    p->depth = depth;
    p->compute = static_cast<cudaStream_t>(stream);
    const size_t rows = static_cast<size_t>(B) * H * N;
    p->tensor_bytes = rows * d * 2;
    p->lse_bytes = rows * 4;
    p->ws_bytes = fa_bwd_workspace_size(B, H, N, d);
    if (cudaGetDevice(&p->device) != cudaSuccess) {
        p->device = -1;
        release(p);
        return FA_ERR_CUDA;
    }
    fa_status s = cuda_ok(cudaStreamCreateWithFlags(&p->h2d, cudaStreamNonBlocking));
    if (s == FA_OK) s = cuda_ok(cudaStreamCreateWithFlags(&p->d2h, cudaStreamNonBlocking));
    for (int i = 0; i < depth && s == FA_OK; ++i) {
        BufferSet& b = p->set[i];
        void** tens[] = {&b.q, &b.k, &b.v, &b.dout, &b.o, &b.dq, &b.dk, &b.dv};
        for (void** t : tens)
            if (s == FA_OK) s = cuda_ok(cudaMalloc(t, p->tensor_bytes));
        if (s == FA_OK) s = cuda_ok(cudaMalloc(reinterpret_cast<void**>(&b.lse), p->lse_bytes));
        if (s == FA_OK) s = cuda_ok(cudaMalloc(&b.ws, p->ws_bytes));
        cudaEvent_t* evs[] = {&b.loaded, &b.done, &b.freed};
        for (cudaEvent_t* e : evs)
            if (s == FA_OK) s = cuda_ok(cudaEventCreateWithFlags(e, cudaEventDisableTiming));
    }
    if (s != FA_OK) {
        release(p);
        return s;
    }
    *out = p;
    return FA_OK;
}

fa_status fa_host_pipeline_step(fa_host_pipeline* p, const void* hQ, const void* hK,
                                const void* hV, const void* hdO, void* hO, float* hLSE, void* hdQ,
                                void* hdK, void* hdV) {
    if (p == nullptr) return FA_ERR_INVALID_ARG;
    const void* ins[] = {hQ, hK, hV, hdO};
    const void* outs[] = {hO, hLSE, hdQ, hdK, hdV};
    for (const void* x : ins)
        if (x == nullptr) return FA_ERR_INVALID_ARG;
    for (const void* x : outs)
        if (x == nullptr) return FA_ERR_INVALID_ARG;
    if (cudaSetDevice(p->device) != cudaSuccess) return cuda_ok(cudaErrorInvalidDevice);
    BufferSet& b = p->set[p->steps % p->depth];
    ++p->steps;
    const size_t tb = p->tensor_bytes;
    // copies in, once this set's previous kernels are done
    fa_status s = cuda_ok(cudaStreamWaitEvent(p->h2d, b.done, 0));
    const void* src[] = {hQ, hK, hV, hdO};
    void* dst[] = {b.q, b.k, b.v, b.dout};
    for (int i = 0; i < 4 && s == FA_OK; ++i)
        s = cuda_ok(cudaMemcpyAsync(dst[i], src[i], tb, cudaMemcpyHostToDevice, p->h2d));
    if (s == FA_OK) s = cuda_ok(cudaEventRecord(b.loaded, p->h2d));
    // the kernels, once the inputs are in and the previous copy out has read the outputs
    if (s == FA_OK) s = cuda_ok(cudaStreamWaitEvent(p->compute, b.loaded, 0));
    if (s == FA_OK) s = cuda_ok(cudaStreamWaitEvent(p->compute, b.freed, 0));
    if (s == FA_OK)
        s = fa_fwd(b.q, b.k, b.v, b.o, b.lse, p->B, p->H, p->N, p->d, p->tau, p->causal, p->compute);
    if (s == FA_OK)
        s = fa_bwd(b.q, b.k, b.v, b.o, b.dout, b.lse, b.dq, b.dk, b.dv, b.ws, p->ws_bytes, p->B, p->H,
                   p->N, p->d, p->tau, p->causal, p->compute);
    if (s == FA_OK) s = cuda_ok(cudaEventRecord(b.done, p->compute));
    // copies out
    if (s == FA_OK) s = cuda_ok(cudaStreamWaitEvent(p->d2h, b.done, 0));
    const void* osrc[] = {b.o, b.dq, b.dk, b.dv};
    void* odst[] = {hO, hdQ, hdK, hdV};
    for (int i = 0; i < 4 && s == FA_OK; ++i)
        s = cuda_ok(cudaMemcpyAsync(odst[i], osrc[i], tb, cudaMemcpyDeviceToHost, p->d2h));
    if (s == FA_OK)
        s = cuda_ok(cudaMemcpyAsync(hLSE, b.lse, p->lse_bytes, cudaMemcpyDeviceToHost, p->d2h));
    if (s == FA_OK) s = cuda_ok(cudaEventRecord(b.freed, p->d2h));
    return s;
}

fa_status fa_host_pipeline_mark(fa_host_pipeline* p, void* event) {
    if (p == nullptr || event == nullptr) return FA_ERR_INVALID_ARG;
    if (cudaSetDevice(p->device) != cudaSuccess) return cuda_ok(cudaErrorInvalidDevice);
    cudaEvent_t e = static_cast<cudaEvent_t>(event);
    // everything enqueued so far, copies included, precedes the mark; every
    // copy enqueued later follows it
    fa_status s = cuda_ok(cudaEventRecord(e, p->h2d));
    if (s == FA_OK) s = cuda_ok(cudaStreamWaitEvent(p->compute, e, 0));
    if (s == FA_OK) s = cuda_ok(cudaEventRecord(e, p->d2h));
    if (s == FA_OK) s = cuda_ok(cudaStreamWaitEvent(p->compute, e, 0));
    if (s == FA_OK) s = cuda_ok(cudaEventRecord(e, p->compute));
    if (s == FA_OK) s = cuda_ok(cudaStreamWaitEvent(p->h2d, e, 0));
    if (s == FA_OK) s = cuda_ok(cudaStreamWaitEvent(p->d2h, e, 0));
    return s;
}

fa_status fa_host_pipeline_sync(fa_host_pipeline* p) {
    if (p == nullptr) return FA_ERR_INVALID_ARG;
    if (cudaSetDevice(p->device) != cudaSuccess) return cuda_ok(cudaErrorInvalidDevice);
    fa_status s = cuda_ok(cudaStreamSynchronize(p->h2d));
    if (s == FA_OK) s = cuda_ok(cudaStreamSynchronize(p->compute));
    if (s == FA_OK) s = cuda_ok(cudaStreamSynchronize(p->d2h));
    return s;
}

fa_status fa_host_pipeline_destroy(fa_host_pipeline* p) {
    if (p == nullptr) return FA_OK;
    const fa_status s = fa_host_pipeline_sync(p);
    release(p);
    return s;
}

}  // extern "C"
