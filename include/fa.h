/*
 * Exact IO-aware attention on GB300 (sm_103a): the C ABI.
 *
 * What is computed (tonho.wtf "flash attention" entry, section "como
 * funciona"; "Atencao eficiente - FlashAttention, sparse e hibrida", sections
 * "Insight 1 - Tiling" and "Insight 2 - Online softmax"):
 *
 *   forward   O = softmax(tau * Q K^T [+ causal mask]) V, computed tile by tile
 *             with a running row max m and row sum l, so the N x N score
 *             matrix never reaches device memory; the per-row statistics are
 *             returned packed as LSE = m + ln l.
 *   backward  keeps only O and LSE, rebuilds S and P on chip, and uses
 *             D_i = dO_i . O_i (equal to sum_j P_ij dP_ij) to form
 *             dS = P o (dP - D); returns dQ, dK, dV.
 *
 * Conventions shared by every entry point
 *   - Q, K, V, O, dO, dQ, dK, dV: bf16, contiguous [B][H][N][d] (d fastest).
 *     LSE: fp32 [B][H][N], natural log of sum_j exp(tau q_i . k_j).
 *   - d must be 64 or 128.  N may be any value >= 1 (a ragged last tile is
 *     handled inside the kernels).  B, H, N, d are ints >= 0; B, H or N equal
 *     to 0 is an empty problem: FA_OK, nothing is launched, pointers unused.
 *   - causal = 1 hides key j from query i when j > i (query and key lengths
 *     are equal, so top-left and bottom-right alignment coincide); 0 = no mask.
 *   - tau is the score scale, finite and > 0 (usually 1/sqrt(d)).
 *   - Every pointer is a device pointer (cudaMalloc / PyTorch CUDA memory)
 *     aligned to 16 bytes, except the host buffers of fa_host_pipeline_step.
 *     The caller owns every buffer; apart from a host pipeline object's
 *     buffers and fa_bwd_noalloc's fixed scratch array, the library keeps no
 *     device allocation between calls.  Outputs must not overlap inputs.
 *   - stream is a cudaStream_t (NULL = the legacy default stream).  Calls only
 *     enqueue work on it and never synchronise the host.
 *   - Errors are returned, never printed: invalid arguments are caught before
 *     anything is launched.  A kernel whose internal pipeline wait exceeds the
 *     watchdog limit gives up cleanly and records FA_ERR_TIMEOUT in a device
 *     word that fa_last_device_error() reads.
 */
#ifndef FA_GB300_FA_H
#define FA_GB300_FA_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define FA_API __attribute__((visibility("default")))
#else
#define FA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum fa_status {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, negative size, bad tau, overlap */
    FA_ERR_UNSUPPORTED = 2,  /* d not in {64, 128}, or no sm_103a device */
    FA_ERR_WORKSPACE = 3,    /* workspace given but smaller than fa_bwd_workspace_size */
    FA_ERR_CUDA = 4,         /* a CUDA runtime call or kernel launch failed */
    FA_ERR_TIMEOUT = 5       /* a kernel's bounded pipeline wait ran out */
} fa_status;

/*
 * Forward pass.  Reads Q, K, V; writes O (bf16) and LSE (fp32).
 * Source: tonho.wtf "flash attention", section "como funciona" (scores
 * tau*Q_i K_j^T, running max and sum, store of O and the statistics).
 */
FA_API fa_status fa_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE,
                 int B, int H, int N, int d, float tau, int causal, void* stream);

/*
 * Forward pass with an fp32 O output (same kernel; only the final store
 * differs).  For checks whose tolerance is below the bf16 rounding of O.
 * O: fp32 [B][H][N][d].  Same source as fa_fwd.
 */
FA_API fa_status fa_fwd_o32(const void* Q, const void* K, const void* V, float* O, float* LSE,
                     int B, int H, int N, int d, float tau, int causal, void* stream);

/*
 * Bytes of device scratch fa_bwd needs: D (fp32 [B][H][N]) and the fp32 dQ
 * accumulator ([B][H][N][d]), each padded to 256 bytes.  0 for an empty or
 * unsupported problem.
 */
FA_API size_t fa_bwd_workspace_size(int B, int H, int N, int d);

/*
 * Backward pass.  Reads Q, K, V, O, dO (bf16) and LSE (fp32, as written by
 * fa_fwd for the same Q, K, V, tau, causal); writes dQ, dK, dV (bf16; every
 * element is written, nothing is accumulated into them).
 * workspace: device scratch of at least fa_bwd_workspace_size() bytes, owned
 * by the caller and free for the duration of the call on this stream; NULL
 * asks the library to take it with cudaMallocAsync on the stream and give it
 * back with cudaFreeAsync after the last kernel.
 * Arithmetic: S, dP and every product accumulate in fp32. P and dS enter the
 * tensor-core products as bf16. dS is the bf16 product of the bf16 P and
 * dP - D, which is formed in fp32 and rounded to bf16. dQ is summed over the
 * key tiles in an fp32 accumulator in the workspace.
 * Source: tonho.wtf "flash attention", section "como funciona", backward
 * paragraph (keep O and the statistics, rebuild S and P, D_i = dO_i . O_i);
 * "FlashAttention: O Que E e Como Acelera LLMs na Pratica", pillar 2
 * (recomputation in the backward pass).
 */
FA_API fa_status fa_bwd(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                 const float* LSE, void* dQ, void* dK, void* dV,
                 void* workspace, size_t workspace_bytes,
                 int B, int H, int N, int d, float tau, int causal, void* stream);

/* Static, human-readable name of a status code. */
FA_API const char* fa_status_string(fa_status s);

/*
 * Synchronises `stream`, then reads and clears the library's device error
 * word for the current device.  FA_ERR_TIMEOUT if some kernel launched since
 * the last call gave up on a bounded wait, FA_ERR_CUDA if the stream reports
 * an error, else FA_OK.
 */
FA_API fa_status fa_last_device_error(void* stream);

/*
 * Sets how long (nanoseconds) one pipeline wait inside a kernel may take
 * before the kernel gives up (default 2e9 = 2 s).  Applies to launches made
 * after the call, from any thread.  0 restores the default.
 */
FA_API fa_status fa_set_wait_limit_ns(unsigned long long ns);

/*
 * Watchdog self-test: launches one small kernel whose barrier wait is never
 * satisfied, so it times out after `limit_ns` and exits cleanly.  The caller
 * then sees FA_ERR_TIMEOUT from fa_last_device_error().  No fault, trap or
 * unbounded wait is involved.
 */
FA_API fa_status fa_watchdog_selftest(unsigned long long limit_ns, void* stream);

/*
 * Sliding-window (local) causal attention, forward.  Key j is visible from
 * query i iff i - window < j <= i: each query attends to its `window` most
 * recent keys, itself included ("Atencao eficiente - FlashAttention, sparse e
 * hibrida", section "Atencao hibrida: local + global intercalados": local
 * layers with windows of 4096 or 128 tokens).  Same buffers and conventions
 * as fa_fwd with causal = 1; key blocks outside every row's window are never
 * loaded.  window >= 1 (else FA_ERR_INVALID_ARG); window >= N is plain causal
 * attention.
 */
FA_API fa_status fa_fwd_window(const void* Q, const void* K, const void* V, void* O, float* LSE,
                               int B, int H, int N, int d, float tau, int window, void* stream);

/*
 * Sliding-window backward: fa_bwd for the mask of fa_fwd_window (LSE must come
 * from fa_fwd_window with the same window).  Same workspace rules as fa_bwd.
 */
FA_API fa_status fa_bwd_window(const void* Q, const void* K, const void* V, const void* O,
                               const void* dO, const float* LSE, void* dQ, void* dK, void* dV,
                               void* workspace, size_t workspace_bytes, int B, int H, int N, int d,
                               float tau, int window, void* stream);

/*
 * Block-sparse attention, forward ("FlashAttention e o gargalo real de
 * inferencia", section "o que isso custou": the block-sparse variant skips
 * blocks, an approximation by design; "Atencao eficiente - FlashAttention,
 * sparse e hibrida", section "Sparse e hibrida": each token attends to a
 * subset, e.g. a local window plus global anchor tokens).
 *
 * block_mask: DEVICE pointer to bytes [mask_heads][nb][nb], nb = ceil(N / 128)
 * (FA_BLOCK_MASK_EDGE), row-major: entry [h][i][j] nonzero means the queries
 * of 128-row block i of head h see the keys of 128-key block j.  mask_heads
 * is 1 (one mask for every batch and head) or B*H (head bh = b*H + h uses
 * mask bh); anything else is FA_ERR_INVALID_ARG.  With causal = 1 a key is
 * visible only if it is also at or before the query.  Blocks that are not set
 * are never loaded.  A row that sees no key is the empty sum: O = 0 and
 * LSE = -inf.  The mask is read on the stream; it must stay valid until the
 * call's work is done and must not overlap O or LSE.  N <= FA_BLOCK_MASK_MAX_N
 * (else FA_ERR_UNSUPPORTED).  Other buffers and conventions as fa_fwd.
 */
#define FA_BLOCK_MASK_EDGE 128
#define FA_BLOCK_MASK_MAX_N 131072
FA_API fa_status fa_fwd_blocks(const void* Q, const void* K, const void* V, void* O, float* LSE,
                               int B, int H, int N, int d, float tau, int causal,
                               const unsigned char* block_mask, int mask_heads, void* stream);

/*
 * Block-sparse backward: fa_bwd for the mask of fa_fwd_blocks (LSE must come
 * from fa_fwd_blocks with the same mask).  Rows that see no key get dQ = 0;
 * keys that no query sees get dK = dV = 0.  Same workspace rules as fa_bwd;
 * the mask must not overlap dQ, dK, dV or the workspace.  Until its last
 * kernel writes dQ, the call keeps in dQ's memory the plan that splits key
 * tiles seen by many query tiles over extra CTAs, and their partial dK, dV.
 */
FA_API fa_status fa_bwd_blocks(const void* Q, const void* K, const void* V, const void* O,
                               const void* dO, const float* LSE, void* dQ, void* dK, void* dV,
                               void* workspace, size_t workspace_bytes, int B, int H, int N, int d,
                               float tau, int causal, const unsigned char* block_mask,
                               int mask_heads, void* stream);

/*
 * Decode forward: Nq new query rows per (batch, head) against a KV cache of Nk
 * keys ("Atencao eficiente - FlashAttention, sparse e hibrida", box
 * "FlashAttention nao acelera o decode token a token": each decode step brings
 * one new query row that reads the whole KV cache, so the step is bound by
 * memory bandwidth).  Same result as the forward on the rectangular problem:
 *   O_i = sum_j softmax_j(tau q_i . k_j) v_j,  LSE_i = ln sum_j exp(tau q_i . k_j),
 * over the visible keys j: all Nk, or with causal = 1 (the queries being the
 * last Nq positions of the sequence) j <= i + Nk - Nq.
 *
 * Q, O: bf16 [B,H,Nq,d]; K, V: bf16 [B,H,Nk,d]; LSE: fp32 [B,H,Nq]; all device
 * pointers, contiguous, 16-byte aligned.  1 <= Nq <= 8 (else
 * FA_ERR_UNSUPPORTED); Nk >= 1, and Nq <= Nk when causal (else
 * FA_ERR_INVALID_ARG); d in {64, 128}.  The KV cache is cut into chunks
 * processed in parallel; their partial results go to `workspace`, which needs
 * fa_decode_workspace_size(B, H, Nq, Nk, d) bytes (0 when one chunk suffices;
 * NULL: the call takes it with cudaMallocAsync on `stream` and frees it with
 * cudaFreeAsync).  Asynchronous on `stream`.
 */
FA_API size_t fa_decode_workspace_size(int B, int H, int Nq, int Nk, int d);
FA_API fa_status fa_fwd_decode(const void* Q, const void* K, const void* V, void* O, float* LSE,
                               int B, int H, int Nq, int Nk, int d, float tau, int causal,
                               void* workspace, size_t workspace_bytes, void* stream);

/*
 * FP8 forward ("Atencao eficiente - FlashAttention, sparse e hibrida", the
 * FlashAttention-4 note: FlashAttention-3 added FP8 for Hopper).  Q, K, V are
 * e4m3 (OCP FP8 E4M3: 1 sign, 4 exponent bits with bias 7, 3 mantissa bits,
 * no infinities, max 448) stored one byte per element, [B,H,N,d] contiguous,
 * with one scale per tensor: the value of element x is x * scale.  Computes
 * the attention of those values, O = softmax(tau (sq Q)(sk K)^T [causal])
 * (sv V), with both products on FP8 tensor cores; the softmax numerator is
 * rounded to e4m3 before the second product, which is what limits accuracy
 * (O agrees with the exact result to about 1e-2 relative; LSE, computed from
 * the unrounded numerator, to about 1e-3).  O: bf16 [B,H,N,d]; LSE: fp32
 * [B,H,N], natural log.  d = 128 only (else FA_ERR_UNSUPPORTED); scales finite
 * and > 0 (else FA_ERR_INVALID_ARG).  Other conventions as fa_fwd.
 */
FA_API fa_status fa_fwd_fp8(const void* Q, const void* K, const void* V, void* O, float* LSE,
                            int B, int H, int N, int d, float tau, int causal, float q_scale,
                            float k_scale, float v_scale, void* stream);

/*
 * Kernel timing hook.  With both events non-NULL (cudaEvent_t created by the
 * caller), every later forward or backward call made from the
 * calling host thread records `start` on its stream right before the
 * attention kernel proper (the forward kernel; the backward's main kernel,
 * after its D/zeroing pre-kernel) and `stop` right after it, so the caller
 * can read that kernel's duration with cudaEventElapsedTime.  NULL, NULL
 * turns it off.  The events stay owned by the caller.  Not part of the
 * method: a measurement aid.
 */
FA_API fa_status fa_set_timing_events(void* start, void* stop);

/*
 * Backward pass that allocates nothing.
 *
 * The pages have no counterpart for this entry point; it exists for callers
 * that are not allowed to allocate device memory while they run: hosts that
 * reserve a fixed memory budget up front and forbid libraries from calling
 * cudaMalloc or cudaMallocAsync later (inference servers, plugins inside a
 * framework that owns every allocation, latency-bound loops where an
 * allocation could stall or fail).  Such a caller cannot pass a NULL
 * workspace to fa_bwd, and may have no spare buffer to lend it either.
 *
 * It computes exactly what fa_bwd computes (same arguments, minus the
 * workspace), using as scratch a fixed array of FA_NOALLOC_SCRATCH_BYTES that
 * lives in the library's device image.  Every GPU on which the library is
 * used holds that array until the process exits.  The problem must satisfy
 * fa_bwd_workspace_size(B, H, N, d) <= FA_NOALLOC_SCRATCH_BYTES, otherwise
 * the call returns FA_ERR_WORKSPACE before doing anything.  The call makes no
 * cudaMalloc/cudaFree (or any other allocating) call.
 *
 * The first call on a device looks up the array's device address (with that
 * device current) and keeps it; make that first call before any stream
 * capture begins.  A lookup that fails returns FA_ERR_CUDA and is retried on
 * the next call.  On a device other than sm_103 the call returns
 * FA_ERR_UNSUPPORTED, as every other entry point does.  All calls share the one array and it keeps the previous
 * call's contents (the kernels clear what must start at zero), so two calls
 * whose work overlaps on the GPU (different streams, or different host
 * threads, on the same device) race on it and give wrong results: order them.
 */
#define FA_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)
FA_API fa_status fa_bwd_noalloc(const void* Q, const void* K, const void* V, const void* O,
                                const void* dO, const float* LSE, void* dQ, void* dK, void* dV,
                                int B, int H, int N, int d, float tau, int causal, void* stream);

/*
 * Host-buffer pipeline: forward + backward steps on tensors that live in host
 * memory.  Not part of the method (the pages describe device-resident
 * tensors); it is the runtime a caller with host-resident batches uses, and
 * the library's end-to-end measurement goes through it.
 *
 * fa_host_pipeline_create allocates `depth` (1..8) device buffer sets for one
 * problem shape (Q, K, V, dO, O, LSE, dQ, dK, dV and the backward workspace,
 * on the current device; the only allocations the library makes on its own,
 * owned by the object until fa_host_pipeline_destroy) and two copy streams.
 * The kernels run on `stream` (NULL = the legacy default stream).
 *
 * fa_host_pipeline_step enqueues one step and returns: copy hQ, hK, hV, hdO
 * (host, bf16 [B][H][N][d]) in; fa_fwd and fa_bwd on the next buffer set; copy
 * O, LSE (fp32 [B][H][N]), dQ, dK, dV out to hO, hLSE, hdQ, hdK, hdV.  Events
 * order each set's reuse, so with depth >= 2 the copies of neighbouring steps
 * overlap the kernels.  Host buffers should be page-locked (cudaHostAlloc /
 * pinned): pageable memory works but its copies do not overlap.  The caller
 * must not touch a step's host buffers until that step has finished
 * (fa_host_pipeline_sync, or an event from fa_host_pipeline_mark).
 *
 * fa_host_pipeline_mark records `event` (a cudaEvent_t) on `stream` at a point
 * after everything enqueued so far, copies included, and makes every copy
 * enqueued later wait for it: two marks bracket whole steps for timing.
 * fa_host_pipeline_sync blocks the host until all enqueued work is done.
 * fa_host_pipeline_destroy synchronises, then frees everything (NULL is a
 * no-op).  An object is not thread-safe; use one per host thread.
 * Errors: FA_ERR_INVALID_ARG (null pointers, bad sizes or depth),
 * FA_ERR_UNSUPPORTED (d not 64 or 128), FA_ERR_CUDA (an allocation or CUDA
 * call failed), and whatever fa_fwd / fa_bwd return.
 */
typedef struct fa_host_pipeline fa_host_pipeline;
FA_API fa_status fa_host_pipeline_create(int B, int H, int N, int d, float tau, int causal,
                                         int depth, void* stream, fa_host_pipeline** out);
FA_API fa_status fa_host_pipeline_step(fa_host_pipeline* p, const void* hQ, const void* hK,
                                       const void* hV, const void* hdO, void* hO, float* hLSE,
                                       void* hdQ, void* hdK, void* hdV);
FA_API fa_status fa_host_pipeline_mark(fa_host_pipeline* p, void* event);
FA_API fa_status fa_host_pipeline_sync(fa_host_pipeline* p);
FA_API fa_status fa_host_pipeline_destroy(fa_host_pipeline* p);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_FA_H */
