"""Torch-facing helpers over the C ABI.

PyTorch only supplies device memory and the current stream; the tensors'
data pointers go straight to ``fa_fwd`` / ``fa_bwd``.  Inputs must be CUDA
bf16 tensors, contiguous, shaped [B, H, N, d].
"""
from __future__ import annotations

import math
from typing import Optional, Tuple

import torch

from . import _lib


def _stream_handle(device: torch.device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _check_inputs(*ts: torch.Tensor) -> Tuple[int, int, int, int]:
    ref = ts[0]
    if ref.dim() != 4:
        raise ValueError("expected [B, H, N, d] tensors")
    for t in ts:
        if not t.is_cuda or t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError("inputs must be contiguous CUDA bf16 tensors")
        if t.shape != ref.shape or t.device != ref.device:
            raise ValueError("inputs must share shape and device")
    B, H, N, d = ref.shape
    return B, H, N, d


def _check_blocks(blocks: torch.Tensor, ref: torch.Tensor) -> int:
    """A block mask: CUDA uint8/bool, contiguous, shaped [nb, nb] (one mask) or
    [B, H, nb, nb] / [B*H, nb, nb] (one per head), nb = ceil(N / 128).
    Returns mask_heads."""
    B, H, N, _ = ref.shape
    nb = (N + _lib.BLOCK_MASK_EDGE - 1) // _lib.BLOCK_MASK_EDGE
    if not blocks.is_cuda or blocks.device != ref.device or not blocks.is_contiguous():
        raise ValueError("block mask must be a contiguous tensor on the inputs' device")
    if blocks.dtype not in (torch.uint8, torch.bool):
        raise ValueError("block mask must be uint8 or bool")
    if tuple(blocks.shape[-2:]) != (nb, nb):
        raise ValueError(f"block mask must end in ({nb}, {nb})")
    heads = blocks.numel() // (nb * nb)
    if blocks.dim() == 2:
        return 1
    if heads != B * H:
        raise ValueError(f"block mask has {heads} heads, expected 1 or {B * H}")
    return heads


def fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool,
        tau: Optional[float] = None, out: Optional[torch.Tensor] = None,
        lse: Optional[torch.Tensor] = None, o_fp32: bool = False, window: Optional[int] = None,
        blocks: Optional[torch.Tensor] = None):
    """Forward pass.  Returns (O, LSE): O bf16 (fp32 with ``o_fp32``) and LSE
    fp32 [B, H, N].  ``window`` (with ``causal``): each query sees only its
    ``window`` most recent keys (fa_fwd_window).  ``blocks``: a block mask
    over 128 x 128 blocks (fa_fwd_blocks)."""
    if window is not None and (not causal or o_fp32):
        raise ValueError("a window needs causal=True and a bf16 O")
    if blocks is not None and (o_fp32 or window is not None):
        raise ValueError("a block mask needs a bf16 O and no window")
    B, H, N, d = _check_inputs(q, k, v)
    tau = 1.0 / math.sqrt(d) if tau is None else float(tau)
    o_dtype = torch.float32 if o_fp32 else torch.bfloat16
    if out is None:
        out = torch.empty(q.shape, dtype=o_dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if blocks is not None:
        heads = _check_blocks(blocks, q)
        code = _lib.fa_fwd_blocks(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                  lse.data_ptr(), B, H, N, d, tau, int(bool(causal)),
                                  blocks.data_ptr(), heads, _stream_handle(q.device))
        _lib.check(code, "fa_fwd_blocks")
        return out, lse
    if window is not None:
        code = _lib.fa_fwd_window(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                  lse.data_ptr(), B, H, N, d, tau, int(window),
                                  _stream_handle(q.device))
        _lib.check(code, "fa_fwd_window")
        return out, lse
    fn = _lib.fa_fwd_o32 if o_fp32 else _lib.fa_fwd
    code = fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
              B, H, N, d, tau, int(bool(causal)), _stream_handle(q.device))
    _lib.check(code, "fa_fwd_o32" if o_fp32 else "fa_fwd")
    return out, lse


def workspace_bytes(B: int, H: int, N: int, d: int) -> int:
    return _lib.fa_bwd_workspace_size(B, H, N, d)


def bwd(q, k, v, o, do, lse, causal: bool, tau: Optional[float] = None,
        dq: Optional[torch.Tensor] = None, dk: Optional[torch.Tensor] = None,
        dv: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
        window: Optional[int] = None, blocks: Optional[torch.Tensor] = None):
    """Backward pass.  Returns (dQ, dK, dV), bf16.  ``workspace`` (a byte
    tensor of at least ``workspace_bytes`` bytes) is allocated with torch when
    not given, so the library itself allocates nothing."""
    B, H, N, d = _check_inputs(q, k, v, o, do)
    if lse.dtype != torch.float32 or not lse.is_contiguous() or lse.shape != (B, H, N):
        raise ValueError("lse must be contiguous fp32 [B, H, N]")
    tau = 1.0 / math.sqrt(d) if tau is None else float(tau)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    need = workspace_bytes(B, H, N, d)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    if blocks is not None:
        if window is not None:
            raise ValueError("a block mask needs no window")
        heads = _check_blocks(blocks, q)
        code = _lib.fa_bwd_blocks(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                  do.data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                                  dv.data_ptr(), workspace.data_ptr(), workspace.numel(), B, H, N,
                                  d, tau, int(bool(causal)), blocks.data_ptr(), heads,
                                  _stream_handle(q.device))
        _lib.check(code, "fa_bwd_blocks")
        return dq, dk, dv
    if window is not None:
        if not causal:
            raise ValueError("a window needs causal=True")
        code = _lib.fa_bwd_window(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                  do.data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                                  dv.data_ptr(), workspace.data_ptr(), workspace.numel(), B, H, N,
                                  d, tau, int(window), _stream_handle(q.device))
        _lib.check(code, "fa_bwd_window")
        return dq, dk, dv
    code = _lib.fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(),
                       lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                       workspace.data_ptr(), workspace.numel(), B, H, N, d, tau,
                       int(bool(causal)), _stream_handle(q.device))
    _lib.check(code, "fa_bwd")
    return dq, dk, dv


def fwd_fp8(q8: torch.Tensor, k8: torch.Tensor, v8: torch.Tensor, q_scale: float, k_scale: float,
            v_scale: float, causal: bool, tau: Optional[float] = None,
            out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None):
    """FP8 forward (fa_fwd_fp8): q8, k8, v8 hold e4m3 bytes (uint8 or
    float8_e4m3fn tensors, contiguous, [B, H, N, 128]) whose values are
    byte * scale.  Returns (O bf16 [B, H, N, 128], LSE fp32 [B, H, N])."""
    ts = (q8, k8, v8)
    for t in ts:
        if not t.is_cuda or t.element_size() != 1 or not t.is_contiguous() or t.dim() != 4:
            raise ValueError("q8, k8, v8 must be contiguous CUDA [B, H, N, d] 1-byte tensors")
        if t.shape != q8.shape or t.device != q8.device:
            raise ValueError("q8, k8, v8 must share shape and device")
    B, H, N, d = q8.shape
    tau = 1.0 / math.sqrt(d) if tau is None else float(tau)
    if out is None:
        out = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=q8.device)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q8.device)
    code = _lib.fa_fwd_fp8(q8.data_ptr(), k8.data_ptr(), v8.data_ptr(), out.data_ptr(),
                           lse.data_ptr(), B, H, N, d, tau, int(bool(causal)), float(q_scale),
                           float(k_scale), float(v_scale), _stream_handle(q8.device))
    _lib.check(code, "fa_fwd_fp8")
    return out, lse


def decode_workspace_bytes(B: int, H: int, Nq: int, Nk: int, d: int) -> int:
    return _lib.fa_decode_workspace_size(B, H, Nq, Nk, d)


def fwd_decode(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool,
               tau: Optional[float] = None, out: Optional[torch.Tensor] = None,
               lse: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None):
    """Decode forward (fa_fwd_decode): q [B, H, Nq, d] (1 <= Nq <= 8) against
    the KV cache k, v [B, H, Nk, d]; with ``causal`` the queries are the last Nq
    positions.  Returns (O bf16 [B, H, Nq, d], LSE fp32 [B, H, Nq]).  The
    split workspace is allocated with torch when not given."""
    if q.dim() != 4:
        raise ValueError("expected [B, H, Nq, d] queries")
    B, H, Nq, d = q.shape
    _check_inputs(k, v)
    for t in (q, k, v):
        if not t.is_cuda or t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError("inputs must be contiguous CUDA bf16 tensors")
    if k.shape[:2] != (B, H) or k.shape[3] != d or k.device != q.device:
        raise ValueError("k, v must be [B, H, Nk, d] on q's device")
    Nk = k.shape[2]
    tau = 1.0 / math.sqrt(d) if tau is None else float(tau)
    if out is None:
        out = torch.empty(q.shape, dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    need = decode_workspace_bytes(B, H, Nq, Nk, d)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    wp, wn = (workspace.data_ptr(), workspace.numel()) if workspace is not None else (None, 0)
    code = _lib.fa_fwd_decode(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                              lse.data_ptr(), B, H, Nq, Nk, d, tau, int(bool(causal)), wp, wn,
                              _stream_handle(q.device))
    _lib.check(code, "fa_fwd_decode")
    return out, lse


def last_device_error(device: Optional[torch.device] = None) -> int:
    device = device or torch.device("cuda", torch.cuda.current_device())
    return _lib.fa_last_device_error(_stream_handle(device))


class _Attention(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, causal, tau):
        o, lse = fwd(q, k, v, causal, tau)
        ctx.save_for_backward(q, k, v, o, lse)
        ctx.causal, ctx.tau = causal, tau
        return o

    @staticmethod
    def backward(ctx, do):
        q, k, v, o, lse = ctx.saved_tensors
        dq, dk, dv = bwd(q, k, v, o, do.contiguous(), lse, ctx.causal, ctx.tau)
        return dq, dk, dv, None, None


def attention(q, k, v, causal: bool = False, tau: Optional[float] = None) -> torch.Tensor:
    """O = softmax(tau Q K^T [causal]) V with autograd support."""
    return _Attention.apply(q, k, v, causal, tau)


class HostPipeline:
    """Forward + backward steps on tensors that live in pinned host memory,
    through the library's native host pipeline (fa_host_pipeline_* in
    include/fa.h).

    Each step copies its Q, K, V, dO in, runs fwd and bwd, and copies O, LSE,
    dQ, dK, dV back out.  The library owns ``depth`` device buffer sets
    (default 2) and one stream per copy direction; the kernels run on the
    caller's current stream.  The copies of neighbouring steps overlap each
    other's kernels, as a training or serving loop overlaps the next batch's
    transfer with the current step.  ``step`` only enqueues work;
    ``synchronize`` waits for all of it.  Host tensors must be pinned,
    contiguous, of the configured shape (bf16; LSE fp32), and must not be
    touched until the step has finished."""

    def __init__(self, B: int, H: int, N: int, d: int, causal: bool, tau: Optional[float] = None,
                 device: Optional[torch.device] = None, depth: int = 2):
        self.shape = (B, H, N, d)
        self.tau = 1.0 / math.sqrt(d) if tau is None else float(tau)
        self.device = device or torch.device("cuda", torch.cuda.current_device())
        self.stream = torch.cuda.current_stream(self.device)
        with torch.cuda.device(self.device):
            code, self._p = _lib.fa_host_pipeline_create(B, H, N, d, self.tau, int(bool(causal)),
                                                         int(depth), self.stream.cuda_stream)
        _lib.check(code, "fa_host_pipeline_create")

    def _check(self, ts, dtype, shape):
        for t in ts:
            if t.is_cuda or t.dtype != dtype or tuple(t.shape) != shape or not t.is_contiguous():
                raise ValueError(f"host tensors must be contiguous CPU {dtype} of shape {shape}")

    def step(self, q, k, v, do, o_out, lse_out, dq_out, dk_out, dv_out) -> None:
        self._check((q, k, v, do, o_out, dq_out, dk_out, dv_out), torch.bfloat16, self.shape)
        self._check((lse_out,), torch.float32, self.shape[:3])
        code = _lib.fa_host_pipeline_step(self._p, q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                          do.data_ptr(), o_out.data_ptr(), lse_out.data_ptr(),
                                          dq_out.data_ptr(), dk_out.data_ptr(), dv_out.data_ptr())
        _lib.check(code, "fa_host_pipeline_step")

    def mark(self) -> torch.cuda.Event:
        """A timing event on the kernels' stream after every step enqueued so
        far, copies included; copies enqueued later start after it."""
        e = torch.cuda.Event(enable_timing=True)
        e.record(self.stream)  # materialise the handle
        _lib.check(_lib.fa_host_pipeline_mark(self._p, e.cuda_event), "fa_host_pipeline_mark")
        return e

    def finish_event(self) -> torch.cuda.Event:
        return self.mark()

    def synchronize(self) -> None:
        _lib.check(_lib.fa_host_pipeline_sync(self._p), "fa_host_pipeline_sync")

    def close(self) -> None:
        if getattr(self, "_p", None) is not None and self._p.value:
            code = _lib.fa_host_pipeline_destroy(self._p)
            self._p = None
            _lib.check(code, "fa_host_pipeline_destroy")

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
