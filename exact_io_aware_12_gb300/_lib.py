"""ctypes binding of the C ABI in include/fa.h (names and arguments as in C).

Only argument marshalling happens here: every step of the computation runs in
the CUDA kernels of ``_build/libfa_gb300.so``.  There is no fallback: if the
library cannot be built or loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import threading

from . import build as _build

FA_OK = 0
FA_ERR_INVALID_ARG = 1
FA_ERR_UNSUPPORTED = 2
FA_ERR_WORKSPACE = 3
FA_ERR_CUDA = 4
FA_ERR_TIMEOUT = 5

# (name, restype, argtypes) for every entry point declared in include/fa.h
_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_SZ = ctypes.c_size_t
_ULL = ctypes.c_ulonglong
SIGNATURES = {
    "fa_fwd": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _I, _P]),
    "fa_fwd_o32": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _I, _P]),
    "fa_bwd_workspace_size": (_SZ, [_I, _I, _I, _I]),
    "fa_bwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _I, _I, _I, _I, _F, _I, _P]),
    "fa_status_string": (ctypes.c_char_p, [_I]),
    "fa_last_device_error": (_I, [_P]),
    "fa_set_wait_limit_ns": (_I, [_ULL]),
    "fa_watchdog_selftest": (_I, [_ULL, _P]),
    "fa_set_timing_events": (_I, [_P, _P]),
    "fa_fwd_window": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _I, _P]),
    "fa_bwd_window": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _I, _I, _I, _I, _F, _I, _P]),
    "fa_bwd_noalloc": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _I, _P]),
    "fa_fwd_fp8": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _I, _F, _F, _F, _P]),
    "fa_decode_workspace_size": (_SZ, [_I, _I, _I, _I, _I]),
    "fa_fwd_decode": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _P, _SZ, _P]),
    "fa_fwd_blocks": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _I, _P, _I, _P]),
    "fa_bwd_blocks": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _I, _I, _I, _I, _F, _I,
                           _P, _I, _P]),
    "fa_host_pipeline_create": (_I, [_I, _I, _I, _I, _F, _I, _I, _P, ctypes.POINTER(_P)]),
    "fa_host_pipeline_step": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "fa_host_pipeline_mark": (_I, [_P, _P]),
    "fa_host_pipeline_sync": (_I, [_P]),
    "fa_host_pipeline_destroy": (_I, [_P]),
}

# Block-mask geometry (FA_BLOCK_MASK_EDGE, FA_BLOCK_MASK_MAX_N).
BLOCK_MASK_EDGE = 128
BLOCK_MASK_MAX_N = 131072

# Size of the fixed scratch array fa_bwd_noalloc uses (FA_NOALLOC_SCRATCH_BYTES).
NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024

_lock = threading.Lock()
_lib = None


class FAError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {status_string(code)} (code {code})")


def load() -> ctypes.CDLL:
    """Load the library, building it first if it is missing or stale."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build()
            lib = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
        return _lib


def library_path() -> str:
    return _build.LIB_PATH


def status_string(code: int) -> str:
    return load().fa_status_string(int(code)).decode()


def _call(name: str, *args) -> int:
    return getattr(load(), name)(*args)


def fa_fwd(Q, K, V, O, LSE, B, H, N, d, tau, causal, stream) -> int:
    return _call("fa_fwd", Q, K, V, O, LSE, B, H, N, d, tau, causal, stream)


def fa_fwd_o32(Q, K, V, O, LSE, B, H, N, d, tau, causal, stream) -> int:
    return _call("fa_fwd_o32", Q, K, V, O, LSE, B, H, N, d, tau, causal, stream)


def fa_fwd_window(Q, K, V, O, LSE, B, H, N, d, tau, window, stream) -> int:
    return _call("fa_fwd_window", Q, K, V, O, LSE, B, H, N, d, tau, window, stream)


def fa_bwd_window(Q, K, V, O, dO, LSE, dQ, dK, dV, workspace, workspace_bytes, B, H, N, d, tau,
                  window, stream) -> int:
    return _call("fa_bwd_window", Q, K, V, O, dO, LSE, dQ, dK, dV, workspace, workspace_bytes, B,
                 H, N, d, tau, window, stream)


def fa_fwd_fp8(Q, K, V, O, LSE, B, H, N, d, tau, causal, q_scale, k_scale, v_scale, stream) -> int:
    return _call("fa_fwd_fp8", Q, K, V, O, LSE, B, H, N, d, tau, causal, q_scale, k_scale, v_scale,
                 stream)


def fa_decode_workspace_size(B, H, Nq, Nk, d) -> int:
    return int(_call("fa_decode_workspace_size", B, H, Nq, Nk, d))


def fa_fwd_decode(Q, K, V, O, LSE, B, H, Nq, Nk, d, tau, causal, workspace, workspace_bytes,
                  stream) -> int:
    return _call("fa_fwd_decode", Q, K, V, O, LSE, B, H, Nq, Nk, d, tau, causal, workspace,
                 workspace_bytes, stream)


def fa_fwd_blocks(Q, K, V, O, LSE, B, H, N, d, tau, causal, block_mask, mask_heads, stream) -> int:
    return _call("fa_fwd_blocks", Q, K, V, O, LSE, B, H, N, d, tau, causal, block_mask, mask_heads,
                 stream)


def fa_bwd_blocks(Q, K, V, O, dO, LSE, dQ, dK, dV, workspace, workspace_bytes, B, H, N, d, tau,
                  causal, block_mask, mask_heads, stream) -> int:
    return _call("fa_bwd_blocks", Q, K, V, O, dO, LSE, dQ, dK, dV, workspace, workspace_bytes, B,
                 H, N, d, tau, causal, block_mask, mask_heads, stream)


def fa_bwd_workspace_size(B, H, N, d) -> int:
    return int(_call("fa_bwd_workspace_size", B, H, N, d))


def fa_bwd(Q, K, V, O, dO, LSE, dQ, dK, dV, workspace, workspace_bytes, B, H, N, d, tau, causal,
           stream) -> int:
    return _call("fa_bwd", Q, K, V, O, dO, LSE, dQ, dK, dV, workspace, workspace_bytes, B, H, N,
                 d, tau, causal, stream)


def fa_status_string(code) -> str:
    return status_string(code)


def fa_last_device_error(stream) -> int:
    return _call("fa_last_device_error", stream)


def fa_set_wait_limit_ns(ns) -> int:
    return _call("fa_set_wait_limit_ns", ns)


def fa_watchdog_selftest(limit_ns, stream) -> int:
    return _call("fa_watchdog_selftest", limit_ns, stream)


def fa_set_timing_events(start, stop) -> int:
    return _call("fa_set_timing_events", start, stop)


def fa_bwd_noalloc(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N, d, tau, causal, stream) -> int:
    """fa_bwd without any device allocation, for callers that may not allocate
    while running; its scratch is a fixed array inside the library."""
    return _call("fa_bwd_noalloc", Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N, d, tau, causal,
                 stream)


def check(code: int, where: str) -> None:
    if code != FA_OK:
        raise FAError(code, where)


def fa_host_pipeline_create(B, H, N, d, tau, causal, depth, stream):
    """Returns (status, handle)."""
    h = ctypes.c_void_p()
    code = _call("fa_host_pipeline_create", B, H, N, d, tau, causal, depth, stream, ctypes.byref(h))
    return code, h


def fa_host_pipeline_step(p, hQ, hK, hV, hdO, hO, hLSE, hdQ, hdK, hdV) -> int:
    return _call("fa_host_pipeline_step", p, hQ, hK, hV, hdO, hO, hLSE, hdQ, hdK, hdV)


def fa_host_pipeline_mark(p, event) -> int:
    return _call("fa_host_pipeline_mark", p, event)


def fa_host_pipeline_sync(p) -> int:
    return _call("fa_host_pipeline_sync", p)


def fa_host_pipeline_destroy(p) -> int:
    return _call("fa_host_pipeline_destroy", p)
