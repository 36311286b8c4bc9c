"""Plain fp64 CPU oracle for exact scaled-dot-product attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` import this package.  The product library
(``exact_io_aware_12_gb300``) never imports, links or calls it, and the two
share no code.

The arithmetic lives in ``ref_attn.c`` (plain C, fp64, no BLAS): the textbook
definition of attention and its analytic gradient.  This module only compiles
that file with gcc, loads it with ctypes and marshals numpy float64 arrays.

Every function takes arrays shaped ``[BH, N, d]`` (or ``[B, H, N, d]``; only
the trailing two axes matter) in float64, C-contiguous.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``,
``tests/test_oracle_window_pins.py``, ``tests/test_oracle_blocks_pins.py``,
``tests/test_oracle_decode_pins.py`` and ``tests/test_oracle_fp8_pins.py``
(closed forms, hand-worked golden values, finite differences, invariants,
brute force on tiny inputs and an independent transcription of the pages'
blocked loop).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ref_attn.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ref_attn.c into _build/liboracle.so (gcc, OpenMP, no fast-math)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-fno-fast-math", "-o", tmp, _SRC, "-lm"]
    subprocess.check_call(cmd)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        # FA_ORACLE_LIB lets the mutation test point the pins at a deliberately
        # broken copy of the oracle; it is never set otherwise.
        lib = ctypes.CDLL(os.environ.get("FA_ORACLE_LIB") or build())
        dp = ctypes.POINTER(ctypes.c_double)
        i64 = ctypes.c_int64
        lp = ctypes.POINTER(ctypes.c_int64)
        lib.ora_num_threads.restype = ctypes.c_int
        lib.ora_num_threads.argtypes = []
        lib.ora_set_num_threads.restype = None
        lib.ora_set_num_threads.argtypes = [ctypes.c_int]
        lib.ora_attn_probs.restype = None
        lib.ora_attn_probs.argtypes = [dp, dp, dp, i64, i64, i64, ctypes.c_double,
                                       ctypes.c_int, dp]
        lib.ora_attn_fwd.restype = None
        lib.ora_attn_fwd.argtypes = [dp, dp, dp, i64, i64, i64, ctypes.c_double,
                                     ctypes.c_int, dp, dp]
        lib.ora_attn_fwd_rows.restype = None
        lib.ora_attn_fwd_rows.argtypes = [dp, dp, dp, i64, i64, i64, ctypes.c_double,
                                          ctypes.c_int, lp, i64, dp, dp]
        lib.ora_attn_bwd.restype = None
        lib.ora_attn_bwd.argtypes = [dp, dp, dp, dp, i64, i64, i64, ctypes.c_double,
                                     ctypes.c_int, dp, dp, dp, dp, dp, dp]
        lib.ora_attn_probs_window.restype = None
        lib.ora_attn_probs_window.argtypes = [dp, dp, dp, i64, i64, i64, ctypes.c_double, i64, dp]
        lib.ora_attn_fwd_window.restype = None
        lib.ora_attn_fwd_window.argtypes = [dp, dp, dp, i64, i64, i64, ctypes.c_double, i64, dp, dp]
        lib.ora_attn_fwd_rows_window.restype = None
        lib.ora_attn_fwd_rows_window.argtypes = [dp, dp, dp, i64, i64, i64, ctypes.c_double, i64,
                                                 lp, i64, dp, dp]
        lib.ora_attn_bwd_window.restype = None
        lib.ora_attn_bwd_window.argtypes = [dp, dp, dp, dp, i64, i64, i64, ctypes.c_double, i64,
                                            dp, dp, dp, dp, dp, dp]
        u8 = ctypes.c_void_p
        ci = ctypes.c_int
        lib.ora_attn_probs_blocks.restype = None
        lib.ora_attn_probs_blocks.argtypes = [dp, dp, dp, i64, i64, i64, ctypes.c_double, ci,
                                              u8, i64, i64, dp]
        lib.ora_attn_fwd_blocks.restype = None
        lib.ora_attn_fwd_blocks.argtypes = [dp, dp, dp, i64, i64, i64, ctypes.c_double, ci,
                                            u8, i64, i64, dp, dp]
        lib.ora_attn_fwd_rows_blocks.restype = None
        lib.ora_attn_fwd_rows_blocks.argtypes = [dp, dp, dp, i64, i64, i64, ctypes.c_double, ci,
                                                 u8, i64, i64, lp, i64, dp, dp]
        lib.ora_attn_bwd_blocks.restype = None
        lib.ora_attn_bwd_blocks.argtypes = [dp, dp, dp, dp, i64, i64, i64, ctypes.c_double, ci,
                                            u8, i64, i64, dp, dp, dp, dp, dp, dp]
        lib.ora_e4m3_decode.restype = None
        lib.ora_e4m3_decode.argtypes = [ctypes.c_void_p, i64, dp]
        lib.ora_attn_fwd_decode.restype = None
        lib.ora_attn_fwd_decode.argtypes = [dp, dp, dp, i64, i64, i64, i64, ctypes.c_double,
                                            ctypes.c_int, dp, dp]
        _lib = lib
        return lib


def _f64(a) -> np.ndarray:
    """Accept numpy arrays or CPU torch tensors; return C-contiguous float64."""
    if hasattr(a, "detach"):
        a = a.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _dims(q: np.ndarray):
    if q.ndim < 2:
        raise ValueError("expected [..., N, d]")
    N, d = q.shape[-2], q.shape[-1]
    BH = int(np.prod(q.shape[:-2])) if q.ndim > 2 else 1
    return BH, N, d


def num_threads() -> int:
    return int(_load().ora_num_threads())


def set_num_threads(n: int) -> None:
    _load().ora_set_num_threads(int(n))


def _window(causal: bool, window):
    """window=None: no window.  Otherwise the causal sliding window of `window`
    keys (key j visible from query i iff i - window < j <= i)."""
    if window is None:
        return None
    if not causal or int(window) < 1:
        raise ValueError("a window needs causal=True and window >= 1")
    return int(window)


def _blocks(blocks, BH: int, N: int, blk: int, window):
    """blocks=None: no block mask.  Otherwise a block mask of blk x blk blocks,
    shaped [nb, nb] (one mask for every head) or [BH, nb, nb] / [B, H, nb, nb]
    (one per head), nb = ceil(N / blk); nonzero entries are visible blocks.
    Returns (uint8 array, mask_heads) or None."""
    if blocks is None:
        return None
    if window is not None:
        raise ValueError("a block mask and a window do not combine")
    if hasattr(blocks, "detach"):
        blocks = blocks.detach().to("cpu").numpy()
    m = np.ascontiguousarray(np.asarray(blocks) != 0, dtype=np.uint8)
    blk = int(blk)
    if blk < 1:
        raise ValueError("blk must be >= 1")
    nb = (N + blk - 1) // blk
    if m.shape[-2:] != (nb, nb):
        raise ValueError(f"block mask must end in ({nb}, {nb}), got {m.shape}")
    heads = int(np.prod(m.shape[:-2])) if m.ndim > 2 else 1
    if m.ndim > 2 and heads != BH:
        raise ValueError(f"block mask has {heads} heads, expected 1 or {BH}")
    return m, (1 if m.ndim == 2 else BH)


def probs(q, k, v, tau: float, causal: bool, window=None, blocks=None, blk: int = 128) -> np.ndarray:
    """Attention probabilities P, shape [..., N, N]."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    BH, N, d = _dims(q)
    P = np.empty(q.shape[:-1] + (N,), dtype=np.float64)
    w = _window(causal, window)
    bm = _blocks(blocks, BH, N, blk, window)
    if bm is not None:
        _load().ora_attn_probs_blocks(_ptr(q), _ptr(k), _ptr(v), BH, N, d, float(tau), int(causal),
                                      bm[0].ctypes.data, int(blk), bm[1], _ptr(P))
    elif w is None:
        _load().ora_attn_probs(_ptr(q), _ptr(k), _ptr(v), BH, N, d, float(tau), int(causal), _ptr(P))
    else:
        _load().ora_attn_probs_window(_ptr(q), _ptr(k), _ptr(v), BH, N, d, float(tau), w, _ptr(P))
    return P


def fwd(q, k, v, tau: float, causal: bool, window=None, blocks=None, blk: int = 128):
    """Full forward: returns (O [..., N, d], LSE [..., N])."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    BH, N, d = _dims(q)
    O = np.empty_like(q)
    L = np.empty(q.shape[:-1], dtype=np.float64)
    w = _window(causal, window)
    bm = _blocks(blocks, BH, N, blk, window)
    if bm is not None:
        _load().ora_attn_fwd_blocks(_ptr(q), _ptr(k), _ptr(v), BH, N, d, float(tau), int(causal),
                                    bm[0].ctypes.data, int(blk), bm[1], _ptr(O), _ptr(L))
    elif w is None:
        _load().ora_attn_fwd(_ptr(q), _ptr(k), _ptr(v), BH, N, d, float(tau), int(causal),
                             _ptr(O), _ptr(L))
    else:
        _load().ora_attn_fwd_window(_ptr(q), _ptr(k), _ptr(v), BH, N, d, float(tau), w,
                                    _ptr(O), _ptr(L))
    return O, L


def fwd_rows(q, k, v, tau: float, causal: bool, rows, window=None, blocks=None, blk: int = 128):
    """Forward on selected rows.

    ``rows`` holds flat row ids ``bh * N + i``.  Returns (O_rows [n, d],
    LSE_rows [n]).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    BH, N, d = _dims(q)
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    if r.size and (r.min() < 0 or r.max() >= BH * N):
        raise ValueError("row id out of range")
    O = np.empty((r.size, d), dtype=np.float64)
    L = np.empty((r.size,), dtype=np.float64)
    rp = r.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))
    w = _window(causal, window)
    bm = _blocks(blocks, BH, N, blk, window)
    if bm is not None:
        _load().ora_attn_fwd_rows_blocks(_ptr(q), _ptr(k), _ptr(v), BH, N, d, float(tau),
                                         int(causal), bm[0].ctypes.data, int(blk), bm[1],
                                         rp, r.size, _ptr(O), _ptr(L))
    elif w is None:
        _load().ora_attn_fwd_rows(_ptr(q), _ptr(k), _ptr(v), BH, N, d, float(tau), int(causal),
                                  rp, r.size, _ptr(O), _ptr(L))
    else:
        _load().ora_attn_fwd_rows_window(_ptr(q), _ptr(k), _ptr(v), BH, N, d, float(tau), w,
                                         rp, r.size, _ptr(O), _ptr(L))
    return O, L


def fwd_decode(q, k, v, tau: float, causal: bool):
    """Decode forward: q [..., Nq, d] against k, v [..., Nk, d] (same leading
    axes).  With causal, query i is position Nk - Nq + i and sees keys
    j <= i + Nk - Nq.  Returns (O [..., Nq, d], LSE [..., Nq])."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    BH, Nq, d = _dims(q)
    BHk, Nk, dk = _dims(k)
    if BHk != BH or dk != d or v.shape != k.shape:
        raise ValueError("q, k, v must share leading axes and d; k and v the same shape")
    if causal and Nq > Nk:
        raise ValueError("causal decode needs Nq <= Nk")
    O = np.empty_like(q)
    L = np.empty(q.shape[:-1], dtype=np.float64)
    _load().ora_attn_fwd_decode(_ptr(q), _ptr(k), _ptr(v), BH, Nq, Nk, d, float(tau), int(causal),
                                _ptr(O), _ptr(L))
    return O, L


def e4m3_to_f64(x) -> np.ndarray:
    """Decode e4m3 bytes (uint8 array or tensor, any shape) to float64."""
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").contiguous().view(-1).numpy().view(np.uint8).reshape(tuple(x.shape))
    b = np.ascontiguousarray(np.asarray(x), dtype=np.uint8)
    out = np.empty(b.shape, dtype=np.float64)
    _load().ora_e4m3_decode(b.ctypes.data, b.size, _ptr(out))
    return out


def fwd_fp8(q8, k8, v8, q_scale: float, k_scale: float, v_scale: float, tau: float,
            causal: bool, rows=None):
    """Forward of the FP8 inputs: the plain forward (or its row subset) of the
    decoded values x * scale."""
    q = e4m3_to_f64(q8) * float(q_scale)
    k = e4m3_to_f64(k8) * float(k_scale)
    v = e4m3_to_f64(v8) * float(v_scale)
    if rows is None:
        return fwd(q, k, v, tau, causal)
    return fwd_rows(q, k, v, tau, causal, rows)


def bwd(q, k, v, do, tau: float, causal: bool, want_fwd: bool = False, window=None,
        blocks=None, blk: int = 128):
    """Analytic backward.  Returns (dQ, dK, dV) or, with ``want_fwd``,
    (dQ, dK, dV, O, LSE, D) where D is the softmax-Jacobian row sum."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    BH, N, d = _dims(q)
    dQ, dK, dV = np.empty_like(q), np.empty_like(q), np.empty_like(q)
    null = ctypes.POINTER(ctypes.c_double)()
    if want_fwd:
        O = np.empty_like(q)
        L = np.empty(q.shape[:-1], dtype=np.float64)
        D = np.empty(q.shape[:-1], dtype=np.float64)
        po, pl, pd = _ptr(O), _ptr(L), _ptr(D)
    else:
        po = pl = pd = null
    w = _window(causal, window)
    bm = _blocks(blocks, BH, N, blk, window)
    if bm is not None:
        _load().ora_attn_bwd_blocks(_ptr(q), _ptr(k), _ptr(v), _ptr(do), BH, N, d, float(tau),
                                    int(causal), bm[0].ctypes.data, int(blk), bm[1],
                                    _ptr(dQ), _ptr(dK), _ptr(dV), po, pl, pd)
    elif w is None:
        _load().ora_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(do), BH, N, d, float(tau),
                             int(causal), _ptr(dQ), _ptr(dK), _ptr(dV), po, pl, pd)
    else:
        _load().ora_attn_bwd_window(_ptr(q), _ptr(k), _ptr(v), _ptr(do), BH, N, d, float(tau), w,
                                    _ptr(dQ), _ptr(dK), _ptr(dV), po, pl, pd)
    if want_fwd:
        return dQ, dK, dV, O, L, D
    return dQ, dK, dV
