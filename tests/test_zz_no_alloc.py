"""fa_bwd_noalloc: the backward for callers that may not allocate device
memory while they run (fixed-budget servers, plugins whose host framework owns
all allocations).  It must give what fa_bwd gives and what the oracle gives,
call after call, while using only the library's fixed scratch array, and it
must not allocate.

The allocation check reads the high-water mark of the device's current
stream-ordered memory pool (the pool cudaMallocAsync draws from) through the
CUDA driver API: reset to zero, run the calls, read it back.  fa_bwd with a
NULL workspace, which does take its workspace from that pool, is the positive
control that shows the check can see an allocation.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test."""
import ctypes
import math

import pytest
import torch

import oracle
from exact_io_aware_12_gb300 import _lib, api
from exact_io_aware_12_gb300.workloads import draw
from tests._parity import check_grad

pytestmark = pytest.mark.gpu

CU_MEMPOOL_ATTR_USED_MEM_HIGH = 8   # CUmemPool_attribute, cuda.h


def _noalloc(q, k, v, o, do, lse, causal, tau):
    B, H, N, d = q.shape
    dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
    code = _lib.fa_bwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                               do.data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                               dv.data_ptr(), B, H, N, d, tau, int(causal),
                               torch.cuda.current_stream().cuda_stream)
    return code, dq, dk, dv


class _PoolHighWater:
    """High-water mark of the current device's current memory pool."""

    def __init__(self):
        self.cu = ctypes.CDLL("libcuda.so.1")
        dev = ctypes.c_int()
        assert self.cu.cuDeviceGet(ctypes.byref(dev), torch.cuda.current_device()) == 0
        self.pool = ctypes.c_void_p()
        assert self.cu.cuDeviceGetMemPool(ctypes.byref(self.pool), dev) == 0

    def reset(self):
        zero = ctypes.c_uint64(0)
        assert self.cu.cuMemPoolSetAttribute(self.pool, CU_MEMPOOL_ATTR_USED_MEM_HIGH,
                                             ctypes.byref(zero)) == 0

    def read(self) -> int:
        v = ctypes.c_uint64(0)
        assert self.cu.cuMemPoolGetAttribute(self.pool, CU_MEMPOOL_ATTR_USED_MEM_HIGH,
                                             ctypes.byref(v)) == 0
        return int(v.value)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("B,H,N,d", [(1, 3, 300, 64), (2, 2, 520, 128)])
def test_noalloc_matches_fa_bwd_and_the_oracle_on_two_calls_in_a_row(B, H, N, d, causal):
    x = draw(B, H, N, d, seed=900 + N + d)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    tau = 1 / math.sqrt(d)
    assert _lib.fa_bwd_workspace_size(B, H, N, d) <= _lib.NOALLOC_SCRATCH_BYTES
    o, lse = api.fwd(q, k, v, causal, tau)
    rq, rk, rv = api.bwd(q, k, v, o, do, lse, causal, tau)     # the existing entry point
    gq, gk, gv = oracle.bwd(x["q"], x["k"], x["v"], x["do"], tau, causal)
    for call in range(2):                                      # the scratch is reused
        code, dq, dk, dv = _noalloc(q, k, v, o, do, lse, causal, tau)
        assert code == _lib.FA_OK, _lib.status_string(code)
        torch.cuda.synchronize()
        assert api.last_device_error() == _lib.FA_OK
        for got, same, ref, name in ((dq, rq, gq, "dQ"), (dk, rk, gk, "dK"), (dv, rv, gv, "dV")):
            check_grad(got, same, f"{name} vs fa_bwd (call {call})")
            check_grad(got, ref, f"{name} vs oracle (call {call})")


def test_noalloc_allocates_nothing():
    B, H, N, d, causal = 1, 2, 384, 128, True
    x = draw(B, H, N, d, seed=77)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    tau = 1 / math.sqrt(d)
    o, lse = api.fwd(q, k, v, causal, tau)
    hw = _PoolHighWater()
    _noalloc(q, k, v, o, do, lse, causal, tau)                 # the first call's one-time lookup
    torch.cuda.synchronize()

    # positive control: a NULL workspace makes fa_bwd allocate from the pool
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    stream = torch.cuda.current_stream().cuda_stream
    hw.reset()
    code = _lib.fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(),
                       lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), None, 0,
                       B, H, N, d, tau, int(causal), stream)
    assert code == _lib.FA_OK
    torch.cuda.synchronize()
    assert hw.read() >= _lib.fa_bwd_workspace_size(B, H, N, d), "the check cannot see allocations"

    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    torch_before = torch.cuda.memory_allocated()
    hw.reset()
    for _ in range(2):
        code = _lib.fa_bwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                   do.data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                                   dv.data_ptr(), B, H, N, d, tau, int(causal), stream)
        assert code == _lib.FA_OK
    torch.cuda.synchronize()
    assert hw.read() == 0, "fa_bwd_noalloc took memory from the stream-ordered pool"
    assert torch.cuda.memory_allocated() == torch_before
    assert api.last_device_error() == _lib.FA_OK


def test_noalloc_rejects_problems_beyond_its_scratch():
    B, H, N, d = 1, 64, 4096, 128          # needs ~129 MiB of scratch
    assert _lib.fa_bwd_workspace_size(B, H, N, d) > _lib.NOALLOC_SCRATCH_BYTES
    q = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(16, dtype=torch.float32, device="cuda")
    p = q.data_ptr()
    code = _lib.fa_bwd_noalloc(p, p, p, p, p, lse.data_ptr(), p, p, p, B, H, N, d, 0.088, 1,
                               torch.cuda.current_stream().cuda_stream)
    assert code == _lib.FA_ERR_WORKSPACE
