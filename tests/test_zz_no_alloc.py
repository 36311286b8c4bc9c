"""fa_bwd_noalloc: the backward for callers that may not allocate device
memory while they run (fixed-budget servers, plugins whose host framework owns
all allocations).  It must give what fa_bwd gives, call after call, while
using only the library's fixed scratch array.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test."""
import math

import pytest
import torch

from exact_io_aware_12_gb300 import _lib, api
from exact_io_aware_12_gb300.workloads import draw
from tests._parity import check_grad

pytestmark = pytest.mark.gpu


def _noalloc(q, k, v, o, do, lse, causal, tau):
    B, H, N, d = q.shape
    dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
    code = _lib.fa_bwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                               do.data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                               dv.data_ptr(), B, H, N, d, tau, int(causal),
                               torch.cuda.current_stream().cuda_stream)
    return code, dq, dk, dv


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("B,H,N,d", [(1, 3, 300, 64), (2, 2, 520, 128)])
def test_noalloc_matches_fa_bwd_on_two_calls_in_a_row(B, H, N, d, causal):
    x = draw(B, H, N, d, seed=900 + N + d)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    tau = 1 / math.sqrt(d)
    assert _lib.fa_bwd_workspace_size(B, H, N, d) <= _lib.NOALLOC_SCRATCH_BYTES
    o, lse = api.fwd(q, k, v, causal, tau)
    rq, rk, rv = api.bwd(q, k, v, o, do, lse, causal, tau)     # the existing entry point
    for call in range(2):                                      # the scratch is reused
        code, dq, dk, dv = _noalloc(q, k, v, o, do, lse, causal, tau)
        assert code == _lib.FA_OK, _lib.status_string(code)
        torch.cuda.synchronize()
        assert api.last_device_error() == _lib.FA_OK
        check_grad(dq, rq, f"dQ (call {call})")
        check_grad(dk, rk, f"dK (call {call})")
        check_grad(dv, rv, f"dV (call {call})")


def test_noalloc_rejects_problems_beyond_its_scratch():
    B, H, N, d = 1, 64, 4096, 128          # needs ~129 MiB of scratch
    assert _lib.fa_bwd_workspace_size(B, H, N, d) > _lib.NOALLOC_SCRATCH_BYTES
    q = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(16, dtype=torch.float32, device="cuda")
    p = q.data_ptr()
    code = _lib.fa_bwd_noalloc(p, p, p, p, p, lse.data_ptr(), p, p, p, B, H, N, d, 0.088, 1,
                               torch.cuda.current_stream().cuda_stream)
    assert code == _lib.FA_ERR_WORKSPACE
