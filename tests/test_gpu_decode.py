"""GPU parity of the decode forward (fa_fwd_decode) against the fp64 oracle.

Reading (oracle/ref_attn.c header): Nq query rows against Nk cached keys; with
causal the queries are the last Nq positions, so query i sees keys
j <= i + Nk - Nq.  Tolerances as the forward: O max-abs <= 1e-2 and rel-L2
<= 5e-3, LSE max-abs <= 1e-3.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_io_aware_12_gb300 import api, _lib
from exact_io_aware_12_gb300.workloads import DECODE_BY_NAME, draw, draw_decode
from tests._parity import check_lse, check_o, max_abs, np64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def gpu(x, causal, tau, **kw):
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    o, lse = api.fwd_decode(q, k, v, causal, tau, **kw)
    torch.cuda.synchronize()
    assert api.last_device_error() == _lib.FA_OK
    return o, lse


CASES = [(nq, nk) for nq in (1, 2, 3, 5, 8) for nk in (1, 2, 63, 64, 65, 700, 5000)] + \
        [(1, 70000), (4, 70001), (8, 40000)]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("Nq,Nk", CASES)
def test_decode_matches_oracle(Nq, Nk, d, causal):
    if causal and Nq > Nk:
        pytest.skip("causal decode needs Nq <= Nk")
    x = draw_decode(2, 2, Nq, Nk, d, seed=900 + Nq + Nk + d)
    tau = 1 / math.sqrt(d)
    o, lse = gpu(x, causal, tau)
    o_ref, l_ref = oracle.fwd_decode(x["q"], x["k"], x["v"], tau, causal)
    check_o(o, o_ref)
    check_lse(lse, l_ref)


@pytest.mark.parametrize("causal", [False, True])
def test_zero_queries_give_the_mean_of_visible_values(causal):
    Nq, Nk, d = 3, 5000, 128
    x = draw_decode(1, 2, Nq, Nk, d, seed=5)
    x["q"].zero_()
    o, lse = gpu(x, causal, 0.1)
    v = np64(x["v"])
    for i in range(Nq):
        n = Nk - Nq + i + 1 if causal else Nk
        check_o(o[:, :, i], v[:, :, :n].mean(2))
        assert max_abs(lse[:, :, i], np.full((1, 2), math.log(n))) <= 1e-3


def test_decode_equals_the_last_rows_of_the_square_forward():
    """The last Nq rows of a causal N x N forward are the decode of those rows."""
    N, d, Nq = 3000, 128, 4
    x = draw(1, 4, N, d, seed=6, with_do=False)
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    o_sq, l_sq = api.fwd(q, k, v, True)
    o, lse = api.fwd_decode(q[:, :, N - Nq:].contiguous(), k, v, True)
    torch.cuda.synchronize()
    assert (o.float() - o_sq[:, :, N - Nq:].float()).abs().max().item() <= 1e-2
    assert (lse - l_sq[:, :, N - Nq:]).abs().max().item() <= 1e-3


def test_workspace_given_or_taken_gives_the_same_result():
    Nq, Nk, d = 2, 20000, 64
    x = draw_decode(1, 3, Nq, Nk, d, seed=7)
    need = api.decode_workspace_bytes(1, 3, Nq, Nk, d)
    assert need > 0
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    a = gpu(x, False, 0.125, workspace=ws)
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    o, lse = torch.empty_like(q), torch.empty(1, 3, Nq, device=DEV)
    s = torch.cuda.current_stream().cuda_stream
    _lib.check(_lib.fa_fwd_decode(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                  lse.data_ptr(), 1, 3, Nq, Nk, d, 0.125, 0, None, 0, s), "decode")
    torch.cuda.synchronize()
    assert torch.equal(a[0], o) and torch.equal(a[1], lse)
    code = _lib.fa_fwd_decode(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                              lse.data_ptr(), 1, 3, Nq, Nk, d, 0.125, 0, ws.data_ptr(), need - 1, s)
    assert code == _lib.FA_ERR_WORKSPACE


def test_bad_arguments_are_rejected():
    x = draw_decode(1, 1, 8, 16, 64, seed=8)
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    o, lse = torch.empty_like(q), torch.empty(1, 1, 8, device=DEV)
    s = torch.cuda.current_stream().cuda_stream
    args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), 1, 1)
    assert _lib.fa_fwd_decode(*args, 9, 16, 64, 0.1, 0, None, 0, s) == _lib.FA_ERR_UNSUPPORTED
    assert _lib.fa_fwd_decode(*args, 8, 4, 64, 0.1, 1, None, 0, s) == _lib.FA_ERR_INVALID_ARG
    assert _lib.fa_fwd_decode(*args, 8, 0, 64, 0.1, 0, None, 0, s) == _lib.FA_ERR_INVALID_ARG
    assert _lib.fa_fwd_decode(*args, 8, 16, 96, 0.1, 0, None, 0, s) == _lib.FA_ERR_UNSUPPORTED
    assert _lib.fa_fwd_decode(*args, 8, 16, 64, -1.0, 0, None, 0, s) == _lib.FA_ERR_INVALID_ARG
    assert _lib.fa_fwd_decode(*args, 0, 16, 64, 0.1, 0, None, 0, s) == _lib.FA_OK


@pytest.mark.parametrize("name", sorted(DECODE_BY_NAME))
def test_decode_workloads_in_full(name):
    """The benchmark's decode workloads, every output row against the oracle."""
    w = DECODE_BY_NAME[name]
    x = draw_decode(w.B, w.H, w.Nq, w.Nk, w.d, w.seed)
    o, lse = gpu(x, w.causal, w.tau)
    o_ref, l_ref = oracle.fwd_decode(x["q"], x["k"], x["v"], w.tau, w.causal)
    check_o(o, o_ref)
    check_lse(lse, l_ref)
