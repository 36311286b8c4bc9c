"""GPU parity of the sliding-window entry points (fa_fwd_window, fa_bwd_window)
against the fp64 oracle with the same window.

Window reading ("Atencao eficiente - FlashAttention, sparse e hibrida",
section "Atencao hibrida: local + global intercalados"): key j is visible from
query i iff i - w < j <= i.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_io_aware_12_gb300 import api, _lib
from exact_io_aware_12_gb300.workloads import BY_NAME, draw, make_inputs
from tests._parity import check_grad, check_lse, check_o

pytestmark = pytest.mark.gpu
DEV = "cuda"


def gpu(x, tau, window, backward=True):
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    o, lse = api.fwd(q, k, v, True, tau, window=window)
    grads = None
    if backward:
        grads = api.bwd(q, k, v, o, x["do"].to(DEV), lse, True, tau, window=window)
    torch.cuda.synchronize()
    assert api.last_device_error() == _lib.FA_OK
    return o, lse, grads


CASES = [(N, w) for N in (100, 300, 1000) for w in (1, 17, 128, 129, 256, 300)] + [(1, 1), (2048, 512)]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N,w", CASES)
def test_window_matches_oracle(N, w, d):
    x = draw(2, 2, N, d, seed=500 + N + w + d)
    tau = 1 / math.sqrt(d)
    o, lse, (dq, dk, dv) = gpu(x, tau, w)
    o_ref, l_ref = oracle.fwd(x["q"], x["k"], x["v"], tau, True, window=w)
    check_o(o, o_ref)
    check_lse(lse, l_ref)
    rq, rk, rv = oracle.bwd(x["q"], x["k"], x["v"], x["do"], tau, True, window=w)
    check_grad(dq, rq, "dQ")
    check_grad(dk, rk, "dK")
    check_grad(dv, rv, "dV")


# d = 128 windows with more (batch*head, tile pair) items than SMs run the
# persistent forward (one CTA per SM walking a list of pairs): parity on a
# ragged shape with an empty second tile in each head's last pair, and one-head
# runs (the one-CTA-per-pair kernel) equal bitwise.
def test_persistent_window_forward():
    B, H, N, d, w = 1, 64, 1100, 128, 300
    x = draw(B, H, N, d, seed=93, with_do=False)
    tau = 1 / math.sqrt(d)
    o, lse, _ = gpu(x, tau, w, backward=False)
    o_ref, l_ref = oracle.fwd(x["q"], x["k"], x["v"], tau, True, window=w)
    check_o(o, o_ref)
    check_lse(lse, l_ref)
    for h in (0, 63):
        xh = {n: x[n][:, h:h + 1].contiguous() for n in ("q", "k", "v")}
        ho, hl, _ = gpu(xh, tau, w, backward=False)
        assert torch.equal(o[:, h:h + 1], ho) and torch.equal(lse[:, h:h + 1], hl)


def test_window_one_returns_own_value_bitwise():
    x = draw(1, 3, 700, 128, seed=7)
    o, _, _ = gpu(x, 1 / math.sqrt(128), 1, backward=False)
    assert torch.equal(o.cpu(), x["v"])


@pytest.mark.parametrize("w", [640, 641, 10 ** 6])
def test_window_at_least_n_is_causal_bitwise(w):
    N, d = 640, 64
    x = draw(1, 2, N, d, seed=8)
    tau = 1 / math.sqrt(d)
    o, lse, g = gpu(x, tau, w)
    q, k, v, do = (x[n].to(DEV) for n in ("q", "k", "v", "do"))
    oc, lc = api.fwd(q, k, v, True, tau)
    assert torch.equal(o, oc) and torch.equal(lse, lc)
    gc = api.bwd(q, k, v, oc, do, lc, True, tau)
    assert torch.equal(g[1], gc[1]) and torch.equal(g[2], gc[2])   # dK, dV are deterministic


def test_window_rejects_bad_width():
    x = draw(1, 1, 128, 64, seed=9, with_do=False)
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    o = torch.empty_like(q)
    lse = torch.empty(1, 1, 128, device=DEV)
    for w in (0, -3):
        code = _lib.fa_fwd_window(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                  lse.data_ptr(), 1, 1, 128, 64, 0.125, w,
                                  torch.cuda.current_stream().cuda_stream)
        assert code == _lib.FA_ERR_INVALID_ARG


def test_long_context_window_4096_sampled_rows_and_prefix_backward():
    """The 16k workload with the 4096-token window the pages quote for local
    layers: sampled forward rows against the oracle, and the backward on the
    causal 2048-token prefix (prefix rows see only prefix keys)."""
    w_ = BY_NAME["long_sink_b1h16_n16384_d128_causal"]
    x = make_inputs(w_)
    W = 4096
    o, lse, _ = gpu(x, w_.tau, W, backward=False)
    rng = np.random.default_rng(77)
    rows = np.concatenate([h * w_.N + np.unique(np.concatenate(
        [[0, 4095, 4096, 4097, 8191, 8192, w_.N - 1], rng.integers(0, w_.N, 64)]))
        for h in range(w_.H)])
    o_ref, l_ref = oracle.fwd_rows(x["q"], x["k"], x["v"], w_.tau, True, rows, window=W)
    idx = torch.from_numpy(rows).to(DEV)
    check_o(o.reshape(-1, w_.d)[idx], o_ref)
    check_lse(lse.reshape(-1)[idx], l_ref)
    xs = {n: t[:, :, :2048].contiguous() for n, t in x.items()}
    _, _, (dq, dk, dv) = gpu(xs, w_.tau, 512)
    rq, rk, rv = oracle.bwd(xs["q"], xs["k"], xs["v"], xs["do"], w_.tau, True, window=512)
    check_grad(dq, rq, "dQ")
    check_grad(dk, rk, "dK")
    check_grad(dv, rv, "dV")
