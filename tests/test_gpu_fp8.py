"""GPU parity of the FP8 (e4m3) forward (fa_fwd_fp8) against the fp64 oracle on
the decoded inputs.

Tolerance, derived from the arithmetic (tests/_parity.py, checked on the CPU by
tests/test_fp8_error_model.py): the inputs are exact (the oracle decodes the
same e4m3 bytes) and S and l are accumulated in fp32, so LSE keeps the bf16
path's 1e-3.  The one coarse step is the softmax numerator P, rounded to e4m3
(3 mantissa bits: half an ulp is 2^-4 of P, or 2^-10 among the subnormals)
before the P V product.  Every element of O is held to six standard deviations
of the sum of those roundings plus the bf16 rounding of O (fp8_o_bound), and
the whole O to rel-L2 <= 4e-2 (1.6x the emulated rounding's worst rel-L2 on
these workloads).  Cases where P is exact in e4m3 (Q = 0, one dominant logit)
are held to the bf16 path's tolerance.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_io_aware_12_gb300 import api, _lib
from exact_io_aware_12_gb300.workloads import draw_fp8
from tests._parity import FP8_O_REL_L2, check_lse, check_o, fp8_o_bound, max_abs, np64, rel_l2

pytestmark = pytest.mark.gpu
DEV = "cuda"


def gpu(x, causal, tau):
    q8, k8, v8 = (x[n].to(DEV) for n in ("q8", "k8", "v8"))
    o, lse = api.fwd_fp8(q8, k8, v8, x["q_scale"], x["k_scale"], x["v_scale"], causal, tau)
    torch.cuda.synchronize()
    assert api.last_device_error() == _lib.FA_OK
    return o, lse


def check_fp8(o, lse, o_ref, l_ref, P, V):
    """O within the per-element rounding bound (P: the rows' exact probabilities
    [n, N], V: their values [N, d], per head) and the rel-L2 bar; LSE as bf16."""
    o, o_ref = np64(o).reshape(len(P), -1, 128), np64(o_ref).reshape(len(P), -1, 128)
    for h in range(len(P)):
        bound = fp8_o_bound(P[h], V[h], o_ref[h])
        over = np.abs(o[h] - o_ref[h]) / bound
        assert over.max() <= 1.0, f"head {h}: O error {over.max():.2f}x its rounding bound"
    rl = rel_l2(o, o_ref)
    assert rl <= FP8_O_REL_L2, f"O rel-L2 {rl:.3e}"
    check_lse(lse, l_ref)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 100, 128, 129, 300, 640, 1000, 2048])
def test_fp8_matches_oracle(N, causal):
    x = draw_fp8(2, 2, N, 128, seed=1200 + N + causal)
    tau = 1 / math.sqrt(128)
    o, lse = gpu(x, causal, tau)
    o_ref, l_ref = oracle.fwd_fp8(x["q8"], x["k8"], x["v8"], x["q_scale"], x["k_scale"],
                                  x["v_scale"], tau, causal)
    q, k, v = (oracle.e4m3_to_f64(x[n + "8"]) * x[n + "_scale"] for n in ("q", "k", "v"))
    P = oracle.probs(q, k, v, tau, causal).reshape(4, N, N)
    check_fp8(o, lse, o_ref, l_ref, P, v.reshape(4, N, 128))


@pytest.mark.parametrize("causal", [False, True])
def test_zero_queries_give_the_mean_of_values(causal):
    """Q = 0: every visible P is 2^6, exact in e4m3, so O is the mean of V to
    the bf16 path's tolerance."""
    N = 700
    x = draw_fp8(1, 2, N, 128, seed=3)
    x["q8"].zero_()
    o, lse = gpu(x, causal, 0.1)
    v = oracle.e4m3_to_f64(x["v8"]) * x["v_scale"]
    cnt = np.arange(1, N + 1) if causal else np.full(N, N)
    mean = np.cumsum(v, axis=2) / cnt[:, None] if causal else np.broadcast_to(v.mean(2, keepdims=True), v.shape)
    check_o(o, mean)
    assert max_abs(lse, np.broadcast_to(np.log(cnt), (1, 2, N))) <= 1e-3


def test_dominant_logit_selects_the_value_row():
    """Q_i and K_j one-hot at 16.0 (byte 0x58) with tau = 60 / 256: the logit of
    key pi(i) is 60, every other is 0, so P is 2^6 at pi(i) and rounds to 0
    elsewhere; O_i = V_pi(i) exactly (up to bf16)."""
    N = 128
    rng = np.random.default_rng(4)
    pi = rng.permutation(N)
    k8 = torch.zeros(1, 1, N, 128, dtype=torch.uint8)
    q8 = torch.zeros(1, 1, N, 128, dtype=torch.uint8)
    k8[0, 0, torch.arange(N), torch.arange(N)] = 0x58
    q8[0, 0, torch.arange(N), torch.from_numpy(pi)] = 0x58
    v8 = torch.randn(1, 1, N, 128).to(torch.float8_e4m3fn).view(torch.uint8)
    x = {"q8": q8, "k8": k8, "v8": v8, "q_scale": 1.0, "k_scale": 1.0, "v_scale": 1.0}
    o, lse = gpu(x, False, 60.0 / 256.0)
    v = oracle.e4m3_to_f64(v8)[0, 0]
    assert torch.equal(o[0, 0].cpu(), torch.from_numpy(v[pi]).to(torch.bfloat16))
    assert max_abs(lse, np.full((1, 1, N), 60.0)) <= 1e-3


def test_long_context_sampled_rows():
    """The 16k causal shape (B=1, H=16, N=16384, d=128) in FP8: sampled rows
    against the oracle, including the first and last rows of every head."""
    N, H = 16384, 16
    x = draw_fp8(1, H, N, 128, seed=3)
    tau = 1 / math.sqrt(128)
    o, lse = gpu(x, True, tau)
    rng = np.random.default_rng(79)
    head_rows = [np.unique(np.concatenate([[0, 1, 127, 128, 8191, N - 1], rng.integers(0, N, 32)]))
                 for _ in range(H)]
    rows = np.concatenate([h * N + r for h, r in enumerate(head_rows)])
    o_ref, l_ref = oracle.fwd_fp8(x["q8"], x["k8"], x["v8"], x["q_scale"], x["k_scale"],
                                  x["v_scale"], tau, True, rows=rows)
    idx = torch.from_numpy(rows).to(DEV)
    # the sampled rows' exact probabilities, per head, for the per-element bound
    q, k, v = (oracle.e4m3_to_f64(x[n + "8"]) * x[n + "_scale"] for n in ("q", "k", "v"))
    og, lg = np64(o.reshape(-1, 128)[idx]), np64(lse.reshape(-1)[idx])
    at = 0
    for h, r in enumerate(head_rows):
        sl = slice(at, at + r.size)
        at += r.size
        s = tau * (q[0, h, r] @ k[0, h].T)
        s[np.arange(N)[None, :] > r[:, None]] = -np.inf
        P = np.exp(s - l_ref[sl, None])
        check_fp8(og[sl], lg[sl], o_ref[sl], l_ref[sl], [P], [v[0, h]])
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()


def test_bad_arguments_are_rejected():
    x = draw_fp8(1, 1, 128, 128, seed=5)
    q8, k8, v8 = (x[n].to(DEV) for n in ("q8", "k8", "v8"))
    o = torch.empty(1, 1, 128, 128, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(1, 1, 128, device=DEV)
    s = torch.cuda.current_stream().cuda_stream
    args = (q8.data_ptr(), k8.data_ptr(), v8.data_ptr(), o.data_ptr(), lse.data_ptr(), 1, 1)
    assert _lib.fa_fwd_fp8(*args, 256, 64, 0.1, 1, 1.0, 1.0, 1.0, s) == _lib.FA_ERR_UNSUPPORTED
    for bad in (0.0, -1.0, float("inf"), float("nan")):
        assert _lib.fa_fwd_fp8(*args, 128, 128, 0.1, 1, 1.0, bad, 1.0, s) == _lib.FA_ERR_INVALID_ARG
