"""GPU parity of the forward kernel against the fp64 oracle (through the C ABI).

Workloads: the five seeded workloads (full tensors where the oracle finishes
in seconds, sampled rows otherwise), ragged sequence lengths that span several
tiles and a partial last tile, and the closed-form cases (Q = 0, first causal
row, one dominant logit) on the GPU itself.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_io_aware_12_gb300 import api, _lib
from exact_io_aware_12_gb300.workloads import WORKLOADS, BY_NAME, draw, make_inputs, sample_rows
from tests._parity import check_lse, check_o, max_abs, np64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def gpu_fwd(x, causal, tau, o32=False):
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    o, lse = api.fwd(q, k, v, causal, tau, o_fp32=o32)
    torch.cuda.synchronize()
    assert api.last_device_error() == _lib.FA_OK
    return o, lse


@pytest.mark.parametrize("w", [w for w in WORKLOADS if w.fwd_rows_per_head is None],
                         ids=lambda w: w.name)
def test_workload_forward_full(w):
    x = make_inputs(w)
    o_ref, l_ref = oracle.fwd(x["q"], x["k"], x["v"], w.tau, w.causal)
    o, lse = gpu_fwd(x, w.causal, w.tau)
    check_o(o, o_ref, bf16_out=True)
    check_lse(lse, l_ref)
    o32, lse32 = gpu_fwd(x, w.causal, w.tau, o32=True)
    check_o(o32, o_ref, bf16_out=False, what="O(fp32)")
    assert torch.equal(lse32, lse)


@pytest.mark.parametrize("w", [w for w in WORKLOADS if w.fwd_rows_per_head is not None],
                         ids=lambda w: w.name)
def test_workload_forward_sampled_rows(w):
    x = make_inputs(w)
    rows = sample_rows(w)
    o_ref, l_ref = oracle.fwd_rows(x["q"], x["k"], x["v"], w.tau, w.causal, rows)
    o, lse = gpu_fwd(x, w.causal, w.tau)
    o_rows = o.reshape(-1, w.d)[torch.from_numpy(rows).to(DEV)]
    l_rows = lse.reshape(-1)[torch.from_numpy(rows).to(DEV)]
    check_o(o_rows, o_ref, bf16_out=True)
    check_lse(l_rows, l_ref)
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()


def test_long_context_prefix_equals_slice():
    """Causal rows [0, 2048) of the 16k workload see only keys [0, 2048), so the
    full run's rows must equal a separate run on the 2048-token prefix."""
    w = BY_NAME["long_sink_b1h16_n16384_d128_causal"]
    x = make_inputs(w)
    o, lse = gpu_fwd(x, True, w.tau)
    xs = {n: x[n][:, :, :2048].contiguous() for n in ("q", "k", "v")}
    o2, lse2 = gpu_fwd(xs, True, w.tau)
    assert torch.equal(o[:, :, :2048], o2)
    assert torch.equal(lse[:, :, :2048], lse2)


RAGGED = [1, 2, 100, 127, 128, 129, 255, 256, 257, 383, 384, 385, 640, 1000]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", RAGGED)
def test_ragged_lengths(N, d, causal):
    x = draw(2, 3, N, d, seed=100 + N + d, with_do=False)
    tau = 1 / math.sqrt(d)
    o_ref, l_ref = oracle.fwd(x["q"], x["k"], x["v"], tau, causal)
    o, lse = gpu_fwd(x, causal, tau)
    check_o(o, o_ref)
    check_lse(lse, l_ref)


# Problems with more (batch*head, tile pair) items than SMs, ragged, and with
# an odd number of query tiles, so the last pair of each head has an empty
# second tile.  At d = 64 beyond 2048 tokens these run the persistent two-tile
# forward (one CTA per SM walking the pairs).
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,N,d", [(1, 40, 1100, 128), (2, 48, 520, 128), (1, 160, 256, 128),
                                     (1, 40, 2100, 64), (2, 24, 2200, 64)])
def test_many_pairs_forward_parity(B, H, N, d, causal):
    x = draw(B, H, N, d, seed=900 + N + H, with_do=False)
    tau = 1 / math.sqrt(d)
    o_ref, l_ref = oracle.fwd(x["q"], x["k"], x["v"], tau, causal)
    o, lse = gpu_fwd(x, causal, tau)
    check_o(o, o_ref)
    check_lse(lse, l_ref)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,d", [(1200, 128), (2300, 64)])
def test_forward_matches_per_head_runs(causal, N, d):
    """A head's O and LSE do not depend on how many heads share the launch (at
    d = 64 and 2300 tokens: the persistent kernel against one-head runs of the
    one-CTA-per-pair kernel): a 48-head run equals, bitwise, one-head runs, and
    the fp32-O kernel's LSE equals the bf16 one's."""
    B, H = 1, 48
    x = draw(B, H, N, d, seed=91, with_do=False)
    o, lse = gpu_fwd(x, causal, 0.1)
    _, lse32 = gpu_fwd(x, causal, 0.1, o32=True)
    assert torch.equal(lse32, lse)
    for h in (0, 23, 47):
        xh = {n: x[n][:, h:h + 1].contiguous() for n in ("q", "k", "v")}
        ho, hl = gpu_fwd(xh, causal, 0.1)
        assert torch.equal(o[:, h:h + 1], ho) and torch.equal(lse[:, h:h + 1], hl)


@pytest.mark.parametrize("causal", [False, True])
def test_non_default_tau(causal):
    x = draw(1, 2, 300, 64, seed=7, with_do=False)
    for tau in (0.02, 0.3):
        o_ref, l_ref = oracle.fwd(x["q"], x["k"], x["v"], tau, causal)
        o, lse = gpu_fwd(x, causal, tau)
        check_o(o, o_ref)
        check_lse(lse, l_ref)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_zero_query_gives_mean_of_values(d, causal):
    B, H, N = 1, 2, 700
    x = draw(B, H, N, d, seed=11, with_do=False)
    x["q"].zero_()
    o, lse = gpu_fwd(x, causal, 1 / math.sqrt(d))
    v = np64(x["v"])
    cnt = np.arange(1, N + 1) if causal else np.full(N, N)
    mean = np.cumsum(v, axis=2) / cnt[:, None] if causal else np.broadcast_to(v.mean(2, keepdims=True), v.shape)
    check_o(o, mean)
    assert max_abs(lse, np.broadcast_to(np.log(cnt), (B, H, N))) <= 1e-3


@pytest.mark.parametrize("d", [64, 128])
def test_first_causal_row_is_first_value_bitwise(d):
    x = draw(2, 2, 513, d, seed=12, with_do=False)
    tau = 1 / math.sqrt(d)
    o, lse = gpu_fwd(x, True, tau)
    assert torch.equal(o[:, :, 0].cpu(), x["v"][:, :, 0])
    l0 = tau * (np64(x["q"][:, :, 0]) * np64(x["k"][:, :, 0])).sum(-1)
    assert max_abs(lse[:, :, 0], l0) <= 1e-3


@pytest.mark.parametrize("causal", [False, True])
def test_dominant_logit_selects_value_row(causal):
    N, d, c = 64, 64, 60.0
    tau = 1 / math.sqrt(d)
    rng = np.random.default_rng(5)
    k = torch.zeros(1, 1, N, d)
    k[0, 0, torch.arange(N), torch.arange(N)] = 1.0
    pi = np.array([rng.integers(0, i + 1) for i in range(N)]) if causal else rng.permutation(N)
    q = torch.zeros(1, 1, N, d)
    q[0, 0, torch.arange(N), torch.from_numpy(pi)] = c / tau     # 480: exact in bf16
    v = torch.randn(1, 1, N, d, generator=torch.Generator().manual_seed(3))
    x = {"q": q.bfloat16(), "k": k.bfloat16(), "v": v.bfloat16()}
    o, lse = gpu_fwd(x, causal, tau)
    assert torch.equal(o[0, 0].cpu(), x["v"][0, 0, torch.from_numpy(pi)])
    assert max_abs(lse, np.full((1, 1, N), c)) <= 1e-3


def test_forward_is_deterministic():
    w = BY_NAME["gpt2s_b8h12_n1024_d64_causal"]
    x = make_inputs(w)
    o1, l1 = gpu_fwd(x, True, w.tau)
    o2, l2 = gpu_fwd(x, True, w.tau)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_guard_bytes_around_outputs_untouched():
    B, H, N, d = 1, 2, 300, 64
    x = draw(B, H, N, d, seed=21, with_do=False)
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    n_o = B * H * N * d
    pad = 4096
    o_buf = torch.full((n_o + 2 * pad,), 7.0, dtype=torch.bfloat16, device=DEV)
    l_buf = torch.full((B * H * N + 2 * pad,), 7.0, dtype=torch.float32, device=DEV)
    o = o_buf[pad:pad + n_o].view(B, H, N, d)
    lse = l_buf[pad:pad + B * H * N].view(B, H, N)
    api.fwd(q, k, v, True, out=o, lse=lse)
    torch.cuda.synchronize()
    assert (o_buf[:pad] == 7).all() and (o_buf[pad + n_o:] == 7).all()
    assert (l_buf[:pad] == 7).all() and (l_buf[pad + B * H * N:] == 7).all()


def test_watchdog_times_out_cleanly_and_context_survives():
    s = torch.cuda.current_stream().cuda_stream
    assert api.last_device_error() == _lib.FA_OK
    assert _lib.fa_watchdog_selftest(50_000_000, s) == _lib.FA_OK
    assert _lib.fa_last_device_error(s) == _lib.FA_ERR_TIMEOUT
    assert _lib.fa_last_device_error(s) == _lib.FA_OK        # the word was cleared
    # the context is still usable
    x = draw(1, 1, 128, 64, seed=1, with_do=False)
    o, lse = gpu_fwd(x, False, 0.125)
    o_ref, _ = oracle.fwd(x["q"], x["k"], x["v"], 0.125, False)
    check_o(o, o_ref)
