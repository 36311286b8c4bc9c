"""The FP8 forward's tolerance, derived on the CPU from the oracle plus the one
rounding the method adds (e4m3 softmax numerators before the P V product).

The GPU tests hold the FP8 O to a per-element bound (fp8_o_bound: six standard
deviations of the summed e4m3 roundings, plus the bf16 rounding of O) and to
rel-L2 FP8_O_REL_L2.  Here the rounding is emulated exactly on the oracle's
probabilities for the same seeded workloads, and the checks are that
  * the emulation harness reproduces the oracle when nothing is rounded;
  * the emulated O stays inside the per-element bound, with room to spare;
  * the rel-L2 bar is at least 1.5x the emulated rel-L2 (an average over every
    element of a workload, so it varies little from one rounding to another);
  * the per-element bound fails when one key tile's values are wrong, which a
    flat max-abs or rel-L2 bar at these sizes would let through.
A flat max-abs bar is not used: at N = 640 causal the emulated rounding alone
reaches max-abs 0.067 on the early rows, which see few keys."""
import math

import numpy as np
import pytest

import oracle
from exact_io_aware_12_gb300.workloads import draw_fp8
from tests._parity import FP8_O_REL_L2, fp8_emulated_o, fp8_o_bound, max_abs, rel_l2

TAU = 1 / math.sqrt(128)
SCALES = (64.0, 256.0)   # the numerator of the true row max, and of a running max 2 below it


def _decoded(x):
    return tuple(oracle.e4m3_to_f64(x[n + "8"]) * x[n + "_scale"] for n in ("q", "k", "v"))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [100, 129, 640, 1000, 2048])
def test_tolerance_covers_the_emulated_rounding(N, causal):
    # the GPU parity test's workloads (tests/test_gpu_fp8.py::test_fp8_matches_oracle)
    x = draw_fp8(2, 2, N, 128, seed=1200 + N + causal)
    q, k, v = _decoded(x)
    P = oracle.probs(q, k, v, TAU, causal).reshape(4, N, N)
    V = v.reshape(4, N, 128)
    o_ref, _ = oracle.fwd(q, k, v, TAU, causal)
    o_ref = o_ref.reshape(4, N, 128)
    # the harness itself: no rounding gives back the oracle's O
    exact = np.stack([fp8_emulated_o(P[h], V[h], rounding=False) for h in range(4)])
    assert max_abs(exact, o_ref) < 1e-12
    for scale in SCALES:
        emu = np.stack([fp8_emulated_o(P[h], V[h], p_scale=scale) for h in range(4)])
        assert max_abs(emu, o_ref) > 1e-3                      # the rounding is really there
        assert FP8_O_REL_L2 >= 1.5 * rel_l2(emu, o_ref)
        for h in range(4):
            ratio = np.abs(emu[h] - o_ref[h]) / fp8_o_bound(P[h], V[h], o_ref[h])
            assert ratio.max() <= 0.8, ratio.max()


def _long_rows(heads=(0, 11)):
    """Sampled rows of the 16k causal FP8 shape, as tests/test_gpu_fp8.py takes
    them, for some of its heads: probabilities, values and the oracle's O."""
    N, H = 16384, 16
    x = draw_fp8(1, H, N, 128, seed=3)
    q, k, v = _decoded(x)
    rng = np.random.default_rng(79)
    out = []
    for h in range(H):
        rows = np.unique(np.concatenate([[0, 1, 127, 128, 8191, N - 1], rng.integers(0, N, 32)]))
        if h not in heads:
            continue
        s = TAU * (q[0, h, rows] @ k[0, h].T)
        s[np.arange(N)[None, :] > rows[:, None]] = -np.inf
        o_ref, lse = oracle.fwd_rows(q, k, v, TAU, True, h * N + rows)
        out.append((np.exp(s - lse[:, None]), v[0, h], o_ref))
    return out


def test_per_element_bound_holds_at_16k_and_catches_a_wrong_tile():
    for P, V, o_ref in _long_rows():
        assert np.allclose(P.sum(axis=1), 1.0, atol=1e-12)
        bound = fp8_o_bound(P, V, o_ref)
        for scale in SCALES:
            emu = fp8_emulated_o(P, V, p_scale=scale)
            assert (np.abs(emu - o_ref) <= 0.8 * bound).all()
            # a planted mistake: one 128-key tile of V replaced by the next tile
            bad_v = V.copy()
            bad_v[4096:4224] = V[4224:4352]
            wrong = fp8_emulated_o(P, bad_v, p_scale=scale)
            hit = P[:, 4096:4224].sum(axis=1) > 0              # rows that see that tile
            assert hit.sum() >= 10
            assert (np.abs(wrong - o_ref)[hit] > bound[hit]).any(axis=1).all()
            # ... which the flat bars would not catch
            assert rel_l2(wrong, o_ref) < FP8_O_REL_L2 and max_abs(wrong, o_ref) < 0.08
