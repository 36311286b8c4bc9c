"""Pins for the oracle's sliding-window mask.

Reading ("Atencao eficiente - FlashAttention, sparse e hibrida", section
"Atencao hibrida: local + global intercalados": local layers attend only to a
window of recent tokens): key j is visible from query i iff i - w < j <= i.
"""
import numpy as np
import pytest

import oracle

rng = np.random.default_rng(2024)


def _band(N, w):
    i = np.arange(N)[:, None]
    j = np.arange(N)[None, :]
    return (j <= i) & (j > i - w)


@pytest.mark.parametrize("w", [1, 2, 5, 37])
def test_probabilities_live_on_the_band(w):
    B, H, N, d = 1, 2, 37, 8
    q, k, v = (rng.standard_normal((B, H, N, d)) for _ in range(3))
    P = oracle.probs(q, k, v, 0.3, True, window=w)
    band = _band(N, w)
    assert (P[..., ~band] == 0).all()
    assert (P[..., band] > 0).all()
    np.testing.assert_allclose(P.sum(-1), 1.0, rtol=0, atol=1e-12)


@pytest.mark.parametrize("w", [50, 51, 1000])
def test_window_at_least_n_is_causal(w):
    B, H, N, d = 1, 2, 50, 8
    q, k, v, do = (rng.standard_normal((B, H, N, d)) for _ in range(4))
    Oc, Lc = oracle.fwd(q, k, v, 0.2, True)
    Ow, Lw = oracle.fwd(q, k, v, 0.2, True, window=w)
    assert np.array_equal(Oc, Ow) and np.array_equal(Lc, Lw)
    gc = oracle.bwd(q, k, v, do, 0.2, True)
    gw = oracle.bwd(q, k, v, do, 0.2, True, window=w)
    for a, b in zip(gc, gw):
        assert np.array_equal(a, b)


def test_window_one_returns_own_value():
    B, H, N, d = 2, 1, 20, 8
    q, k, v = (rng.standard_normal((B, H, N, d)) for _ in range(3))
    O, L = oracle.fwd(q, k, v, 0.4, True, window=1)
    assert np.array_equal(O, v)
    np.testing.assert_allclose(L, 0.4 * (q * k).sum(-1), rtol=0, atol=1e-13)


@pytest.mark.parametrize("w", [1, 3, 16])
def test_zero_query_gives_window_mean(w):
    B, H, N, d = 1, 1, 40, 4
    q = np.zeros((B, H, N, d))
    k, v = (rng.standard_normal((B, H, N, d)) for _ in range(2))
    O, L = oracle.fwd(q, k, v, 0.5, True, window=w)
    for i in range(N):
        lo = max(0, i - w + 1)
        np.testing.assert_allclose(O[0, 0, i], v[0, 0, lo:i + 1].mean(0), rtol=0, atol=1e-13)
        np.testing.assert_allclose(L[0, 0, i], np.log(i + 1 - lo), rtol=0, atol=1e-13)


def _blocked_window(q, k, v, tau, w, Br, Bc):
    """The pages' blocked loop ("como funciona" section of the tonho.wtf entry)
    with the window mask applied inside each score block."""
    N, d = q.shape
    O = np.zeros((N, d))
    m = np.full(N, -np.inf)
    l = np.zeros(N)
    for j0 in range(0, N, Bc):
        kj, vj = k[j0:j0 + Bc], v[j0:j0 + Bc]
        for i0 in range(0, N, Br):
            rows = slice(i0, i0 + Br)
            qi = np.arange(i0, min(i0 + Br, N))[:, None]
            kk = np.arange(j0, min(j0 + Bc, N))[None, :]
            S = np.where((kk <= qi) & (kk > qi - w), tau * q[rows] @ kj.T, -np.inf)
            blk = S.max(axis=1)
            seen = np.isfinite(blk)
            Pb = np.where(seen[:, None], np.exp(S - np.where(seen, blk, 0)[:, None]), 0.0)
            new_m = np.maximum(m[rows], blk)
            with np.errstate(invalid="ignore"):  # -inf - -inf on rows the where() discards
                a_old = np.where(np.isfinite(m[rows]), np.exp(m[rows] - new_m), 0.0)
                a_blk = np.where(seen, np.exp(blk - new_m), 0.0)
            new_l = a_old * l[rows] + a_blk * Pb.sum(axis=1)
            num = l[rows, None] * a_old[:, None] * O[rows] + a_blk[:, None] * (Pb @ vj)
            # a row with no visible key so far keeps O = 0, l = 0 (nothing to normalise)
            O[rows] = np.where(new_l[:, None] > 0, num / np.where(new_l > 0, new_l, 1.0)[:, None], 0.0)
            m[rows], l[rows] = new_m, new_l
    return O, m + np.log(l)


@pytest.mark.parametrize("w,Br,Bc", [(3, 2, 3), (5, 4, 4), (1, 3, 2)])
def test_blocked_loop_with_window_equals_oracle(w, Br, Bc):
    N, d, tau = 13, 5, 0.6
    q, k, v = (rng.standard_normal((N, d)) for _ in range(3))
    Ob, Lb = _blocked_window(q, k, v, tau, w, Br, Bc)
    O, L = oracle.fwd(q[None, None], k[None, None], v[None, None], tau, True, window=w)
    np.testing.assert_allclose(O[0, 0], Ob, rtol=0, atol=1e-12)
    np.testing.assert_allclose(L[0, 0], Lb, rtol=0, atol=1e-12)


@pytest.mark.parametrize("w", [1, 2, 4])
def test_window_backward_matches_central_differences(w):
    N, d, tau = 6, 3, 0.8
    q, k, v, do = (rng.standard_normal((1, 1, N, d)) for _ in range(4))
    dq, dk, dv = oracle.bwd(q, k, v, do, tau, True, window=w)

    def loss(qq, kk, vv):
        return float((oracle.fwd(qq, kk, vv, tau, True, window=w)[0] * do).sum())

    h = 1e-6
    for name, g in (("q", dq), ("k", dk), ("v", dv)):
        fd = np.zeros_like(g)
        for idx in np.ndindex(g.shape):
            plus = {"qq": q.copy(), "kk": k.copy(), "vv": v.copy()}
            minus = {"qq": q.copy(), "kk": k.copy(), "vv": v.copy()}
            plus[name * 2][idx] += h
            minus[name * 2][idx] -= h
            fd[idx] = (loss(**plus) - loss(**minus)) / (2 * h)
        assert np.abs(fd - g).max() <= 1e-6 * max(1.0, np.abs(g).max()), name


def test_window_backward_sum_invariants():
    B, H, N, d = 1, 2, 30, 8
    q, k, v, do = (rng.standard_normal((B, H, N, d)) for _ in range(4))
    dq, dk, dv = oracle.bwd(q, k, v, do, 0.3, True, window=7)
    np.testing.assert_allclose(dk.sum(axis=2), 0.0, rtol=0, atol=1e-12)
    np.testing.assert_allclose(dv.sum(axis=2), do.sum(axis=2), rtol=0, atol=1e-12)


def test_window_needs_causal_and_positive_width():
    q = np.zeros((1, 1, 4, 2))
    with pytest.raises(ValueError):
        oracle.fwd(q, q, q, 1.0, False, window=2)
    with pytest.raises(ValueError):
        oracle.fwd(q, q, q, 1.0, True, window=0)
