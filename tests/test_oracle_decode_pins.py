"""Pins of the oracle's decode forward (Nq query rows against Nk cached keys).

Reading ("Atencao eficiente - FlashAttention, sparse e hibrida", box
"FlashAttention nao acelera o decode token a token": a decode step brings one
new query row that reads the whole KV cache): the Nq queries are the last Nq
positions of the sequence, so with causal query i sees keys j <= i + Nk - Nq.

Each pin reduces a decode problem to the square oracle (pinned on its own in
test_oracle_pins.py) or to a closed form.
"""
import math

import numpy as np
import pytest

import oracle


def draw(BH, N, d, seed):
    rng = np.random.default_rng(seed)
    return [rng.standard_normal((BH, N, d)) for _ in range(3)]


@pytest.mark.parametrize("causal", [False, True])
def test_square_decode_is_the_square_oracle(causal):
    q, k, v = draw(2, 9, 3, seed=1)
    o, l = oracle.fwd_decode(q, k, v, 0.6, causal)
    o0, l0 = oracle.fwd(q, k, v, 0.6, causal)
    assert np.array_equal(o, o0) and np.array_equal(l, l0)


@pytest.mark.parametrize("Nq,Nk", [(1, 1), (1, 17), (3, 17), (5, 6), (4, 40)])
def test_causal_decode_is_the_last_rows_of_the_square_problem(Nq, Nk):
    """The decode queries placed as the last Nq rows of an Nk x Nk causal problem
    (earlier rows arbitrary) give the same rows."""
    _, k, v = draw(2, Nk, 4, seed=Nq + Nk)
    qs = np.random.default_rng(7).standard_normal((2, Nk, 4))
    q = qs[:, Nk - Nq:]
    o, l = oracle.fwd_decode(q, k, v, 0.8, True)
    o0, l0 = oracle.fwd(qs, k, v, 0.8, True)
    assert np.array_equal(o, o0[:, Nk - Nq:]) and np.array_equal(l, l0[:, Nk - Nq:])


@pytest.mark.parametrize("Nq,Nk", [(1, 13), (4, 13), (13, 13)])
def test_noncausal_decode_is_the_first_rows_of_a_padded_square_problem(Nq, Nk):
    _, k, v = draw(1, Nk, 3, seed=3 * Nq)
    qs = np.random.default_rng(8).standard_normal((1, Nk, 3))
    o, l = oracle.fwd_decode(qs[:, :Nq], k, v, 1.2, False)
    o0, l0 = oracle.fwd(qs, k, v, 1.2, False)
    assert np.array_equal(o, o0[:, :Nq]) and np.array_equal(l, l0[:, :Nq])


@pytest.mark.parametrize("causal", [False, True])
def test_zero_queries_give_the_mean_of_the_visible_values(causal):
    """Q = 0: query i averages the values it sees: all Nk keys, or with causal
    the first Nk - Nq + i + 1; LSE = ln(count)."""
    Nq, Nk = 4, 11
    _, k, v = draw(1, Nk, 2, seed=9)
    q = np.zeros((1, Nq, 2))
    o, l = oracle.fwd_decode(q, k, v, 1.0, causal)
    for i in range(Nq):
        n = Nk - Nq + i + 1 if causal else Nk
        np.testing.assert_allclose(o[0, i], v[0, :n].mean(0), rtol=0, atol=1e-14)
        assert abs(l[0, i] - math.log(n)) < 1e-14


def test_bad_shapes_are_rejected():
    q, k, v = draw(1, 5, 2, seed=10)
    with pytest.raises(ValueError):
        oracle.fwd_decode(np.zeros((1, 6, 2)), k, v, 1.0, True)       # Nq > Nk with causal
    with pytest.raises(ValueError):
        oracle.fwd_decode(q[:, :2, :1], k, v, 1.0, False)             # d differs
    with pytest.raises(ValueError):
        oracle.fwd_decode(q[:, :2], k, v[:, :4], 1.0, False)          # k, v differ
