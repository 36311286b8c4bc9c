"""Pins of the oracle's block-mask visibility (block-sparse attention).

Reading ("FlashAttention e o gargalo real de inferencia", section "o que isso
custou": block-sparse FlashAttention skips blocks and is an approximation;
"Atencao eficiente - FlashAttention, sparse e hibrida", section "Sparse e
hibrida": each token attends to a subset of positions): a mask of blk x blk
blocks; key j is visible from query i only if mask[i // blk][j // blk] is set
(and j <= i when causal).  A row that sees no key is the empty sum: O = 0,
LSE = -inf, no gradient.

Nothing here re-types the oracle's formula.  Each pin reduces a masked problem
to one the plain oracle (pinned on its own in test_oracle_pins.py) solves on
slices of the inputs, or to a closed form, or checks the gradient by finite
differences of the oracle's own forward.
"""
import math

import numpy as np
import pytest

import oracle


def draw(BH, N, d, seed):
    rng = np.random.default_rng(seed)
    return [rng.standard_normal((BH, N, d)) for _ in range(4)]


def blk_slice(x, b, blk):
    return x[..., b * blk:(b + 1) * blk, :]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,blk", [(12, 4), (13, 4), (9, 3)])
def test_all_ones_mask_equals_dense(N, blk, causal):
    q, k, v, do = draw(2, N, 3, seed=N + blk)
    nb = -(-N // blk)
    m = np.ones((nb, nb), np.uint8)
    o, l = oracle.fwd(q, k, v, 0.7, causal, blocks=m, blk=blk)
    o0, l0 = oracle.fwd(q, k, v, 0.7, causal)
    assert np.array_equal(o, o0) and np.array_equal(l, l0)
    g = oracle.bwd(q, k, v, do, 0.7, causal, blocks=m, blk=blk)
    g0 = oracle.bwd(q, k, v, do, 0.7, causal)
    for a, b in zip(g, g0):
        assert np.array_equal(a, b)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,blk", [(12, 4), (14, 4)])
def test_block_diagonal_mask_is_independent_blocks(N, blk, causal):
    """Only diagonal blocks: every block of rows is its own attention problem
    over the same block of keys (causal inside it when causal)."""
    q, k, v, do = draw(2, N, 3, seed=3 * N)
    nb = -(-N // blk)
    m = np.eye(nb, dtype=np.uint8)
    o, l = oracle.fwd(q, k, v, 0.5, causal, blocks=m, blk=blk)
    dq, dk, dv = oracle.bwd(q, k, v, do, 0.5, causal, blocks=m, blk=blk)
    for b in range(nb):
        s = [blk_slice(x, b, blk) for x in (q, k, v, do)]
        ob, lb = oracle.fwd(s[0], s[1], s[2], 0.5, causal)
        np.testing.assert_allclose(blk_slice(o, b, blk), ob, rtol=0, atol=1e-13)
        np.testing.assert_allclose(l[..., b * blk:(b + 1) * blk], lb, rtol=0, atol=1e-13)
        gb = oracle.bwd(s[0], s[1], s[2], s[3], 0.5, causal)
        for g, r in zip((dq, dk, dv), gb):
            np.testing.assert_allclose(blk_slice(g, b, blk), r, rtol=0, atol=1e-12)


def test_permutation_mask_routes_each_row_block_to_one_key_block():
    """mask[b][pi(b)] only (no involution, so a transposed index is caught):
    row block b is plain attention of Q_b over K_pi(b), V_pi(b)."""
    N, blk = 16, 4
    pi = [2, 3, 1, 0]
    q, k, v, _ = draw(1, N, 3, seed=11)
    m = np.zeros((4, 4), np.uint8)
    for b, c in enumerate(pi):
        m[b, c] = 1
    o, l = oracle.fwd(q, k, v, 0.9, False, blocks=m, blk=blk)
    for b, c in enumerate(pi):
        ob, lb = oracle.fwd(blk_slice(q, b, blk), blk_slice(k, c, blk), blk_slice(v, c, blk), 0.9, False)
        np.testing.assert_allclose(blk_slice(o, b, blk), ob, rtol=0, atol=1e-13)
        np.testing.assert_allclose(l[..., b * blk:(b + 1) * blk], lb, rtol=0, atol=1e-13)


def test_two_blocks_per_row_equal_attention_over_their_concatenated_keys():
    """Row block 1 sees key blocks 0 and 3: plain attention over [K_0; K_3],
    taken with the query block repeated so the plain oracle's square shape holds."""
    N, blk = 16, 4
    q, k, v, _ = draw(1, N, 2, seed=12)
    m = np.zeros((4, 4), np.uint8)
    m[:, 2] = 1
    m[1] = 0
    m[1, 0] = m[1, 3] = 1
    o, l = oracle.fwd(q, k, v, 1.1, False, blocks=m, blk=blk)
    qq = np.concatenate([blk_slice(q, 1, blk)] * 2, axis=-2)
    kk = np.concatenate([blk_slice(k, 0, blk), blk_slice(k, 3, blk)], axis=-2)
    vv = np.concatenate([blk_slice(v, 0, blk), blk_slice(v, 3, blk)], axis=-2)
    ob, lb = oracle.fwd(qq, kk, vv, 1.1, False)
    np.testing.assert_allclose(blk_slice(o, 1, blk), ob[..., :blk, :], rtol=0, atol=1e-13)
    np.testing.assert_allclose(l[..., blk:2 * blk], lb[..., :blk], rtol=0, atol=1e-13)


def test_per_head_masks_are_used_per_head():
    """Head h routes row block b to key block (b + h + 1) mod 3."""
    N, blk, H = 12, 4, 3
    q, k, v, _ = draw(H, N, 2, seed=13)
    m = np.zeros((H, 3, 3), np.uint8)
    for h in range(H):
        for b in range(3):
            m[h, b, (b + h + 1) % 3] = 1
    o, _ = oracle.fwd(q, k, v, 0.8, False, blocks=m, blk=blk)
    for h in range(H):
        for b in range(3):
            c = (b + h + 1) % 3
            ob, _ = oracle.fwd(blk_slice(q[h], b, blk), blk_slice(k[h], c, blk),
                               blk_slice(v[h], c, blk), 0.8, False)
            np.testing.assert_allclose(blk_slice(o[h], b, blk), ob, rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_zero_query_gives_mean_over_visible_keys(causal):
    """Q = 0: the scores are equal, so O_i is the mean of V over the keys the
    mask shows (counted here from the mask by hand) and LSE_i = ln(count)."""
    N, blk = 10, 3
    rng = np.random.default_rng(14)
    _, k, v, _ = draw(1, N, 2, seed=15)
    q = np.zeros_like(k)
    m = (rng.random((4, 4)) < 0.5).astype(np.uint8)
    m[np.arange(4), np.arange(4)] = 1
    o, l = oracle.fwd(q, k, v, 1.0, causal, blocks=m, blk=blk)
    for i in range(N):
        keys = [j for j in range(N) if m[i // blk, j // blk] and (not causal or j <= i)]
        np.testing.assert_allclose(o[0, i], v[0, keys].mean(0), rtol=0, atol=1e-14)
        assert abs(l[0, i] - math.log(len(keys))) < 1e-14


@pytest.mark.parametrize("causal", [False, True])
def test_rows_that_see_nothing_are_the_empty_sum(causal):
    N, blk = 12, 4
    q, k, v, do = draw(2, N, 3, seed=16)
    m = np.ones((3, 3), np.uint8)
    m[1] = 0                                  # row block 1 sees no key
    if causal:
        m[0, 1:] = 0                          # irrelevant above the diagonal anyway
    o, l = oracle.fwd(q, k, v, 0.6, causal, blocks=m, blk=blk)
    assert np.all(o[:, 4:8] == 0) and np.all(np.isneginf(l[:, 4:8]))
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(np.delete(l, range(4, 8), axis=1)))
    dq, dk, dv, _, _, D = oracle.bwd(q, k, v, do, 0.6, causal, want_fwd=True, blocks=m, blk=blk)
    assert np.all(dq[:, 4:8] == 0) and np.all(D[:, 4:8] == 0)
    # the empty rows' upstream gradient must not matter
    do2 = do.copy()
    do2[:, 4:8] = 7.0
    g2 = oracle.bwd(q, k, v, do2, 0.6, causal, blocks=m, blk=blk)
    for a, b in zip((dq, dk, dv), g2):
        assert np.array_equal(a, b)


@pytest.mark.parametrize("causal", [False, True])
def test_gradient_matches_finite_differences(causal):
    N, blk, d, tau, h = 6, 2, 2, 0.9, 1e-6
    q, k, v, do = draw(1, N, d, seed=17 + causal)
    m = np.array([[1, 0, 1], [0, 1, 0], [1, 1, 1]], np.uint8)

    def loss(qq, kk, vv):
        o, _ = oracle.fwd(qq, kk, vv, tau, causal, blocks=m, blk=blk)
        return float((o * do).sum())

    grads = oracle.bwd(q, k, v, do, tau, causal, blocks=m, blk=blk)
    for which, g in enumerate(grads):
        num = np.zeros_like(g)
        for idx in np.ndindex(g.shape):
            args = [q.copy(), k.copy(), v.copy()]
            args[which][idx] += h
            lp = loss(*args)
            args[which][idx] -= 2 * h
            lm = loss(*args)
            num[idx] = (lp - lm) / (2 * h)
        err = np.abs(num - g).max() / max(1e-12, np.abs(num).max())
        assert err <= 1e-6, (which, err)


def test_causal_mask_ands_with_the_block_mask():
    """Under causal, blocks above the diagonal add nothing: setting them or not
    gives the same result, and a lower-triangular all-ones mask is plain causal."""
    N, blk = 12, 4
    q, k, v, _ = draw(1, N, 2, seed=18)
    low = np.tril(np.ones((3, 3), np.uint8))
    o1, l1 = oracle.fwd(q, k, v, 0.7, True, blocks=low, blk=blk)
    o2, l2 = oracle.fwd(q, k, v, 0.7, True, blocks=np.ones((3, 3), np.uint8), blk=blk)
    o0, l0 = oracle.fwd(q, k, v, 0.7, True)
    assert np.array_equal(o1, o0) and np.array_equal(o2, o0)
    assert np.array_equal(l1, l0) and np.array_equal(l2, l0)


def test_bad_masks_are_rejected():
    q, k, v, _ = draw(2, 12, 2, seed=19)
    with pytest.raises(ValueError):
        oracle.fwd(q, k, v, 1.0, False, blocks=np.ones((2, 2)), blk=4)      # wrong block count
    with pytest.raises(ValueError):
        oracle.fwd(q, k, v, 1.0, False, blocks=np.ones((3, 3, 3)), blk=4)   # 3 heads for 2
    with pytest.raises(ValueError):
        oracle.fwd(q, k, v, 1.0, True, window=4, blocks=np.ones((3, 3)), blk=4)
