"""Pins for the fp64 CPU oracle: facts fixed by the pages or by mathematics,
independent of the oracle's own code.

Sources: tonho.wtf "flash attention" entry, section "como funciona" (scores
tau*Q K^T, running max m and sum l, stored O and statistics, the identity
D_i = P_i . dP_i = dO_i . O_i); "Atencao eficiente - FlashAttention, sparse e
hibrida", "Insight 2 - Online softmax" (blockwise softmax equals the full-row
softmax).
"""
import json
import math
import os

import numpy as np
import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
rng = np.random.default_rng(12345)


def _expr(s):
    # closed-form expressions over rationals and ln(); nothing else is allowed
    allowed = set("0123456789+-*/(). ln")
    assert set(s) <= allowed, s
    return float(eval(s, {"__builtins__": {}}, {"ln": math.log}))


def _arr(x):
    return np.array([[_expr(e) for e in row] for row in x]) if isinstance(x[0], list) \
        else np.array([_expr(e) for e in x])


# ---------------------------------------------------------------- golden ----
def _golden_cases():
    with open(os.path.join(HERE, "golden", "hand_worked.json")) as f:
        doc = json.load(f)
    for case in doc["cases"]:
        for mode in ("noncausal", "causal", "windowed"):
            if mode in case:
                yield pytest.param(case, mode, id=f"{case['name']}-{mode}")


@pytest.mark.parametrize("case,mode", list(_golden_cases()))
def test_golden_hand_worked(case, mode):
    q, k, v, do = (_arr(case[n])[None] for n in ("q", "k", "v", "do"))
    tau = _expr(case["tau"])
    exp = case[mode]
    causal = mode in ("causal", "windowed")
    window = int(_expr(case["window"])) if mode == "windowed" else None
    O, L = oracle.fwd(q, k, v, tau, causal, window=window)
    np.testing.assert_allclose(O[0], _arr(exp["o"]), rtol=0, atol=1e-12)
    np.testing.assert_allclose(L[0], _arr(exp["lse"]), rtol=0, atol=1e-12)
    dq, dk, dv, O2, L2, D = oracle.bwd(q, k, v, do, tau, causal, want_fwd=True, window=window)
    np.testing.assert_allclose(dq[0], _arr(exp["dq"]), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dk[0], _arr(exp["dk"]), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dv[0], _arr(exp["dv"]), rtol=0, atol=1e-12)
    np.testing.assert_allclose(D[0], _arr(exp["D"]), rtol=0, atol=1e-12)
    np.testing.assert_allclose(O2, O, rtol=0, atol=0)
    np.testing.assert_allclose(L2, L, rtol=0, atol=0)


# ------------------------------------------------------ softmax rows (P-a) --
@pytest.mark.parametrize("causal", [False, True])
def test_rows_sum_to_one(causal):
    B, H, N, d = 2, 3, 37, 16
    q, k, v = (rng.standard_normal((B, H, N, d)) * 2 for _ in range(3))
    P = oracle.probs(q, k, v, 0.25, causal)
    assert P.shape == (B, H, N, N)
    np.testing.assert_allclose(P.sum(-1), 1.0, rtol=0, atol=1e-12)
    assert (P >= 0).all()
    if causal:
        upper = np.triu(np.ones((N, N), bool), 1)
        assert (P[..., upper] == 0).all()
    else:
        assert (P > 0).all()


# ------------------------------------------------------ Q = 0 (P-b) ---------
@pytest.mark.parametrize("causal", [False, True])
def test_zero_query_gives_mean_of_visible_values(causal):
    B, H, N, d = 1, 2, 50, 8
    q = np.zeros((B, H, N, d))
    k = rng.standard_normal((B, H, N, d))
    v = rng.standard_normal((B, H, N, d))
    O, L = oracle.fwd(q, k, v, 0.3, causal)
    counts = np.arange(1, N + 1) if causal else np.full(N, N)
    if causal:
        mean = np.cumsum(v, axis=2) / counts[:, None]
    else:
        mean = np.broadcast_to(v.mean(axis=2, keepdims=True), v.shape)
    np.testing.assert_allclose(O, mean, rtol=0, atol=1e-13)
    np.testing.assert_allclose(L, np.broadcast_to(np.log(counts), L.shape), rtol=0, atol=1e-13)


# ------------------------------------------------ dominant logit (P-c) ------
@pytest.mark.parametrize("causal", [False, True])
def test_dominant_logit_selects_value_row(causal):
    N, d, c = 8, 8, 60.0
    tau = 1 / math.sqrt(d)
    k = np.eye(N, d)[None, None]
    pi = np.array([0, 0, 1, 3, 2, 5, 6, 4]) if causal else rng.permutation(N)
    q = np.zeros((1, 1, N, d))
    for i in range(N):
        q[0, 0, i, pi[i]] = c / tau
    v = rng.standard_normal((1, 1, N, d))
    O, L = oracle.fwd(q, k, v, tau, causal)
    np.testing.assert_allclose(O[0, 0], v[0, 0, pi], rtol=0, atol=1e-14)
    nvis = np.arange(1, N + 1) if causal else np.full(N, N)
    np.testing.assert_allclose(L[0, 0], c + np.log1p((nvis - 1) * math.exp(-c)), rtol=0, atol=1e-12)


# ------------------------------------------------ first causal row (P-d) ----
def test_first_causal_row_is_first_value():
    B, H, N, d = 2, 2, 33, 16
    q, k, v = (rng.standard_normal((B, H, N, d)) for _ in range(3))
    tau = 0.125
    O, L = oracle.fwd(q, k, v, tau, True)
    assert np.array_equal(O[:, :, 0], v[:, :, 0])
    np.testing.assert_allclose(L[:, :, 0], tau * (q[:, :, 0] * k[:, :, 0]).sum(-1), rtol=0, atol=1e-13)


# ----------------------------------------- finite differences (P-e) ---------
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 3, 8])
@pytest.mark.parametrize("d", [2, 4])
def test_backward_matches_central_differences(N, d, causal):
    tau = 0.7
    q, k, v, do = (rng.standard_normal((1, 1, N, d)) for _ in range(4))
    dq, dk, dv = oracle.bwd(q, k, v, do, tau, causal)

    def loss(qq, kk, vv):
        return float((oracle.fwd(qq, kk, vv, tau, causal)[0] * do).sum())

    h = 1e-6
    for name, g in (("q", dq), ("k", dk), ("v", dv)):
        fd = np.zeros_like(g)
        for idx in np.ndindex(g.shape):
            plus = {"qq": q.copy(), "kk": k.copy(), "vv": v.copy()}
            minus = {"qq": q.copy(), "kk": k.copy(), "vv": v.copy()}
            plus[name * 2][idx] += h
            minus[name * 2][idx] -= h
            fd[idx] = (loss(**plus) - loss(**minus)) / (2 * h)
        scale = max(1.0, np.abs(g).max())
        assert np.abs(fd - g).max() <= 1e-6 * scale, (name, fd, g)


# --------------------------------------------------- D identity (P-f) -------
@pytest.mark.parametrize("causal", [False, True])
def test_softmax_jacobian_rowsum_equals_dO_dot_O(causal):
    B, H, N, d = 2, 2, 40, 32
    q, k, v, do = (rng.standard_normal((B, H, N, d)) for _ in range(4))
    _, _, _, O, _, D = oracle.bwd(q, k, v, do, 0.2, causal, want_fwd=True)
    np.testing.assert_allclose(D, (do * O).sum(-1), rtol=0, atol=1e-12)


# ------------------------------------------------ bwd invariants (P-g) ------
@pytest.mark.parametrize("causal", [False, True])
def test_backward_sum_invariants(causal):
    B, H, N, d = 1, 3, 45, 8
    q, k, v, do = (rng.standard_normal((B, H, N, d)) for _ in range(4))
    dq, dk, dv = oracle.bwd(q, k, v, do, 0.4, causal)
    np.testing.assert_allclose(dk.sum(axis=2), 0.0, rtol=0, atol=1e-12)
    np.testing.assert_allclose(dv.sum(axis=2), do.sum(axis=2), rtol=0, atol=1e-12)


# ------------------------------------------ shift / permutation (P-h) -------
@pytest.mark.parametrize("causal", [False, True])
def test_key_shift_changes_lse_only(causal):
    B, H, N, d = 1, 2, 30, 8
    tau = 0.35
    q, k, v = (rng.standard_normal((B, H, N, d)) for _ in range(3))
    c = rng.standard_normal((B, H, 1, d))
    O1, L1 = oracle.fwd(q, k, v, tau, causal)
    O2, L2 = oracle.fwd(q, k + c, v, tau, causal)
    np.testing.assert_allclose(O2, O1, rtol=0, atol=1e-12)
    np.testing.assert_allclose(L2, L1 + tau * (q * c).sum(-1), rtol=0, atol=1e-12)


def test_joint_key_value_permutation_leaves_output():
    B, H, N, d = 1, 2, 31, 8
    q, k, v = (rng.standard_normal((B, H, N, d)) for _ in range(3))
    perm = rng.permutation(N)
    O1, L1 = oracle.fwd(q, k, v, 0.3, False)
    O2, L2 = oracle.fwd(q, k[:, :, perm], v[:, :, perm], 0.3, False)
    np.testing.assert_allclose(O2, O1, rtol=0, atol=1e-12)
    np.testing.assert_allclose(L2, L1, rtol=0, atol=1e-12)


def test_query_row_order_is_irrelevant_when_not_causal():
    B, H, N, d = 1, 1, 20, 4
    q, k, v = (rng.standard_normal((B, H, N, d)) for _ in range(3))
    perm = rng.permutation(N)
    O1, L1 = oracle.fwd(q, k, v, 0.5, False)
    O2, L2 = oracle.fwd(q[:, :, perm], k, v, 0.5, False)
    np.testing.assert_allclose(O2, O1[:, :, perm], rtol=0, atol=1e-13)
    np.testing.assert_allclose(L2, L1[:, :, perm], rtol=0, atol=1e-13)


# ---------------------------------- the pages' blocked loop (P-j) -----------
def _blocked_kv_outer(q, k, v, tau, causal, Br, Bc):
    """The tiled forward as the "como funciona" section states it: the outer
    loop walks key/value blocks, the inner loop query blocks; each query block
    carries its output, running max m and running sum l; merging a new block
    rescales what was accumulated by the new max.  Written independently here
    (numpy, fp64, tiny shapes) to confirm the oracle's plain definition is
    what that loop computes."""
    N, d = q.shape
    O = np.zeros((N, d))
    m = np.full(N, -np.inf)
    l = np.zeros(N)
    for j0 in range(0, N, Bc):
        kj, vj = k[j0:j0 + Bc], v[j0:j0 + Bc]
        for i0 in range(0, N, Br):
            rows = slice(i0, i0 + Br)
            S = tau * q[rows] @ kj.T
            if causal:
                qi = np.arange(i0, min(i0 + Br, N))[:, None]
                kk = np.arange(j0, min(j0 + Bc, N))[None, :]
                S = np.where(kk <= qi, S, -np.inf)
            blk_max = S.max(axis=1)
            seen = np.isfinite(blk_max)          # rows with at least one visible key here
            Pb = np.where(seen[:, None], np.exp(S - np.where(seen, blk_max, 0)[:, None]), 0.0)
            new_m = np.maximum(m[rows], blk_max)
            a_old = np.where(np.isfinite(m[rows]), np.exp(m[rows] - new_m), 0.0)
            a_blk = np.where(seen, np.exp(blk_max - new_m), 0.0)
            new_l = a_old * l[rows] + a_blk * Pb.sum(axis=1)
            O[rows] = (l[rows, None] * a_old[:, None] * O[rows]
                       + a_blk[:, None] * (Pb @ vj)) / new_l[:, None]
            m[rows], l[rows] = new_m, new_l
    return O, m + np.log(l)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Br,Bc", [(2, 3), (4, 4), (3, 7)])
def test_pages_blocked_loop_equals_oracle(Br, Bc, causal):
    N, d, tau = 11, 5, 0.6
    q, k, v = (rng.standard_normal((N, d)) * 1.5 for _ in range(3))
    Ob, Lb = _blocked_kv_outer(q, k, v, tau, causal, Br, Bc)
    O, L = oracle.fwd(q[None, None], k[None, None], v[None, None], tau, causal)
    np.testing.assert_allclose(O[0, 0], Ob, rtol=0, atol=1e-12)
    np.testing.assert_allclose(L[0, 0], Lb, rtol=0, atol=1e-12)


# ------------------------------------------------ row-subset entry point ----
def test_row_subset_equals_full_forward():
    B, H, N, d = 2, 3, 64, 16
    q, k, v = (rng.standard_normal((B, H, N, d)) for _ in range(3))
    O, L = oracle.fwd(q, k, v, 0.25, True)
    rows = np.array([0, 5, 63, 64, 100, 191, 250, 383])
    Or, Lr = oracle.fwd_rows(q, k, v, 0.25, True, rows)
    np.testing.assert_array_equal(Or, O.reshape(-1, d)[rows])
    np.testing.assert_array_equal(Lr, L.reshape(-1)[rows])


def test_value_linearity():
    B, H, N, d = 1, 1, 17, 6
    q, k, v1, v2 = (rng.standard_normal((B, H, N, d)) for _ in range(4))
    for causal in (False, True):
        O1, _ = oracle.fwd(q, k, v1, 0.5, causal)
        O2, _ = oracle.fwd(q, k, v2, 0.5, causal)
        O3, _ = oracle.fwd(q, k, 2 * v1 - 3 * v2, 0.5, causal)
        np.testing.assert_allclose(O3, 2 * O1 - 3 * O2, rtol=0, atol=1e-12)


def test_empty_sequence_is_a_no_op():
    q = np.zeros((1, 1, 0, 4))
    O, L = oracle.fwd(q, q, q, 0.5, True)
    assert O.shape == (1, 1, 0, 4) and L.shape == (1, 1, 0)
