"""Shared helpers for the GPU parity tests: tolerances and comparisons.

Tolerances (GPU vs the fp64 oracle on the same bf16 inputs):
  O      max-abs <= 1e-2 and rel-L2 <= 5e-3
  LSE    max-abs <= 1e-3
  dQ/dK/dV rel-L2 <= 1e-2
When O is returned in bf16, the rounding of the exact O to bf16 alone can
exceed 1e-2 where |O| >= 4 (half an ulp there is 2^-6); for such inputs the
bf16 O is held to 1e-2 plus that rounding floor and the fp32-O entry point is
held to the plain 1e-2.
"""
import numpy as np
import torch

O_MAX_ABS = 1e-2
O_REL_L2 = 5e-3
LSE_MAX_ABS = 1e-3
GRAD_REL_L2 = 1e-2


def np64(t):
    if isinstance(t, torch.Tensor):
        return t.detach().to("cpu").double().numpy()
    return np.asarray(t, dtype=np.float64)


def rel_l2(a, ref):
    a, ref = np64(a), np64(ref)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(a - ref) / (den if den > 0 else 1.0))


def max_abs(a, ref):
    a, ref = np64(a), np64(ref)
    return float(np.abs(a - ref).max()) if a.size else 0.0


def bf16_floor(ref):
    ref = np64(ref)
    if ref.size == 0:
        return 0.0
    return float(np.abs(torch.from_numpy(np.array(ref)).to(torch.bfloat16).double().numpy() - ref).max())


def check_o(o, o_ref, bf16_out=True, what="O"):
    floor = bf16_floor(o_ref) if bf16_out else 0.0
    bound = O_MAX_ABS + (floor if floor > O_MAX_ABS else 0.0)
    ma, rl = max_abs(o, o_ref), rel_l2(o, o_ref)
    assert ma <= bound, f"{what} max-abs {ma:.3e} > {bound:.3e} (bf16 floor {floor:.3e})"
    assert rl <= O_REL_L2, f"{what} rel-L2 {rl:.3e} > {O_REL_L2}"
    return ma, rl


def check_lse(lse, lse_ref):
    ma = max_abs(lse, lse_ref)
    assert ma <= LSE_MAX_ABS, f"LSE max-abs {ma:.3e} > {LSE_MAX_ABS}"
    return ma


def check_grad(g, g_ref, what):
    rl = rel_l2(g, g_ref)
    assert rl <= GRAD_REL_L2, f"{what} rel-L2 {rl:.3e} > {GRAD_REL_L2}"
    return rl


# FP8 (e4m3) forward.  The inputs are exact (the oracle decodes the same bytes)
# and S and the row sum are fp32 accumulations, so the one coarse step is the
# softmax numerator, rounded to e4m3 before the P V product.  The kernel keeps
# P = 2^(s - m + 6) (scores in log2 units, m the running row max, at most 2
# below the true one), so P <= 2^8 and e4m3 keeps 3 mantissa bits: each P is off
# by at most half an ulp, 2^-4 P relative, or 2^-10 absolute below 2^-6 (the
# subnormals).  tests/test_fp8_error_model.py emulates exactly that rounding on
# the oracle's probabilities for the GPU tests' workloads and checks that these
# bars are at least twice the emulated error.
FP8_O_MAX_ABS = 0.08
FP8_O_REL_L2 = 4e-2
FP8_P_SCALE = 64.0                 # P of the row max, 2^6
FP8_HALF_ULP_REL = 2.0 ** -4
FP8_HALF_ULP_SUBNORMAL = 2.0 ** -10
BF16_HALF_ULP_REL = 2.0 ** -8


def fp8_emulated_o(P, V, p_scale=FP8_P_SCALE, rounding=True):
    """O as the FP8 kernel forms it from exact probabilities P [n, N] (rows sum
    to 1) and values V [N, d]: numerators p_scale * P / rowmax(P) rounded to
    e4m3 (round to nearest even) for the P V product, divided by the sum of the
    unrounded numerators."""
    P = np64(P)
    num = p_scale * P / P.max(axis=-1, keepdims=True)
    rounded = (torch.from_numpy(num).to(torch.float8_e4m3fn).double().numpy()
               if rounding else num)
    return (rounded @ np64(V)) / num.sum(axis=-1, keepdims=True)


def fp8_o_bound(P, V, o_ref, sigmas=6.0, slack=1e-4):
    """Per-element bound on |O_fp8 - O_ref| for rows with exact probabilities P
    [n, N]: `sigmas` standard deviations of the sum of independent e4m3
    roundings (each uniform within its half-ulp a_ij, variance a_ij^2 / 3, a_ij
    the larger of 2^-4 P'_ij and the subnormal 2^-10, P' = 2^6 P / rowmax P),
    plus the bf16 rounding of O and a small fp32 slack."""
    P = np64(P)
    num = FP8_P_SCALE * P / P.max(axis=-1, keepdims=True)
    a = np.where(num > 0, np.maximum(FP8_HALF_ULP_REL * num, FP8_HALF_ULP_SUBNORMAL), 0.0)
    sigma = np.sqrt((a * a / 3.0) @ (np64(V) ** 2)) / num.sum(axis=-1, keepdims=True)
    return sigmas * sigma + BF16_HALF_ULP_REL * np.abs(np64(o_ref)) + slack
