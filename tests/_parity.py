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
    return float(np.abs(torch.from_numpy(ref).to(torch.bfloat16).double().numpy() - ref).max())


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
