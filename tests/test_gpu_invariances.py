"""Invariances of attention checked on the GPU kernels themselves.

  - Key shift: K_j -> K_j + c for every key leaves the softmax weights unchanged
    (every score of row i moves by tau q_i . c), so O is unchanged and
    LSE_i moves by exactly tau q_i . c.
  - Joint key/value permutation (non-causal): permuting the rows of K and V
    together leaves O and LSE unchanged, and permutes the rows of dK and dV.

Inputs are dyadic (multiples of 1/4, |x| <= 8) so the shifted keys are exact in
bf16 and the comparisons see only the kernels' own rounding.
"""
import math

import numpy as np
import pytest
import torch

from exact_io_aware_12_gb300 import api, _lib
from tests._parity import check_grad, max_abs, np64, rel_l2

pytestmark = pytest.mark.gpu
DEV = "cuda"


def dyadic(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * 2).round().clamp(-16, 16).div(4).to(torch.bfloat16)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_key_shift_moves_lse_only(d, causal):
    B, H, N = 1, 2, 600
    tau = 1 / math.sqrt(d)
    q, k, v = (dyadic((B, H, N, d), seed=s) for s in (1, 2, 3))
    c = dyadic((B, H, 1, d), seed=4)
    k2 = (k.float() + c.float()).to(torch.bfloat16)
    assert torch.equal(k2.float() - k.float(), c.float().expand_as(k2))  # the shift is exact
    o, l = api.fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal, tau)
    o2, l2 = api.fwd(q.to(DEV), k2.to(DEV), v.to(DEV), causal, tau)
    torch.cuda.synchronize()
    assert max_abs(o2, np64(o)) <= 1e-2 and rel_l2(o2, np64(o)) <= 5e-3
    shift = tau * (np64(q) * np64(c)).sum(-1)
    assert max_abs(np64(l2) - np64(l), shift) <= 1e-3


@pytest.mark.parametrize("d", [64, 128])
def test_joint_key_value_permutation(d):
    B, H, N = 1, 2, 500
    tau = 1 / math.sqrt(d)
    q, k, v, do = (dyadic((B, H, N, d), seed=s) for s in (5, 6, 7, 8))
    perm = torch.from_numpy(np.random.default_rng(9).permutation(N))
    kp, vp = k[:, :, perm].contiguous(), v[:, :, perm].contiguous()
    dev = [t.to(DEV) for t in (q, k, v, do, kp, vp)]
    o, l = api.fwd(dev[0], dev[1], dev[2], False, tau)
    op, lp = api.fwd(dev[0], dev[4], dev[5], False, tau)
    dq, dk, dv = api.bwd(dev[0], dev[1], dev[2], o, dev[3], l, False, tau)
    dqp, dkp, dvp = api.bwd(dev[0], dev[4], dev[5], op, dev[3], lp, False, tau)
    torch.cuda.synchronize()
    assert api.last_device_error() == _lib.FA_OK
    assert max_abs(op, np64(o)) <= 1e-2 and max_abs(lp, np64(l)) <= 1e-3
    check_grad(dqp, np64(dq), "dQ")
    check_grad(dkp, np64(dk[:, :, perm.to(DEV)]), "dK")
    check_grad(dvp, np64(dv[:, :, perm.to(DEV)]), "dV")
