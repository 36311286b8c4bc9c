"""GPU parity of the block-sparse entry points (fa_fwd_blocks, fa_bwd_blocks)
against the fp64 oracle with the same block mask.

Reading (oracle/ref_attn.c header): key j is visible from query i only if
mask[i // 128][j // 128] is set (and j <= i when causal); a row that sees no
key has O = 0 and LSE = -inf and contributes no gradient.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_io_aware_12_gb300 import api, _lib
from exact_io_aware_12_gb300.workloads import (BY_NAME, draw, local_global_block_mask, make_inputs,
                                               random_block_mask)
from tests._parity import check_grad, check_lse, check_o, np64

pytestmark = pytest.mark.gpu
DEV = "cuda"
EDGE = _lib.BLOCK_MASK_EDGE


def nblocks(N):
    return (N + EDGE - 1) // EDGE


def gpu(x, causal, tau, mask, backward=True):
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    m = torch.from_numpy(np.ascontiguousarray(mask)).to(DEV)
    o, lse = api.fwd(q, k, v, causal, tau, blocks=m)
    grads = None
    if backward:
        grads = api.bwd(q, k, v, o, x["do"].to(DEV), lse, causal, tau, blocks=m)
    torch.cuda.synchronize()
    assert api.last_device_error() == _lib.FA_OK
    return o, lse, grads


def check_fwd(o, lse, o_ref, l_ref):
    """O against the oracle everywhere (both are 0 on empty rows); LSE on rows
    that see a key, and exactly -inf where the oracle's row is empty."""
    l = np64(lse).reshape(-1)
    l_ref = np.asarray(l_ref).reshape(-1)
    empty = np.isneginf(l_ref)
    assert np.array_equal(np.isneginf(l), empty), "empty rows differ"
    assert not np.isnan(l).any()
    if empty.any():
        assert (np64(o).reshape(-1, o.shape[-1])[empty] == 0).all()
    check_o(o, o_ref)
    if (~empty).any():
        check_lse(l[~empty], l_ref[~empty])


CASES = [(N, c) for N in (128, 300, 640, 1000) for c in (False, True)] + [(1, False), (1, True)]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N,causal", CASES)
def test_random_block_mask_matches_oracle(N, causal, d):
    B, H = 2, 2
    x = draw(B, H, N, d, seed=700 + N + d + causal)
    tau = 1 / math.sqrt(d)
    nb = nblocks(N)
    mask = random_block_mask(nb, B * H, 0.55, seed=N + d, empty_rows=1 if nb > 1 else 0)
    o, lse, (dq, dk, dv) = gpu(x, causal, tau, mask.reshape(B, H, nb, nb))
    o_ref, l_ref = oracle.fwd(x["q"], x["k"], x["v"], tau, causal, blocks=mask, blk=EDGE)
    check_fwd(o, lse, o_ref, l_ref)
    rq, rk, rv = oracle.bwd(x["q"], x["k"], x["v"], x["do"], tau, causal, blocks=mask, blk=EDGE)
    check_grad(dq, rq, "dQ")
    check_grad(dk, rk, "dK")
    check_grad(dv, rv, "dV")


@pytest.mark.parametrize("causal", [False, True])
def test_all_ones_mask_is_the_dense_kernel_bitwise(causal):
    N, d = 700, 128
    x = draw(1, 3, N, d, seed=31)
    tau = 1 / math.sqrt(d)
    nb = nblocks(N)
    o, lse, g = gpu(x, causal, tau, np.ones((nb, nb), np.uint8))
    q, k, v, do = (x[n].to(DEV) for n in ("q", "k", "v", "do"))
    o0, l0 = api.fwd(q, k, v, causal, tau)
    assert torch.equal(o, o0) and torch.equal(lse, l0)
    g0 = api.bwd(q, k, v, o0, do, l0, causal, tau)
    assert torch.equal(g[1], g0[1]) and torch.equal(g[2], g0[2])   # dK, dV are deterministic
    assert (g[0].float() - g0[0].float()).abs().max().item() <= 1e-2


# Key tiles visited by many query tiles (here the two global anchors, seen by all
# 32 query tiles) are split into chunks that extra CTAs run; the last chunk to
# finish adds the partial dK, dV in chunk order.
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_split_key_tiles_match_oracle(causal, d):
    B, H, N = 1, 2, 4096
    x = draw(B, H, N, d, seed=61 + d + int(causal))
    nb = nblocks(N)
    mask = local_global_block_mask(nb, local=2, anchors=2, heads=B * H, extra=0.01, seed=9)
    tau = 1 / math.sqrt(d)
    o, lse, (dq, dk, dv) = gpu(x, causal, tau, mask.reshape(B, H, nb, nb))
    o_ref, l_ref = oracle.fwd(x["q"], x["k"], x["v"], tau, causal, blocks=mask, blk=EDGE)
    check_fwd(o, lse, o_ref, l_ref)
    rq, rk, rv = oracle.bwd(x["q"], x["k"], x["v"], x["do"], tau, causal, blocks=mask, blk=EDGE)
    check_grad(dq, rq, "dQ")
    check_grad(dk, rk, "dK")
    check_grad(dv, rv, "dV")


def test_split_with_a_shared_mask_and_ragged_rows():
    """One mask for every head (the plan counts it once), 26 query tiles with a
    ragged last one, and rows of 26 mask bytes (the plan's byte-wise path): the
    anchors' 26 and 25 query tiles are split in two."""
    B, H, N, d = 1, 2, 3300, 128
    x = draw(B, H, N, d, seed=67)
    nb = nblocks(N)
    mask = local_global_block_mask(nb, local=2, anchors=2, heads=1, seed=11)[0]
    tau = 1 / math.sqrt(d)
    o, lse, (dq, dk, dv) = gpu(x, True, tau, mask)
    rq, rk, rv = oracle.bwd(x["q"], x["k"], x["v"], x["do"], tau, True, blocks=mask, blk=EDGE)
    check_grad(dq, rq, "dQ")
    check_grad(dk, rk, "dK")
    check_grad(dv, rv, "dV")


def test_split_key_tiles_are_deterministic():
    """The split key tiles' dK and dV do not depend on which chunk finishes last:
    two runs agree bit for bit."""
    B, H, N, d = 1, 4, 4096, 128
    x = draw(B, H, N, d, seed=66)
    nb = nblocks(N)
    mask = local_global_block_mask(nb, local=2, anchors=2, heads=B * H, seed=10)
    a = gpu(x, True, 0.09, mask.reshape(B, H, nb, nb))
    b = gpu(x, True, 0.09, mask.reshape(B, H, nb, nb))
    assert torch.equal(a[2][1], b[2][1]) and torch.equal(a[2][2], b[2][2])


def test_shared_mask_equals_the_same_mask_per_head_bitwise():
    N, d, B, H = 520, 64, 2, 3
    x = draw(B, H, N, d, seed=32)
    nb = nblocks(N)
    one = random_block_mask(nb, 1, 0.5, seed=5, empty_rows=1)[0]
    a = gpu(x, True, 0.125, one)
    b = gpu(x, True, 0.125, np.broadcast_to(one, (B, H, nb, nb)))
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    assert torch.equal(a[2][1], b[2][1]) and torch.equal(a[2][2], b[2][2])


@pytest.mark.parametrize("causal", [False, True])
def test_empty_mask_gives_the_empty_sum(causal):
    N, d = 384, 64
    x = draw(1, 2, N, d, seed=33)
    o, lse, (dq, dk, dv) = gpu(x, causal, 0.125, np.zeros((3, 3), np.uint8))
    assert (o == 0).all() and torch.isneginf(lse).all()
    for g in (dq, dk, dv):
        assert (g == 0).all()


def test_bad_masks_are_rejected():
    N, d = 256, 64
    x = draw(1, 3, N, d, seed=34, with_do=False)
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    o = torch.empty_like(q)
    lse = torch.empty(1, 3, N, device=DEV)
    m = torch.ones(3, 2, 2, dtype=torch.uint8, device=DEV)
    s = torch.cuda.current_stream().cuda_stream
    args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), 1, 3)
    for heads in (0, 2, 4, -1):
        assert _lib.fa_fwd_blocks(*args, N, d, 0.125, 1, m.data_ptr(), heads, s) == _lib.FA_ERR_INVALID_ARG
    assert _lib.fa_fwd_blocks(*args, N, d, 0.125, 1, None, 1, s) == _lib.FA_ERR_INVALID_ARG
    # more key blocks than the kernels' per-tile bit sets hold: refused before any launch
    assert (_lib.fa_fwd_blocks(*args, _lib.BLOCK_MASK_MAX_N + 1, d, 0.125, 1, m.data_ptr(), 1, s)
            == _lib.FA_ERR_UNSUPPORTED)
    # the mask may not overlap an output
    assert (_lib.fa_fwd_blocks(*args, N, d, 0.125, 1, o.data_ptr(), 1, s) == _lib.FA_ERR_INVALID_ARG)


def test_long_context_local_global_mask_sampled_rows_and_prefix_backward():
    """The 16k workload with a local + global-anchor mask per head (4 local
    blocks = 512 tokens, 2 anchor blocks = 256 tokens, 2% random extra blocks):
    sampled forward rows against the oracle, and the backward on the
    2048-token prefix with the mask's leading 16 x 16 blocks."""
    w = BY_NAME["long_sink_b1h16_n16384_d128_causal"]
    x = make_inputs(w)
    nb = nblocks(w.N)
    mask = local_global_block_mask(nb, local=4, anchors=2, heads=w.H, extra=0.02, seed=3)
    o, lse, _ = gpu(x, True, w.tau, mask.reshape(1, w.H, nb, nb), backward=False)
    rng = np.random.default_rng(78)
    rows = np.concatenate([h * w.N + np.unique(np.concatenate(
        [[0, 127, 128, 255, 256, 4095, 4096, w.N - 1], rng.integers(0, w.N, 48)]))
        for h in range(w.H)])
    o_ref, l_ref = oracle.fwd_rows(x["q"], x["k"], x["v"], w.tau, True, rows, blocks=mask, blk=EDGE)
    idx = torch.from_numpy(rows).to(DEV)
    check_fwd(o.reshape(-1, w.d)[idx], lse.reshape(-1)[idx], o_ref, l_ref)
    P = 2048
    xs = {n: t[:, :, :P].contiguous() for n, t in x.items()}
    ms = np.ascontiguousarray(mask[:, :P // EDGE, :P // EDGE])
    _, _, (dq, dk, dv) = gpu(xs, True, w.tau, ms.reshape(1, w.H, P // EDGE, P // EDGE))
    rq, rk, rv = oracle.bwd(xs["q"], xs["k"], xs["v"], xs["do"], w.tau, True, blocks=ms, blk=EDGE)
    check_grad(dq, rq, "dQ")
    check_grad(dk, rk, "dK")
    check_grad(dv, rv, "dV")
