"""Argument checks of the variant entry points (window, block mask, FP8,
decode) and the decode workspace size, through the C ABI without a GPU: every
case here is rejected (or found empty) before the library touches a device.
The pointers are 16-byte aligned addresses that are never dereferenced."""
import pytest

from exact_io_aware_12_gb300 import _lib

FAKE = 0x7F0000000000
STEP = 0x10000000  # 256 MB between fake buffers: no accidental overlap
ptrs = [FAKE + i * STEP for i in range(8)]


def _window(**kw):
    a = dict(Q=ptrs[0], K=ptrs[1], V=ptrs[2], O=ptrs[3], LSE=ptrs[4], B=1, H=2, N=300, d=128,
             tau=0.1, window=64)
    a.update(kw)
    return _lib.fa_fwd_window(a["Q"], a["K"], a["V"], a["O"], a["LSE"], a["B"], a["H"], a["N"],
                              a["d"], a["tau"], a["window"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(window=0), _lib.FA_ERR_INVALID_ARG),
    (dict(window=-3), _lib.FA_ERR_INVALID_ARG),
    (dict(V=None), _lib.FA_ERR_INVALID_ARG),
    (dict(d=80), _lib.FA_ERR_UNSUPPORTED),
    (dict(O=ptrs[1] + 0x40), _lib.FA_ERR_INVALID_ARG),  # O overlaps K
    (dict(B=0), _lib.FA_OK),
])
def test_window_argument_checks(kw, code):
    assert _window(**kw) == code


def _blocks(**kw):
    a = dict(Q=ptrs[0], K=ptrs[1], V=ptrs[2], O=ptrs[3], LSE=ptrs[4], B=1, H=2, N=300, d=64,
             tau=0.1, causal=1, mask=ptrs[5], heads=1)
    a.update(kw)
    return _lib.fa_fwd_blocks(a["Q"], a["K"], a["V"], a["O"], a["LSE"], a["B"], a["H"], a["N"],
                              a["d"], a["tau"], a["causal"], a["mask"], a["heads"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(mask=None), _lib.FA_ERR_INVALID_ARG),
    (dict(heads=0), _lib.FA_ERR_INVALID_ARG),
    (dict(heads=3), _lib.FA_ERR_INVALID_ARG),                  # neither 1 nor B*H
    (dict(N=1024 * 128 + 1, heads=2), _lib.FA_ERR_UNSUPPORTED),  # more than 1024 key blocks
    (dict(O=ptrs[5]), _lib.FA_ERR_INVALID_ARG),                # O overlaps the mask
    (dict(causal=3), _lib.FA_ERR_INVALID_ARG),
    (dict(N=0), _lib.FA_OK),
])
def test_block_mask_argument_checks(kw, code):
    assert _blocks(**kw) == code


def _fp8(**kw):
    a = dict(Q=ptrs[0], K=ptrs[1], V=ptrs[2], O=ptrs[3], LSE=ptrs[4], B=1, H=1, N=256, d=128,
             tau=0.09, causal=1, qs=1.0, ks=1.0, vs=1.0)
    a.update(kw)
    return _lib.fa_fwd_fp8(a["Q"], a["K"], a["V"], a["O"], a["LSE"], a["B"], a["H"], a["N"], a["d"],
                           a["tau"], a["causal"], a["qs"], a["ks"], a["vs"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(d=64), _lib.FA_ERR_UNSUPPORTED),
    (dict(qs=0.0), _lib.FA_ERR_INVALID_ARG),
    (dict(ks=-1.0), _lib.FA_ERR_INVALID_ARG),
    (dict(vs=float("nan")), _lib.FA_ERR_INVALID_ARG),
    (dict(vs=float("inf")), _lib.FA_ERR_INVALID_ARG),
    (dict(K=None), _lib.FA_ERR_INVALID_ARG),
    (dict(LSE=ptrs[3] + 0x100), _lib.FA_ERR_INVALID_ARG),  # LSE inside O
    (dict(tau=-0.1), _lib.FA_ERR_INVALID_ARG),
    (dict(H=0), _lib.FA_OK),
])
def test_fp8_argument_checks(kw, code):
    assert _fp8(**kw) == code


def _decode(**kw):
    a = dict(Q=ptrs[0], K=ptrs[1], V=ptrs[2], O=ptrs[3], LSE=ptrs[4], B=1, H=2, Nq=1, Nk=65536,
             d=128, tau=0.09, causal=0, ws=ptrs[6], wsb=1 << 28)
    a.update(kw)
    return _lib.fa_fwd_decode(a["Q"], a["K"], a["V"], a["O"], a["LSE"], a["B"], a["H"], a["Nq"],
                              a["Nk"], a["d"], a["tau"], a["causal"], a["ws"], a["wsb"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(Nq=9), _lib.FA_ERR_UNSUPPORTED),
    (dict(d=96), _lib.FA_ERR_UNSUPPORTED),
    (dict(Nk=0), _lib.FA_ERR_INVALID_ARG),
    (dict(Nq=5, Nk=4, causal=1), _lib.FA_ERR_INVALID_ARG),  # causal needs Nq <= Nk
    (dict(tau=0.0), _lib.FA_ERR_INVALID_ARG),
    (dict(causal=2), _lib.FA_ERR_INVALID_ARG),
    (dict(Q=None), _lib.FA_ERR_INVALID_ARG),
    (dict(wsb=64), _lib.FA_ERR_WORKSPACE),                  # split plan needs more
    (dict(ws=ptrs[1]), _lib.FA_ERR_INVALID_ARG),            # workspace overlaps K
    (dict(Nq=0), _lib.FA_OK),
])
def test_decode_argument_checks(kw, code):
    assert _decode(**kw) == code


def test_decode_workspace_size():
    size = _lib.fa_decode_workspace_size
    # a long cache over few heads is split, so it needs a workspace: per split
    # and query row d partial outputs plus two statistics, fp32, 256-byte rounded
    long = size(1, 2, 1, 65536, 128)
    assert long > 0 and long % 256 == 0
    assert size(1, 2, 1, 100, 128) == 0                  # a short cache is not split
    assert size(1, 2, 4, 65536, 128) >= 4 * long - 256  # four query rows need ~4x
    assert size(1, 2, 1, 65536, 64) < long               # smaller rows at d = 64
    # invalid shapes need nothing
    for args in [(0, 2, 1, 100, 128), (1, 2, 9, 100, 128), (1, 2, 1, 0, 128), (1, 2, 1, 100, 80)]:
        assert size(*args) == 0
