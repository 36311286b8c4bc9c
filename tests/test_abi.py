"""The C-ABI library builds for sm_103a, loads, exports every entry point that
include/fa.h declares, and rejects bad arguments before launching anything.
No compute call is made here (these run without a GPU)."""
import ctypes
import os
import re
import subprocess

import pytest

from exact_io_aware_12_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")


def _read(path):
    with open(path) as f:
        return f.read()


def declared_symbols():
    text = _read(HEADER)
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    syms = declared_symbols()
    for must in ("fa_fwd", "fa_bwd", "fa_bwd_workspace_size", "fa_status_string",
                 "fa_last_device_error"):
        assert must in syms


def test_library_loads_and_exports_every_declared_symbol():
    lib = _lib.load()
    assert os.path.basename(_lib.library_path()) == "libfa_gb300.so"
    for name in declared_symbols():
        assert hasattr(lib, name), name
        assert name in _lib.SIGNATURES, name


def test_no_undeclared_exports():
    # the .so exports only the C ABI (hidden visibility for everything else)
    out = subprocess.run(["nm", "-D", "--defined-only", _lib.library_path()], capture_output=True, text=True,
                         check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    fa_syms = {s for s in exported if s.startswith("fa_")}
    assert fa_syms == set(declared_symbols())


def test_status_strings():
    for code in range(6):
        s = _lib.status_string(code)
        assert s.startswith("FA_")
    assert "unknown" in _lib.status_string(99)


FAKE = 0x7F0000000000  # 16-byte aligned, never dereferenced: validation fails first


def _fwd(**kw):
    a = dict(Q=FAKE, K=FAKE + 0x10000000, V=FAKE + 0x20000000, O=FAKE + 0x30000000,
             LSE=FAKE + 0x40000000, B=1, H=1, N=128, d=64, tau=0.125, causal=1, stream=None)
    a.update(kw)
    return _lib.fa_fwd(a["Q"], a["K"], a["V"], a["O"], a["LSE"], a["B"], a["H"], a["N"], a["d"],
                       a["tau"], a["causal"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(Q=None), _lib.FA_ERR_INVALID_ARG),
    (dict(LSE=None), _lib.FA_ERR_INVALID_ARG),
    (dict(O=FAKE + 0x30000008), _lib.FA_ERR_INVALID_ARG),       # misaligned
    (dict(B=-1), _lib.FA_ERR_INVALID_ARG),
    (dict(N=-5), _lib.FA_ERR_INVALID_ARG),
    (dict(tau=0.0), _lib.FA_ERR_INVALID_ARG),
    (dict(tau=float("nan")), _lib.FA_ERR_INVALID_ARG),
    (dict(tau=float("inf")), _lib.FA_ERR_INVALID_ARG),
    (dict(causal=2), _lib.FA_ERR_INVALID_ARG),
    (dict(d=96), _lib.FA_ERR_UNSUPPORTED),
    (dict(d=256), _lib.FA_ERR_UNSUPPORTED),
    (dict(N=65535 * 128 + 1), _lib.FA_ERR_UNSUPPORTED),
    (dict(O=FAKE + 0x100), _lib.FA_ERR_INVALID_ARG),             # O overlaps Q
    (dict(B=0), _lib.FA_OK),                                     # empty: nothing launched
    (dict(N=0, Q=None, K=None, V=None, O=None, LSE=None), _lib.FA_OK),
    (dict(H=0, d=96), _lib.FA_OK),
])
def test_fwd_argument_checks(kw, code):
    assert _fwd(**kw) == code


def test_workspace_size():
    B, H, N, d = 2, 3, 1000, 128
    rows = B * H * N
    r256 = lambda x: (x + 255) // 256 * 256
    assert _lib.fa_bwd_workspace_size(B, H, N, d) == r256(rows * 4) + r256(rows * d * 4)
    assert _lib.fa_bwd_workspace_size(0, 3, 10, 64) == 0
    assert _lib.fa_bwd_workspace_size(1, 1, 10, 80) == 0


def _bwd(**kw):
    base = dict(Q=FAKE, K=FAKE + 0x1 * 0x10000000, V=FAKE + 0x2 * 0x10000000,
                O=FAKE + 0x3 * 0x10000000, dO=FAKE + 0x4 * 0x10000000, LSE=FAKE + 0x5 * 0x10000000,
                dQ=FAKE + 0x6 * 0x10000000, dK=FAKE + 0x7 * 0x10000000, dV=FAKE + 0x8 * 0x10000000,
                ws=FAKE + 0x9 * 0x10000000, wsb=1 << 30, B=1, H=2, N=256, d=128, tau=0.1, causal=1)
    base.update(kw)
    b = base
    return _lib.fa_bwd(b["Q"], b["K"], b["V"], b["O"], b["dO"], b["LSE"], b["dQ"], b["dK"], b["dV"],
                       b["ws"], b["wsb"], b["B"], b["H"], b["N"], b["d"], b["tau"], b["causal"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(dO=None), _lib.FA_ERR_INVALID_ARG),
    (dict(dK=FAKE + 0x7 * 0x10000000 + 4), _lib.FA_ERR_INVALID_ARG),
    (dict(wsb=100), _lib.FA_ERR_WORKSPACE),
    (dict(ws=FAKE + 0x9 * 0x10000000 + 8), _lib.FA_ERR_INVALID_ARG),
    (dict(dQ=FAKE + 0x40), _lib.FA_ERR_INVALID_ARG),               # dQ overlaps Q
    (dict(dV=FAKE + 0x7 * 0x10000000 + 0x100), _lib.FA_ERR_INVALID_ARG),  # dV overlaps dK
    (dict(ws=FAKE + 0x8 * 0x10000000), _lib.FA_ERR_INVALID_ARG),   # workspace overlaps dV
    (dict(d=32), _lib.FA_ERR_UNSUPPORTED),
    (dict(causal=-1), _lib.FA_ERR_INVALID_ARG),
    (dict(N=0), _lib.FA_OK),
])
def test_bwd_argument_checks(kw, code):
    assert _bwd(**kw) == code


def test_watchdog_selftest_rejects_bad_limits():
    assert _lib.fa_watchdog_selftest(0, None) == _lib.FA_ERR_INVALID_ARG
    assert _lib.fa_watchdog_selftest(10 ** 12, None) == _lib.FA_ERR_INVALID_ARG


def test_product_and_oracle_share_no_code():
    """The CUDA library never imports or links the oracle, and the oracle
    includes nothing from the library."""
    out = subprocess.run(["nm", "-D", _lib.library_path()], capture_output=True, text=True, check=True).stdout
    assert "ora_" not in out
    pkg = os.path.join(ROOT, "exact_io_aware_12_gb300")
    for dirpath, _, files in os.walk(pkg):
        if "_build" in dirpath:
            continue
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = _read(os.path.join(dirpath, f))
                assert not re.search(r"^\s*(import|from)\s+oracle", text, re.M), f
                assert "ref_attn" not in text and "liboracle" not in text, f
    for f in os.listdir(os.path.join(ROOT, "oracle")):
        if f.endswith((".py", ".c", ".h")):
            text = _read(os.path.join(ROOT, "oracle", f))
            assert not re.search(r"^\s*(import|from)\s+exact_io_aware_12_gb300", text, re.M), f
            assert "#include \"" not in text and "csrc" not in text, f


def _header_define(name):
    """Value of an integer #define in include/fa.h (products of unsigned literals)."""
    m = re.search(rf"#define\s+{name}\s+\(?([0-9u\s*]+)\)?", _read(HEADER))
    assert m, name
    value = 1
    for factor in m.group(1).split("*"):
        value *= int(factor.strip().rstrip("u"))
    return value


def test_python_constants_match_the_header():
    assert _lib.NOALLOC_SCRATCH_BYTES == _header_define("FA_NOALLOC_SCRATCH_BYTES")
    assert _lib.BLOCK_MASK_EDGE == _header_define("FA_BLOCK_MASK_EDGE")
    assert _lib.BLOCK_MASK_MAX_N == _header_define("FA_BLOCK_MASK_MAX_N")


def test_host_pipeline_argument_checks():
    """Rejected before any CUDA call, so these run without a GPU."""
    for args in [(0, 1, 128, 64, 0.1, 1, 2), (1, 1, 128, 64, 0.1, 1, 0), (1, 1, 128, 64, 0.1, 1, 9),
                 (1, 1, 128, 64, float("nan"), 1, 2), (1, 1, 128, 64, 0.1, 2, 2)]:
        code, h = _lib.fa_host_pipeline_create(*args, None)
        assert code == _lib.FA_ERR_INVALID_ARG and not h.value
    code, h = _lib.fa_host_pipeline_create(1, 1, 128, 96, 0.1, 1, 2, None)
    assert code == _lib.FA_ERR_UNSUPPORTED and not h.value
    assert _lib.fa_host_pipeline_step(None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE) == \
        _lib.FA_ERR_INVALID_ARG
    assert _lib.fa_host_pipeline_mark(None, None) == _lib.FA_ERR_INVALID_ARG
    assert _lib.fa_host_pipeline_sync(None) == _lib.FA_ERR_INVALID_ARG
    assert _lib.fa_host_pipeline_destroy(None) == _lib.FA_OK
