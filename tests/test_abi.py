"""The C-ABI library: builds, loads without a GPU, exports every symbol that
include/sdpa.h declares, and rejects bad arguments before touching CUDA."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sdpa.h")


@pytest.fixture(scope="module")
def lib():
    from scaled_dot_product_04_gb300 import _lib
    return _lib.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(sdpa_[a-z_0-9]+)\s*\(",
                                 text, flags=re.M)))


def test_header_lists_the_entry_points():
    names = declared_functions()
    for required in ("sdpa_fwd", "sdpa_varlen_fwd", "sdpa_bwd", "sdpa_varlen_bwd",
                     "sdpa_bwd_workspace_size", "sdpa_last_error"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    from scaled_dot_product_04_gb300 import _lib
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in sdpa.h but not exported"
    assert set(declared_functions()) <= set(_lib.EXPORTS) | set(declared_functions())
    assert set(_lib.EXPORTS) == set(declared_functions())


def test_version(lib):
    from scaled_dot_product_04_gb300 import _lib
    assert "sm_103a" in _lib.sdpa_version()


def _fwd(lib, q=0x10000, k=0x20000, v=0x30000, o=0x40000, lse=None, b=1, h=1, s_q=128, s_kv=128,
         d=64, scale=0.125, causal=1, dtype=0):
    return lib.sdpa_fwd(q, k, v, o, lse, b, h, s_q, s_kv, d, scale, causal, dtype, None)


def test_validation_before_any_cuda_call(lib):
    from scaled_dot_product_04_gb300 import _lib as L
    assert _fwd(lib, d=96) == L.SDPA_ERR_UNSUPPORTED
    assert "d=96" in L.sdpa_last_error()
    assert _fwd(lib, dtype=7) == L.SDPA_ERR_UNSUPPORTED
    assert _fwd(lib, b=-1) == L.SDPA_ERR_INVALID_ARG
    assert _fwd(lib, causal=2) == L.SDPA_ERR_INVALID_ARG
    assert _fwd(lib, scale=0.0) == L.SDPA_ERR_INVALID_ARG
    assert _fwd(lib, scale=float("nan")) == L.SDPA_ERR_INVALID_ARG
    assert _fwd(lib, q=0x10001) == L.SDPA_ERR_MISALIGNED
    assert _fwd(lib, q=None) == L.SDPA_ERR_INVALID_ARG
    # o overlaps q (q spans 128*64*2 bytes from 0x10000)
    assert _fwd(lib, o=0x10000 + 4096) == L.SDPA_ERR_INVALID_ARG
    assert "overlaps" in L.sdpa_last_error()
    # empty problems succeed without launching anything
    assert _fwd(lib, b=0) == L.SDPA_OK
    assert _fwd(lib, s_q=0) == L.SDPA_OK
    assert L.sdpa_last_error() == ""


def test_varlen_validation(lib):
    from scaled_dot_product_04_gb300 import _lib as L

    def call(cu_q=0x50000, cu_kv=0x60000, n=2, tq=100, tkv=100, mq=60, mkv=60, d=64):
        return lib.sdpa_varlen_fwd(0x10000, 0x20000, 0x30000, 0x40000, None, cu_q, cu_kv, n, tq,
                                   tkv, mq, mkv, 2, d, 0.125, 1, 0, None)

    assert call(cu_q=None) == L.SDPA_ERR_INVALID_ARG  # cu_seqlens_kv without cu_seqlens_q
    assert "without cu_seqlens_q" in L.sdpa_last_error()
    assert call(mq=200) == L.SDPA_ERR_INVALID_ARG
    assert call(mq=0) == L.SDPA_ERR_INVALID_ARG
    assert call(n=-1) == L.SDPA_ERR_INVALID_ARG
    assert call(cu_q=0x50002) == L.SDPA_ERR_MISALIGNED
    assert call(d=80) == L.SDPA_ERR_UNSUPPORTED
    assert call(n=0, tq=0, tkv=0, mq=0, mkv=0) == L.SDPA_OK


def test_workspace_sizes(lib):
    from scaled_dot_product_04_gb300 import _lib as L
    assert L.sdpa_bwd_workspace_size(0, 4, 128, 64) == 0
    ws = L.sdpa_bwd_workspace_size(2, 3, 100, 128)
    assert ws >= 2 * 3 * 100 * (128 + 1) * 4 and ws % 256 == 0
    assert L.sdpa_varlen_bwd_workspace_size(200, 3, 128) == ws
    assert L.sdpa_bwd_workspace_size(1, 1, 1, 96) == ctypes.c_size_t(-1).value


def test_extended_validation_before_any_cuda_call(lib):
    """The extended, FP8 and self-test entry points reject bad arguments on
    the host, before any CUDA call (so this runs without a GPU)."""
    from scaled_dot_product_04_gb300 import _lib as L

    def fwd_ex(h=4, h_kv=2, mask=1, window=-1, d=64, dtype=0, b=1):
        return lib.sdpa_fwd_ex(0x10000, 0x20000, 0x30000, 0x40000, None, b, h, h_kv, 128, 128, d,
                               0.125, mask, window, dtype, None)

    assert fwd_ex(h_kv=3) == L.SDPA_ERR_INVALID_ARG
    assert "multiple of h_kv" in L.sdpa_last_error()
    assert fwd_ex(h_kv=0) == L.SDPA_ERR_INVALID_ARG
    assert fwd_ex(mask=3) == L.SDPA_ERR_INVALID_ARG
    assert fwd_ex(window=-2) == L.SDPA_ERR_INVALID_ARG
    assert fwd_ex(d=96) == L.SDPA_ERR_UNSUPPORTED
    assert fwd_ex(b=0) == L.SDPA_OK  # empty: nothing launched

    def fwd8(d=128, out=0, dq=0x70000, dk=0x70010, dv=0x70020, so=None, scale=0.088):
        return lib.sdpa_fwd_fp8(0x10000, 0x20000, 0x30000, 0x40000, None, dq, dk, dv, so, None,
                                1, 2, 2, 128, 128, d, scale, 1, -1, out, None)

    assert fwd8(d=64) == L.SDPA_ERR_UNSUPPORTED
    assert fwd8(out=5) == L.SDPA_ERR_UNSUPPORTED
    assert fwd8(dk=None) == L.SDPA_ERR_INVALID_ARG
    assert fwd8(out=L.SDPA_FP8_E4M3) == L.SDPA_ERR_INVALID_ARG  # needs scale_o
    assert "scale_o" in L.sdpa_last_error()
    assert fwd8(scale=float("inf")) == L.SDPA_ERR_INVALID_ARG

    assert lib.sdpa_bwd_ex_workspace_size(1, 4, 128, 128, 2) == ctypes.c_size_t(-1).value
    assert lib.sdpa_selftest_wait_timeout(0, None) == L.SDPA_ERR_INVALID_ARG
    assert lib.sdpa_selftest_wait_timeout(2000001, None) == L.SDPA_ERR_INVALID_ARG
    assert "limit_us" in L.sdpa_last_error()
    assert lib.sdpa_set_forward_variant(3) == L.SDPA_ERR_INVALID_ARG
    assert lib.sdpa_set_forward_variant(0) == L.SDPA_OK


def test_problem_too_large_for_one_launch(lib):
    """Sizes whose row, tile or slice counts pass 2^31 - 1 (the TMA coordinates and
    the grid are 32-bit) are refused on the host, before any CUDA call."""
    from scaled_dot_product_04_gb300 import _lib as L
    big = 65536  # b * h = 2^32 slices
    assert _fwd(lib, b=big, h=big) == L.SDPA_ERR_INVALID_ARG
    assert "too large" in L.sdpa_last_error()
    assert lib.sdpa_fwd_ex(0x10000, 0x20000, 0x30000, 0x40000, None, big, big, big, 128, 128, 64,
                           0.125, 1, -1, 0, None) == L.SDPA_ERR_INVALID_ARG
    # backward: b * h * s_q = 2^32 accumulator rows
    rc = lib.sdpa_bwd(0x10000, 0x20000, 0x30000, 0x40000, 0x50000, 0x60000, 0x70000, 0x80000,
                      0x90000, 1, 32, 1 << 27, 128, 64, 0.125, 1, 0, 0xa0000, 1 << 20, None)
    assert rc == L.SDPA_ERR_INVALID_ARG
    assert "too large" in L.sdpa_last_error()
    # packed backward: total_q * h = 2^32 accumulator rows
    rc = lib.sdpa_varlen_bwd(0x10000, 0x20000, 0x30000, 0x40000, 0x50000, 0x60000, 0x70000,
                             0x80000, 0x90000, 0xb0000, 0xc0000, 1, 1 << 27, 1 << 27, 1 << 27,
                             1 << 27, 32, 64, 0.125, 1, 0, 0xa0000, 1 << 20, None)
    assert rc == L.SDPA_ERR_INVALID_ARG
    assert "too large" in L.sdpa_last_error()


def test_missing_library_fails_loudly(tmp_path):
    """No fallback: pointing the binding at a library that does not exist raises
    (in a fresh process, since this one may have loaded the real one)."""
    import subprocess
    import sys
    code = ("import sys; sys.path.insert(0, %r)\n"
            "from scaled_dot_product_04_gb300 import _lib\n"
            "try:\n"
            "    _lib.load(%r)\n"
            "except ImportError as e:\n"
            "    print('raised:', e)\n"
            "    sys.exit(0)\n"
            "sys.exit(1)\n") % (ROOT, str(tmp_path / "absent.so"))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and "not found" in r.stdout, r.stdout + r.stderr


def test_product_package_never_uses_the_oracle():
    """The package (binding, wrappers, build step) imports neither the oracle
    nor the test input generators: every step of the path runs in the CUDA
    library."""
    pkg = os.path.join(ROOT, "scaled_dot_product_04_gb300")
    for name in os.listdir(pkg):
        if name.endswith(".py"):
            text = open(os.path.join(pkg, name)).read()
            assert not re.search(r"^\s*(import|from)\s+(oracle|sdpa_inputs)\b", text, flags=re.M), name
