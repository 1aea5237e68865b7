"""The C ABI library loads and exports every entry point include/tvl.h
declares; host-side validation answers without a GPU."""
import ctypes
import os
import re
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tvl.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tvl_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("nvcc not available")
    from paged_kv_cache_198_gb300 import _build

    path = _build.build()
    return ctypes.CDLL(path)


def test_header_declares_the_three_hot_path_calls():
    names = _declared()
    for n in ("tvl_paged_kv_write", "tvl_paged_attention_decode",
              "tvl_paged_attention_prefill"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings_and_version(lib):
    lib.tvl_status_string.restype = ctypes.c_char_p
    lib.tvl_status_string.argtypes = [ctypes.c_int]
    assert lib.tvl_status_string(0) == b"ok"
    assert lib.tvl_status_string(3).startswith(b"workspace")
    lib.tvl_version.restype = ctypes.c_int
    assert lib.tvl_version() >= 100


def test_validation_rejects_before_any_cuda_call(lib):
    import paged_kv_cache_198_gb300 as tvl

    P = ctypes.c_void_p
    dummy = P(16)
    # head_dim 128 is not supported
    rc = lib.tvl_paged_kv_write(dummy, dummy, dummy, dummy, dummy, 4, 8, 128, 16, 4, P(0))
    assert rc == tvl.ERR_UNSUPPORTED
    # misaligned cache pointer
    rc = lib.tvl_paged_kv_write(dummy, dummy, P(18), dummy, dummy, 4, 8, 64, 16, 4, P(0))
    assert rc == tvl.ERR_INVALID_ARG
    # block_size 24 unsupported by the decode
    size = ctypes.c_size_t(0)
    lib.tvl_paged_attention_decode_workspace_size.argtypes = [ctypes.c_int] * 7 + [
        ctypes.POINTER(ctypes.c_size_t)]
    rc = lib.tvl_paged_attention_decode_workspace_size(4, 32, 8, 64, 16, 24, 0,
                                                       ctypes.byref(size))
    assert rc == tvl.ERR_UNSUPPORTED
    # partition not a multiple of the block size
    rc = lib.tvl_paged_attention_decode_workspace_size(4, 32, 8, 64, 16, 16, 100,
                                                       ctypes.byref(size))
    assert rc == tvl.ERR_INVALID_ARG
    # fixed partition needing no split: no workspace, no device query
    rc = lib.tvl_paged_attention_decode_workspace_size(4, 32, 8, 64, 16, 16, 256,
                                                       ctypes.byref(size))
    assert rc == 0 and size.value == 0
    # 512-token windows over 8192 blocks of 16: S * 256 records of Hq * (D + 2) floats
    rc = lib.tvl_paged_attention_decode_workspace_size(8, 32, 8, 64, 8192, 16, 512,
                                                       ctypes.byref(size))
    assert rc == 0 and size.value >= 8 * 256 * 32 * 66 * 4
    # GQA group 3 is not supported
    rc = lib.tvl_paged_attention_decode_workspace_size(4, 24, 8, 64, 16, 16, 512,
                                                       ctypes.byref(size))
    assert rc == tvl.ERR_UNSUPPORTED


def test_decode_step_validation_before_any_cuda_call(lib):
    import paged_kv_cache_198_gb300 as tvl

    P, I, F, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.tvl_paged_decode_step.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, F, I, P,
                                          SZ, P]
    lib.tvl_paged_decode_step.restype = I
    d = P(256)
    # no new K / V for a step with sequences
    rc = lib.tvl_paged_decode_step(d, d, None, None, d, d, d, d, 4, 32, 8, 64, 16, 64, 16,
                                   0.125, 256, None, 0, None)
    assert rc == tvl.ERR_INVALID_ARG
    # misaligned new K
    rc = lib.tvl_paged_decode_step(d, d, P(258), d, d, d, d, d, 4, 32, 8, 64, 16, 64, 16,
                                   0.125, 256, None, 0, None)
    assert rc == tvl.ERR_INVALID_ARG
    # unsupported block size is reported as such
    rc = lib.tvl_paged_decode_step(d, d, d, d, d, d, d, d, 4, 32, 8, 64, 24, 64, 16,
                                   0.125, 240, None, 0, None)
    assert rc == tvl.ERR_UNSUPPORTED
