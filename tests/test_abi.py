"""The C-ABI library builds for sm_103a, loads, and exports every function the
public header declares (no compute calls: no GPU needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "llama_block.h")


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(llama_[a-z_]+)\s*\(", text)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib_path():
    from dense_decoder_block_gb300 import build
    return build.build()


def test_header_declares_the_block_api():
    names = _declared_functions()
    for must in ("llama_block_create", "llama_block_prefill", "llama_block_decode", "llama_block_destroy",
                 "llama_block_workspace_bytes", "llama_block_decode_devpos", "llama_block_poll_error"):
        assert must in names


def test_library_exports_every_declared_symbol(lib_path):
    lib = ctypes.CDLL(lib_path)
    for name in _declared_functions():
        assert hasattr(lib, name), f"{name} declared in llama_block.h but not exported"


def test_binding_covers_exactly_the_header(lib_path):
    from dense_decoder_block_gb300 import _native
    assert sorted(_native.SIGNATURES) == _declared_functions()
    lib = _native.load(lib_path)
    for name in _native.SIGNATURES:
        assert getattr(lib, name).argtypes is not None


def test_null_arguments_are_rejected_without_a_gpu(lib_path):
    from dense_decoder_block_gb300 import _native
    lib = _native.load(lib_path)
    h = ctypes.c_void_p()
    assert lib.llama_block_create(None, None, ctypes.byref(h)) == _native.LLAMA_ERR_INVALID_ARG
    dims = _native.llama_block_dims(4096, 32, 7, 128, 14336, 1024, 1e-5, 5e5, _native.LLAMA_BF16)
    w = _native.llama_block_weights()
    assert lib.llama_block_create(ctypes.byref(dims), ctypes.byref(w), ctypes.byref(h)) == \
        _native.LLAMA_ERR_UNSUPPORTED_DIMS
    dims = _native.llama_block_dims(4096, 32, 8, 64, 14336, 1024, 1e-5, 5e5, _native.LLAMA_BF16)
    assert lib.llama_block_create(ctypes.byref(dims), ctypes.byref(w), ctypes.byref(h)) == \
        _native.LLAMA_ERR_UNSUPPORTED_DIMS
    dims = _native.llama_block_dims(4096, 32, 8, 128, 14336, 1024, 1e-5, 5e5, _native.LLAMA_BF16)
    assert lib.llama_block_create(ctypes.byref(dims), ctypes.byref(w), ctypes.byref(h)) == \
        _native.LLAMA_ERR_INVALID_ARG
    assert lib.llama_block_workspace_bytes(None, 1, 1) == 0
    assert lib.llama_block_prefill(None, None, 1, 1, None, None, None, 0, None) == _native.LLAMA_ERR_INVALID_ARG
    assert lib.llama_lmhead_workspace_bytes(0, 4096, 128256) == 0
    assert lib.llama_embed(None, 1, None, 10, 4096, None, None, None) == _native.LLAMA_ERR_INVALID_ARG
    assert lib.llama_block_decode_seqpos(None, None, 1, None, None, None, None, 0, None) == \
        _native.LLAMA_ERR_INVALID_ARG
    assert lib.llama_block_launch_count(None) == 0
    assert lib.llama_block_workspace_offsets(None, 1, 1, None, 6) == _native.LLAMA_ERR_INVALID_ARG
    assert lib.llama_sample(None, 1, 10, ctypes.c_float(1.0), 0, ctypes.c_float(1.0), None, None, None) == \
        _native.LLAMA_ERR_INVALID_ARG
    assert lib.llama_sample(None, 1, 10, ctypes.c_float(-1.0), 0, ctypes.c_float(1.0), None, None, None) == \
        _native.LLAMA_ERR_INVALID_ARG
    assert lib.llama_block_create_scaled(None, None, None, ctypes.byref(h)) == _native.LLAMA_ERR_INVALID_ARG
    dev = ctypes.c_void_p(1)
    assert lib.llama_device_ptr_of_host(None, ctypes.byref(dev)) == _native.LLAMA_ERR_INVALID_ARG
    assert lib.llama_block_set_stage_events(None, None, 0) == _native.LLAMA_ERR_INVALID_ARG
    assert lib.llama_block_selftest_wait_timeout(None, 1000000, None) == _native.LLAMA_ERR_INVALID_ARG


def test_product_package_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "dense_decoder_block_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                src = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in re.findall(r"(?:import|from)\s+(\w+)", src), f
