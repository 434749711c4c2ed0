"""ctypes declarations of libllama_block.so (the C ABI in include/llama_block.h)."""
from __future__ import annotations

import ctypes as C
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libllama_block.so")

LLAMA_OK = 0
LLAMA_ERR_INVALID_ARG = -1
LLAMA_ERR_UNSUPPORTED_DIMS = -2
LLAMA_ERR_POS_RANGE = -3
LLAMA_ERR_WORKSPACE = -4
LLAMA_ERR_CUDA = -5
LLAMA_ERR_DEVICE_TIMEOUT = -6
LLAMA_F32 = 0
LLAMA_BF16 = 1
LLAMA_BLOCK_INTERMEDIATES = 6

ERROR_NAMES = {
    LLAMA_ERR_INVALID_ARG: "LLAMA_ERR_INVALID_ARG",
    LLAMA_ERR_UNSUPPORTED_DIMS: "LLAMA_ERR_UNSUPPORTED_DIMS",
    LLAMA_ERR_POS_RANGE: "LLAMA_ERR_POS_RANGE",
    LLAMA_ERR_WORKSPACE: "LLAMA_ERR_WORKSPACE",
    LLAMA_ERR_CUDA: "LLAMA_ERR_CUDA",
    LLAMA_ERR_DEVICE_TIMEOUT: "LLAMA_ERR_DEVICE_TIMEOUT",
}


class llama_block_dims(C.Structure):
    _fields_ = [("d_model", C.c_int32), ("n_heads", C.c_int32), ("n_kv_heads", C.c_int32),
                ("head_dim", C.c_int32), ("d_ff", C.c_int32), ("max_seq", C.c_int32),
                ("eps", C.c_float), ("rope_theta", C.c_float), ("dtype", C.c_int32)]


class llama_block_weights(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in ("g_attn", "wq", "wk", "wv", "wo", "g_ffn", "w_gate", "w_up", "w_down")]


class llama_rope_scaling(C.Structure):
    _fields_ = [("factor", C.c_float), ("low_freq_factor", C.c_float), ("high_freq_factor", C.c_float),
                ("original_max_pos", C.c_int32)]


class llama_kv_cache(C.Structure):
    _fields_ = [("k", C.c_void_p), ("v", C.c_void_p), ("batch", C.c_int32), ("max_seq", C.c_int32)]


# name -> (restype, argtypes); the exact set of symbols include/llama_block.h declares
SIGNATURES = {
    "llama_block_create": (C.c_int, [C.POINTER(llama_block_dims), C.POINTER(llama_block_weights),
                                     C.POINTER(C.c_void_p)]),
    "llama_block_create_scaled": (C.c_int, [C.POINTER(llama_block_dims), C.POINTER(llama_block_weights),
                                            C.POINTER(llama_rope_scaling), C.POINTER(C.c_void_p)]),
    "llama_block_destroy": (None, [C.c_void_p]),
    "llama_block_workspace_bytes": (C.c_size_t, [C.c_void_p, C.c_int, C.c_int]),
    "llama_block_workspace_offsets": (C.c_int, [C.c_void_p, C.c_int, C.c_int, C.POINTER(C.c_size_t), C.c_int]),
    "llama_block_prefill": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.POINTER(llama_kv_cache),
                                      C.c_void_p, C.c_void_p, C.c_size_t, C.c_void_p]),
    "llama_block_prefill_at": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.c_int,
                                         C.POINTER(llama_kv_cache), C.c_void_p, C.c_void_p, C.c_size_t,
                                         C.c_void_p]),
    "llama_block_decode": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int, C.POINTER(llama_kv_cache), C.c_int,
                                     C.c_void_p, C.c_void_p, C.c_size_t, C.c_void_p]),
    "llama_block_decode_devpos": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int, C.POINTER(llama_kv_cache),
                                            C.c_void_p, C.c_void_p, C.c_void_p, C.c_size_t, C.c_void_p]),
    "llama_block_decode_seqpos": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int, C.POINTER(llama_kv_cache),
                                            C.c_void_p, C.c_void_p, C.c_void_p, C.c_size_t, C.c_void_p]),
    "llama_block_poll_error": (C.c_int, [C.c_void_p, C.c_void_p]),
    "llama_block_last_error": (C.c_char_p, [C.c_void_p]),
    "llama_block_selftest_wait_timeout": (C.c_int, [C.c_void_p, C.c_ulonglong, C.c_void_p]),
    "llama_trace_begin": (C.c_int, [C.c_void_p, C.c_void_p, C.c_uint]),
    "llama_trace_end": (C.c_int, []),
    "llama_block_set_stage_events": (C.c_int, [C.c_void_p, C.POINTER(C.c_void_p), C.c_int]),
    "llama_block_launch_count": (C.c_int, [C.c_void_p]),
    "llama_device_ptr_of_host": (C.c_int, [C.c_void_p, C.POINTER(C.c_void_p)]),
    "llama_embed": (C.c_int, [C.c_void_p, C.c_int, C.c_void_p, C.c_int, C.c_int, C.c_void_p, C.c_void_p,
                              C.c_void_p]),
    "llama_lmhead_workspace_bytes": (C.c_size_t, [C.c_int, C.c_int, C.c_int]),
    "llama_lmhead_argmax": (C.c_int, [C.c_void_p, C.c_int, C.c_int, C.c_void_p, C.c_void_p, C.c_int, C.c_int,
                                      C.c_float, C.c_void_p, C.c_void_p, C.c_void_p, C.c_size_t, C.c_void_p]),
    "llama_lmhead_argmax_noalloc": (C.c_int, [C.c_void_p, C.c_int, C.c_int, C.c_void_p, C.c_void_p, C.c_int,
                                              C.c_int, C.c_float, C.c_void_p, C.c_void_p, C.c_void_p]),
    "llama_sample": (C.c_int, [C.c_void_p, C.c_int, C.c_int, C.c_float, C.c_int, C.c_float, C.c_void_p,
                               C.c_void_p, C.c_void_p]),
    "llama_rmsnorm": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.c_float, C.c_int,
                                C.c_void_p]),
}

_lib = None


def load(path: str = LIB_PATH):
    """Load the shared library; raise if it is missing (there is no fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with `python -m dense_decoder_block_gb300.build` "
                          "(the block has no CPU or PyTorch fallback)")
    lib = C.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib
