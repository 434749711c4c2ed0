"""GB300 (sm_103a) Llama-3-style decoder block: Python binding of libllama_block.so.

The functions here keep the C ABI's names and only marshal arguments (torch
tensors -> device pointers, the current CUDA stream -> cudaStream_t); every
step of the block runs in the library's CUDA kernels.  There is no fallback:
importing works without the library, but every call raises if it is missing.

    blk = LlamaBlock(dims, weights)            # weights: dict of CUDA tensors
    ws = blk.workspace(batch, tokens)
    blk.prefill(x, kv, y, ws)                  # x, y [B, T, d]
    blk.decode(x, kv, pos, y, ws)              # x, y [B, 1, d]
"""
from __future__ import annotations

import ctypes as C
from typing import Dict, Optional

import torch

from . import _native
from ._native import (LLAMA_BF16, LLAMA_F32, LLAMA_OK, LLAMA_ERR_INVALID_ARG, LLAMA_ERR_UNSUPPORTED_DIMS,
                      LLAMA_ERR_POS_RANGE, LLAMA_ERR_WORKSPACE, LLAMA_ERR_CUDA, LLAMA_ERR_DEVICE_TIMEOUT,
                      llama_block_dims, llama_block_weights, llama_kv_cache, llama_rope_scaling)

__all__ = [
    "LlamaBlock", "LlamaError", "KVCache", "lib", "llama_block_create", "llama_block_create_scaled",
    "llama_block_destroy",
    "llama_block_workspace_bytes", "llama_block_workspace_offsets", "llama_block_prefill", "llama_block_prefill_at", "llama_block_decode",
    "llama_block_decode_devpos", "llama_block_decode_seqpos",
    "llama_block_poll_error", "llama_block_last_error", "llama_block_selftest_wait_timeout", "Trace", "llama_block_set_stage_events", "llama_block_launch_count", "HostMapped",
    "llama_embed", "llama_lmhead_workspace_bytes",
    "llama_lmhead_argmax", "llama_lmhead_argmax_noalloc", "llama_sample", "llama_rmsnorm", "LLAMA_BF16", "LLAMA_F32",
]


class LlamaError(RuntimeError):
    def __init__(self, code: int, msg: str = ""):
        self.code = code
        super().__init__(f"{_native.ERROR_NAMES.get(code, code)}: {msg}")


def lib():
    return _native.load()


class HostMapped:
    """A pinned host tensor seen through its device address: passed as x or y of
    prefill/decode, the kernels read or write the host memory directly."""

    def __init__(self, t: torch.Tensor):
        if t.is_cuda or not t.is_pinned():
            raise ValueError("HostMapped needs a pinned host tensor")
        if not t.is_contiguous():
            raise ValueError("HostMapped needs a contiguous tensor")
        dev = C.c_void_p()
        rc = lib().llama_device_ptr_of_host(C.c_void_p(t.data_ptr()), C.byref(dev))
        if rc != LLAMA_OK or not dev.value:
            raise LlamaError(rc, "llama_device_ptr_of_host: not pinned and mapped")
        self.t = t
        self.dev_ptr = dev.value
        self.shape = t.shape


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, HostMapped):
        return C.c_void_p(t.dev_ptr)
    if not t.is_cuda:
        raise ValueError("tensors passed to the block library must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensors passed to the block library must be contiguous")
    return C.c_void_p(t.data_ptr())


def _stream(stream: Optional[torch.cuda.Stream] = None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream)


def _dtype_code(dt: torch.dtype) -> int:
    if dt == torch.bfloat16:
        return LLAMA_BF16
    if dt == torch.float32:
        return LLAMA_F32
    raise ValueError(f"unsupported dtype {dt}")


# ----------------------------------------------------------------------------- same-named wrappers

def llama_block_create(dims: llama_block_dims, weights: llama_block_weights) -> C.c_void_p:
    h = C.c_void_p()
    rc = lib().llama_block_create(C.byref(dims), C.byref(weights), C.byref(h))
    if rc != LLAMA_OK:
        raise LlamaError(rc, "llama_block_create")
    return h


def llama_block_create_scaled(dims: llama_block_dims, weights: llama_block_weights,
                              scaling: Optional[llama_rope_scaling]) -> C.c_void_p:
    h = C.c_void_p()
    rc = lib().llama_block_create_scaled(C.byref(dims), C.byref(weights),
                                         C.byref(scaling) if scaling is not None else None, C.byref(h))
    if rc != LLAMA_OK:
        raise LlamaError(rc, "llama_block_create_scaled")
    return h


def llama_block_destroy(h) -> None:
    lib().llama_block_destroy(h)


def llama_block_workspace_bytes(h, batch: int, tokens: int) -> int:
    return int(lib().llama_block_workspace_bytes(h, batch, tokens))


INTERMEDIATES = ("xn", "q", "o", "h", "hn", "u")


def llama_block_workspace_offsets(h, batch: int, tokens: int):
    """Byte offsets in the workspace of xn, q, o, h, hn, u for a call of this shape."""
    arr = (C.c_size_t * _native.LLAMA_BLOCK_INTERMEDIATES)()
    rc = lib().llama_block_workspace_offsets(h, batch, tokens, arr, _native.LLAMA_BLOCK_INTERMEDIATES)
    if rc != _native.LLAMA_BLOCK_INTERMEDIATES:
        raise LlamaError(rc, "llama_block_workspace_offsets")
    return dict(zip(INTERMEDIATES, (int(v) for v in arr)))


def llama_block_last_error(h) -> str:
    r = lib().llama_block_last_error(h)
    return r.decode() if r else ""


def _check(h, rc, what):
    if rc != LLAMA_OK:
        raise LlamaError(rc, f"{what}: {llama_block_last_error(h)}")


def llama_block_prefill(h, x, batch, tokens, kv: llama_kv_cache, y, ws, ws_bytes, stream=None) -> None:
    _check(h, lib().llama_block_prefill(h, _ptr(x), batch, tokens, C.byref(kv), _ptr(y), _ptr(ws), ws_bytes,
                                        _stream(stream)), "llama_block_prefill")


def llama_block_prefill_at(h, x, batch, tokens, start_pos, kv: llama_kv_cache, y, ws, ws_bytes, stream=None) -> None:
    _check(h, lib().llama_block_prefill_at(h, _ptr(x), batch, tokens, start_pos, C.byref(kv), _ptr(y), _ptr(ws),
                                           ws_bytes, _stream(stream)), "llama_block_prefill_at")


def llama_block_decode(h, x, batch, kv: llama_kv_cache, pos, y, ws, ws_bytes, stream=None) -> None:
    _check(h, lib().llama_block_decode(h, _ptr(x), batch, C.byref(kv), int(pos), _ptr(y), _ptr(ws), ws_bytes,
                                       _stream(stream)), "llama_block_decode")


def llama_block_decode_devpos(h, x, batch, kv: llama_kv_cache, pos_dev, y, ws, ws_bytes, stream=None) -> None:
    _check(h, lib().llama_block_decode_devpos(h, _ptr(x), batch, C.byref(kv), _ptr(pos_dev), _ptr(y), _ptr(ws),
                                              ws_bytes, _stream(stream)), "llama_block_decode_devpos")


def llama_block_decode_seqpos(h, x, batch, kv: llama_kv_cache, pos_seq, y, ws, ws_bytes, stream=None) -> None:
    _check(h, lib().llama_block_decode_seqpos(h, _ptr(x), batch, C.byref(kv), _ptr(pos_seq), _ptr(y), _ptr(ws),
                                              ws_bytes, _stream(stream)), "llama_block_decode_seqpos")


def llama_block_set_stage_events(h, events) -> None:
    """events: None, or a list of LLAMA_BLOCK_STAGES + 1 torch.cuda.Event (enable_timing=True)."""
    if events is None:
        rc = lib().llama_block_set_stage_events(h, None, 0)
    else:
        arr = (C.c_void_p * len(events))(*[C.c_void_p(e.cuda_event) for e in events])
        rc = lib().llama_block_set_stage_events(h, arr, len(events))
    if rc != LLAMA_OK:
        raise LlamaError(rc, "llama_block_set_stage_events")


def llama_block_launch_count(h) -> int:
    """Kernels enqueued by the last successful prefill/decode call on the handle."""
    return int(lib().llama_block_launch_count(h))


def llama_block_poll_error(h, stream=None) -> int:
    return int(lib().llama_block_poll_error(h, _stream(stream)))


class Trace:
    """Per-CTA timeline of the block's kernels while the context is open
    (llama_trace_begin / llama_trace_end; the trace build of the library only:
    load it with `_native.load(build.build(trace=True))` before the first call).
    After exit, `records()` gives the columns kernel, sm, cta, t_start,
    t_release, t_end (ns) on the host."""

    def __init__(self, capacity: int = 1 << 16, device=None):
        import torch
        dev = device if device is not None else torch.device("cuda", torch.cuda.current_device())
        self.capacity = int(capacity)
        self.buf = torch.zeros(self.capacity, 4, dtype=torch.int64, device=dev)
        self.count = torch.zeros(1, dtype=torch.int32, device=dev)

    def __enter__(self):
        rc = lib().llama_trace_begin(_ptr(self.buf), _ptr(self.count), self.capacity)
        if rc != LLAMA_OK:
            raise LlamaError(rc, "llama_trace_begin")
        return self

    def __exit__(self, *exc):
        lib().llama_trace_end()
        return False

    def records(self):
        import torch
        torch.cuda.synchronize(self.buf.device)
        n = min(int(self.count.item()), self.capacity)
        r = self.buf[:n].cpu()
        w0 = r[:, 0]
        return {"kernel": (w0 & 0xffff).tolist(), "sm": ((w0 >> 16) & 0xffff).tolist(),
                "cta": ((w0 >> 32) & 0xffffffff).tolist(), "t_start": r[:, 1].tolist(),
                "t_release": r[:, 2].tolist(), "t_end": r[:, 3].tolist(), "claimed": int(self.count.item())}


def llama_block_selftest_wait_timeout(h, budget_ns, stream=None) -> None:
    _check(h, lib().llama_block_selftest_wait_timeout(h, int(budget_ns), _stream(stream)),
           "llama_block_selftest_wait_timeout")


def llama_rmsnorm(x, g, y, rows, d, eps, stream=None) -> None:
    rc = lib().llama_rmsnorm(_ptr(x), _ptr(g), _ptr(y), rows, d, C.c_float(eps), _dtype_code(x.dtype),
                             _stream(stream))
    if rc != LLAMA_OK:
        raise LlamaError(rc, "llama_rmsnorm")


def llama_embed(ids, n_tokens, w_embed, vocab, d_model, x, err_dev=None, stream=None) -> None:
    rc = lib().llama_embed(_ptr(ids), n_tokens, _ptr(w_embed), vocab, d_model, _ptr(x), _ptr(err_dev),
                           _stream(stream))
    if rc != LLAMA_OK:
        raise LlamaError(rc, "llama_embed")


def llama_lmhead_workspace_bytes(batch, d_model, vocab) -> int:
    return int(lib().llama_lmhead_workspace_bytes(batch, d_model, vocab))


def llama_lmhead_argmax(h, batch, h_stride, g_final, w_out, vocab, d_model, eps, ids, logits, ws, ws_bytes,
                        stream=None) -> None:
    rc = lib().llama_lmhead_argmax(_ptr(h), batch, h_stride, _ptr(g_final), _ptr(w_out), vocab, d_model,
                                   C.c_float(eps), _ptr(ids), _ptr(logits), _ptr(ws), ws_bytes, _stream(stream))
    if rc != LLAMA_OK:
        raise LlamaError(rc, "llama_lmhead_argmax")


def llama_lmhead_argmax_noalloc(h, batch, h_stride, g_final, w_out, vocab, d_model, eps, ids, logits,
                                stream=None) -> None:
    """The LM head + greedy choice without a workspace (library-owned scratch; see the header)."""
    rc = lib().llama_lmhead_argmax_noalloc(_ptr(h), batch, h_stride, _ptr(g_final), _ptr(w_out), vocab, d_model,
                                           C.c_float(eps), _ptr(ids), _ptr(logits), _stream(stream))
    if rc != LLAMA_OK:
        raise LlamaError(rc, "llama_lmhead_argmax_noalloc")


def llama_sample(logits, batch, vocab, temperature, top_k, top_p, uniforms, ids, stream=None) -> None:
    """ids[b] drawn from softmax(logits[b] / temperature) after top-k / top-p, with uniforms[b]."""
    rc = lib().llama_sample(_ptr(logits), batch, vocab, C.c_float(temperature), int(top_k), C.c_float(top_p),
                            _ptr(uniforms), _ptr(ids), _stream(stream))
    if rc != LLAMA_OK:
        raise LlamaError(rc, "llama_sample")


# ----------------------------------------------------------------------------- convenience

class KVCache:
    """K and V buffers [batch, n_kv_heads, max_seq, head_dim] (caller-owned torch tensors)."""

    def __init__(self, k: torch.Tensor, v: torch.Tensor):
        assert k.shape == v.shape and k.dim() == 4
        self.k, self.v = k, v
        self.c = llama_kv_cache(C.c_void_p(k.data_ptr()), C.c_void_p(v.data_ptr()), k.shape[0], k.shape[2])


class LlamaBlock:
    """Owns a handle; borrows the weight tensors (kept referenced here)."""

    def __init__(self, dims, weights: Dict[str, torch.Tensor], gains: Dict[str, torch.Tensor], max_seq: int):
        dt = weights["wq"].dtype
        self.dims = dims
        self._keep = dict(weights, **gains)
        self.c_dims = llama_block_dims(dims.d_model, dims.n_heads, dims.n_kv_heads, dims.head_dim, dims.d_ff,
                                       max_seq, dims.eps, dims.rope_theta, _dtype_code(dt))
        names = ("g_attn", "wq", "wk", "wv", "wo", "g_ffn", "w_gate", "w_up", "w_down")
        self.c_w = llama_block_weights(*[_ptr(self._keep[n]) for n in names])
        sc = getattr(dims, "rope_scaling", None)   # (factor, low, high, original context) or None
        self.c_scaling = None if sc is None else llama_rope_scaling(float(sc[0]), float(sc[1]), float(sc[2]),
                                                                    int(sc[3]))
        self.h = llama_block_create_scaled(self.c_dims, self.c_w, self.c_scaling)

    def __del__(self):
        h = getattr(self, "h", None)
        if h is not None and _native._lib is not None:
            llama_block_destroy(h)
            self.h = None

    def workspace_bytes(self, batch: int, tokens: int) -> int:
        return llama_block_workspace_bytes(self.h, batch, tokens)

    def workspace(self, batch: int, tokens: int, device=None) -> torch.Tensor:
        n = self.workspace_bytes(batch, tokens)
        return torch.empty(n, dtype=torch.uint8, device=device or self._keep["wq"].device)

    def intermediates(self, ws: torch.Tensor, batch: int, tokens: int) -> Dict[str, torch.Tensor]:
        """Views of the workspace `ws` of a finished call (batch, tokens) as the block's
        intermediates xn, q, o, h, hn, u, each [batch * tokens, width]."""
        off = llama_block_workspace_offsets(self.h, batch, tokens)
        d = self.dims
        dt = self._keep["wq"].dtype
        es = torch.finfo(dt).bits // 8
        widths = {"xn": d.d_model, "q": d.q_dim, "o": d.q_dim, "h": d.d_model, "hn": d.d_model, "u": d.d_ff}
        M = batch * tokens
        out = {}
        for name, width in widths.items():
            nbytes = M * width * es
            out[name] = ws[off[name]:off[name] + nbytes].view(dt).view(M, width)
        return out

    def prefill(self, x, kv: KVCache, y, ws, stream=None):
        B, T = x.shape[0], x.shape[1]
        llama_block_prefill(self.h, x, B, T, kv.c, y, ws, ws.numel(), stream)

    def prefill_at(self, x, kv: KVCache, start_pos: int, y, ws, stream=None):
        """x [B, T, d] holds the tokens at positions start_pos .. start_pos + T - 1."""
        B, T = x.shape[0], x.shape[1]
        llama_block_prefill_at(self.h, x, B, T, start_pos, kv.c, y, ws, ws.numel(), stream)

    def decode(self, x, kv: KVCache, pos: int, y, ws, stream=None):
        llama_block_decode(self.h, x, x.shape[0], kv.c, pos, y, ws, ws.numel(), stream)

    def decode_devpos(self, x, kv: KVCache, pos_dev, y, ws, stream=None):
        llama_block_decode_devpos(self.h, x, x.shape[0], kv.c, pos_dev, y, ws, ws.numel(), stream)

    def decode_seqpos(self, x, kv: KVCache, pos_seq, y, ws, stream=None):
        """pos_seq: int32 CUDA tensor [batch], sequence b at position pos_seq[b]."""
        llama_block_decode_seqpos(self.h, x, x.shape[0], kv.c, pos_seq, y, ws, ws.numel(), stream)

    def poll_error(self, stream=None) -> int:
        return llama_block_poll_error(self.h, stream)

    def selftest_wait_timeout(self, budget_ns, stream=None) -> None:
        llama_block_selftest_wait_timeout(self.h, budget_ns, stream)

    def launch_count(self) -> int:
        return llama_block_launch_count(self.h)
