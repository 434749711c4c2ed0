"""Seeded synthetic inputs for the Llama-3-style decoder block workloads.

This module is shared by the tests, the benchmark and the CPU oracle's callers.
It holds shapes and random draws only: none of the block's arithmetic lives
here (no norm, projection, rotation, attention or activation).

Shapes follow the pages:
  * tiny block: d=256, 4 query / 2 KV heads, head_dim 64, d_ff 768;
  * 8B block: d=4096, 32 query / 8 KV heads, head_dim 128, d_ff 14336
    ("Llama 3 8B · Prepare Q, K, V", sku_list arch_args; "How Llama 3.1
    Generates the Next Token", Weight dimensions);
  * 70B block: d=8192, 64 query / 8 KV heads, head_dim 128, d_ff 28672
    ("Llama 3.1 70B", Grouped-Query Attention and SwiGLU MLP boxes).

Draw recipe (torch CPU generators): the seven projection matrices in ABI
order (wq, wk, wv, wo, w_gate, w_up, w_down) from a generator seeded with
``seed`` (0 by default), the activations x from ``seed + 1``, then the K and
V cache rows that precede the first decode position from ``seed + 2``.  The
weights therefore do not depend on the batch size.  Every draw is fp32
N(0, std) from ``torch.randn``; bf16 workloads round it to bf16
(round-to-nearest-even) and both the GPU path and the oracle consume those
rounded values.  RMSNorm gains are ones (the page's init) unless
``random_gains`` is set, in which case they are U(0.5, 1.5) drawn after the
matrices.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, Optional

import torch

WEIGHT_NAMES = ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down")
GAIN_NAMES = ("g_attn", "g_ffn")


@dataclasses.dataclass(frozen=True)
class BlockDims:
    d_model: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    d_ff: int
    eps: float = 1e-5
    rope_theta: float = 500000.0
    # None, or Llama 3.1's long-context RoPE schedule as
    # (factor, low_freq_factor, high_freq_factor, original_context)
    rope_scaling: Optional[tuple] = None

    @property
    def q_dim(self) -> int:
        return self.n_heads * self.head_dim

    @property
    def kv_dim(self) -> int:
        return self.n_kv_heads * self.head_dim

    def weight_shapes(self) -> Dict[str, tuple]:
        """[out, in] row-major, as torch.nn.Linear stores them."""
        d, q, kv, f = self.d_model, self.q_dim, self.kv_dim, self.d_ff
        return {
            "wq": (q, d), "wk": (kv, d), "wv": (kv, d), "wo": (d, q),
            "w_gate": (f, d), "w_up": (f, d), "w_down": (d, f),
        }


TINY = BlockDims(256, 4, 2, 64, 768)
LLAMA3_8B = BlockDims(4096, 32, 8, 128, 14336)
LLAMA31_70B = BlockDims(8192, 64, 8, 128, 28672)
VOCAB = 128256
# Llama 3.1's released RoPE scaling configuration (the pages name the x8 factor only)
LLAMA31_ROPE_SCALING = (8.0, 1.0, 4.0, 8192)


def _randn(gen: torch.Generator, shape, std: float, dtype: torch.dtype) -> torch.Tensor:
    t = torch.randn(*shape, generator=gen, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(dtype)


@dataclasses.dataclass
class BlockInputs:
    dims: BlockDims
    dtype: torch.dtype
    x: torch.Tensor                     # [B, T, d]
    weights: Dict[str, torch.Tensor]    # [out, in]
    gains: Dict[str, torch.Tensor]      # [d]
    k_cache: Optional[torch.Tensor]     # [B, Hkv, S_max, dh]
    v_cache: Optional[torch.Tensor]
    start_pos: int


def make_weights(dims: BlockDims, *, dtype=torch.bfloat16, weight_std: float = 0.02, seed: int = 0,
                 random_gains: bool = False):
    """The seven projection matrices (ABI order, fp32 N(0, weight_std) rounded to
    ``dtype``) and the two RMSNorm gains (ones, or U(0.5, 1.5) drawn after the
    matrices when ``random_gains``).  Generator seeded with ``seed``."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    weights = {}
    for name in WEIGHT_NAMES:
        weights[name] = _randn(gen, dims.weight_shapes()[name], weight_std, dtype)
    if random_gains:
        gains = {n: (torch.rand(dims.d_model, generator=gen) + 0.5).to(dtype) for n in GAIN_NAMES}
    else:
        gains = {n: torch.ones(dims.d_model, dtype=dtype) for n in GAIN_NAMES}
    return weights, gains


def make_x(batch: int, tokens: int, d_model: int, *, dtype=torch.bfloat16, seed: int = 1) -> torch.Tensor:
    """Block input x [B, T, d], N(0, 1), generator seeded with ``seed``."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    return _randn(gen, (batch, tokens, d_model), 1.0, dtype)


def make_cache(dims: BlockDims, batch: int, max_seq: int, cache_len: int, tokens: int, *, dtype=torch.bfloat16,
               seed: int = 2, poison_tail: bool = True):
    """K and V caches [B, Hkv, max_seq, dh]: rows 0..cache_len-1 N(0, 1) (K first,
    then V, generator seeded with ``seed``; taken as already-rotated keys), rows
    cache_len..cache_len+tokens-1 zero (the call writes them), the rest NaN when
    ``poison_tail`` so that any read past the attended range shows."""
    shape = (batch, dims.n_kv_heads, max_seq, dims.head_dim)
    k_cache = torch.zeros(shape, dtype=dtype)
    v_cache = torch.zeros(shape, dtype=dtype)
    if cache_len > 0:
        gen = torch.Generator(device="cpu")
        gen.manual_seed(seed)
        k_cache[:, :, :cache_len] = _randn(gen, (batch, dims.n_kv_heads, cache_len, dims.head_dim), 1.0, dtype)
        v_cache[:, :, :cache_len] = _randn(gen, (batch, dims.n_kv_heads, cache_len, dims.head_dim), 1.0, dtype)
    if poison_tail and cache_len + tokens < max_seq:
        k_cache[:, :, cache_len + tokens:] = float("nan")
        v_cache[:, :, cache_len + tokens:] = float("nan")
    return k_cache, v_cache


def make_block_inputs(dims: BlockDims, batch: int, tokens: int, *, dtype=torch.bfloat16,
                      weight_std: float = 0.02, cache_len: int = 0, max_seq: Optional[int] = None,
                      seed: int = 0, random_gains: bool = False, poison_tail: bool = True,
                      device: str = "cpu", weights=None) -> BlockInputs:
    """One workload: weights (seed), x (seed + 1), cache (seed + 2).  ``tokens``
    rows of x per sequence start at position ``cache_len``.  Pass ``weights`` =
    (weights, gains) to reuse already drawn matrices."""
    if weights is None:
        weights = make_weights(dims, dtype=dtype, weight_std=weight_std, seed=seed, random_gains=random_gains)
    w, gains = weights
    x = make_x(batch, tokens, dims.d_model, dtype=dtype, seed=seed + 1)
    if max_seq is None:
        max_seq = cache_len + tokens
    k_cache, v_cache = make_cache(dims, batch, max_seq, cache_len, tokens, dtype=dtype, seed=seed + 2,
                                  poison_tail=poison_tail)
    inp = BlockInputs(dims, dtype, x, w, gains, k_cache, v_cache, cache_len)
    if device != "cpu":
        inp = to_device(inp, device)
    return inp


def to_device(inp: BlockInputs, device) -> BlockInputs:
    mv = lambda t: None if t is None else t.to(device)
    return BlockInputs(inp.dims, inp.dtype, mv(inp.x), {k: mv(v) for k, v in inp.weights.items()},
                       {k: mv(v) for k, v in inp.gains.items()}, mv(inp.k_cache), mv(inp.v_cache),
                       inp.start_pos)


def to_numpy64(t: torch.Tensor):
    """Exact float64 copy of a (bf16 / fp32) tensor for the oracle."""
    return t.detach().to("cpu", torch.float64).numpy()


# --- the five workloads, by what they are -------------------------------------------------

TINY_FP32 = dict(dims=TINY, dtype=torch.float32, batch=1, prefill_tokens=16, decode_steps=4,
                 weight_std=0.02)
DECODE_8B = dict(dims=LLAMA3_8B, dtype=torch.bfloat16, batches=(1, 8, 32), cache_len=1000,
                 weight_std=0.02)
PREFILL_8B = dict(dims=LLAMA3_8B, dtype=torch.bfloat16, batch=1, tokens=(512, 2048, 8192),
                  weight_std=0.02)
BLOCK_70B = dict(dims=LLAMA31_70B, dtype=torch.bfloat16, decode_batch=16, cache_len=8192,
                 prefill_tokens=4096, weight_std=0.01)
STACK_8B = dict(dims=LLAMA3_8B, dtype=torch.bfloat16, n_layers=32, batch=32, prefill_tokens=1024,
                decode_steps=256, vocab=VOCAB, weight_std=0.02)


def make_token_ids(batch: int, tokens: int, vocab: int = VOCAB, seed: int = 0) -> torch.Tensor:
    """Uniform token ids in [0, vocab), int32."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    return torch.randint(0, vocab, (batch, tokens), generator=gen, dtype=torch.int64).to(torch.int32)
