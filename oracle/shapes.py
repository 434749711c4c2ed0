"""Parameter, d_ff and FLOP accounting for dense Llama-style configs.

Follows [Block] "Inside a Transformer Block: FFN, the Residual Stream, and
Normalization", section 04 (the 2/3 rule) and section 06 (counting parameters
and FLOPs); [QKV] "Llama 3 8B · Prepare Q, K, V", Parameters table; [Next]
"How Llama 3.1 Generates the Next Token", Unembedding (Parameters); [70B]
"Llama 3.1 70B", Token embedding.
"""
from __future__ import annotations

import math


def ffn_hidden_dim(d_model: int, ffn_dim_multiplier: float | None, multiple_of: int) -> int:
    """d_ff from the 2/3 rule ([Block] section 04, "The 2/3 rule"): take 2/3 of 4d,
    truncate to an integer, scale by the optional multiplier (truncating again),
    then round up to a multiple of ``multiple_of``."""
    hidden = int(2 * (4 * d_model) / 3)
    if ffn_dim_multiplier is not None:
        hidden = int(ffn_dim_multiplier * hidden)
    return multiple_of * ((hidden + multiple_of - 1) // multiple_of)


def qkv_params(d_model: int, n_heads: int, n_kv_heads: int) -> int:
    """Q, K and V projection parameters of one block, bias-free ([QKV] Parameters)."""
    head_dim = d_model // n_heads
    return d_model * n_heads * head_dim + 2 * d_model * n_kv_heads * head_dim


def block_params(d_model: int, d_ff: int, n_heads: int, n_kv_heads: int,
                 qkv_bias: bool = False, swiglu: bool = True) -> int:
    """Parameters of one pre-norm block ([Block] section 06): W_Q and W_O are d x d,
    W_K and W_V are d x kv_dim, the FFN has 3 (SwiGLU) or 2 matrices of d x d_ff,
    plus two RMSNorm gains of d.  Optional Q/K/V biases (Qwen2.5)."""
    head_dim = d_model // n_heads
    kv_dim = n_kv_heads * head_dim
    attn = 2 * d_model * d_model + 2 * d_model * kv_dim
    if qkv_bias:
        attn += d_model + 2 * kv_dim
    ffn = (3 if swiglu else 2) * d_model * d_ff
    return attn + ffn + 2 * d_model


def ffn_share(d_model: int, d_ff: int, n_heads: int, n_kv_heads: int, qkv_bias: bool = False) -> float:
    return 3 * d_model * d_ff / block_params(d_model, d_ff, n_heads, n_kv_heads, qkv_bias)


def model_params(d_model: int, d_ff: int, n_layers: int, n_heads: int, n_kv_heads: int,
                 vocab: int, tied: bool = False, qkv_bias: bool = False):
    """(total, non-embedding) parameters: L blocks + final norm + embedding + LM head."""
    block = block_params(d_model, d_ff, n_heads, n_kv_heads, qkv_bias)
    embed = vocab * d_model
    head = 0 if tied else vocab * d_model
    total = n_layers * block + d_model + embed + head
    return total, total - embed - head


def lm_head_params(d_model: int, vocab: int) -> int:
    """[Next] Unembedding: W_out is d x V, bias-free."""
    return d_model * vocab


def embedding_params(d_model: int, vocab: int) -> int:
    """[70B] Token embedding: a V x d lookup table."""
    return vocab * d_model


def kaplan_params(d_model: int, n_layers: int) -> int:
    """Kaplan's 12 * L * d^2 estimate ([Block] section 06, Kaplan's formula)."""
    return 12 * n_layers * d_model * d_model


def kaplan_context_flops(n_layers: int, n_ctx: int, d_attn: int) -> int:
    """Context-dependent forward FLOPs per token, 2 * n_layer * n_ctx * d_attn
    ([Block] section 06, FLOPs: 2N for the forward pass)."""
    return 2 * n_layers * n_ctx * d_attn


# --- exact algorithmic work of the block path (used by the roofline) -----------------------

def block_weight_macs(d_model: int, d_ff: int, n_heads: int, n_kv_heads: int, head_dim: int) -> int:
    """Multiply-accumulates per token over the seven projection matrices."""
    q, kv = n_heads * head_dim, n_kv_heads * head_dim
    return d_model * (q + 2 * kv) + q * d_model + 3 * d_model * d_ff


def attention_pairs_causal(T: int, start: int = 0) -> int:
    """Unmasked (query, key) pairs for T queries at positions start..start+T-1."""
    return sum(start + t + 1 for t in range(T))


def block_flops(d_model, d_ff, n_heads, n_kv_heads, head_dim, batch, T, start=0) -> int:
    """2 FLOPs per weight MAC per token plus 4*Hq*dh per unmasked (q, k) pair
    (QK^T and PV); norm, rotation and softmax work is not counted."""
    macs = block_weight_macs(d_model, d_ff, n_heads, n_kv_heads, head_dim)
    return batch * (2 * macs * T + 4 * n_heads * head_dim * attention_pairs_causal(T, start))


def decode_block_bytes(d_model, d_ff, n_heads, n_kv_heads, head_dim, batch, pos, elem=2) -> int:
    """Bytes one decode step must move at minimum: every weight once, the two gains,
    K and V rows 0..pos read once per KV head, the new K/V row written, x in, y out."""
    weights = block_weight_macs(d_model, d_ff, n_heads, n_kv_heads, head_dim) + 2 * d_model
    kv_read = 2 * batch * n_kv_heads * (pos + 1) * head_dim
    kv_write = 2 * batch * n_kv_heads * head_dim
    act = 2 * batch * d_model
    return elem * (weights + kv_read + kv_write + act)


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def is_close_rel(a: float, b: float, rel: float) -> bool:
    return math.isclose(a, b, rel_tol=rel)
