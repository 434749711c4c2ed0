"""The Llama-3-style pre-norm decoder block, written out plainly on the CPU.

TEST INFRASTRUCTURE ONLY (see the package docstring).  Plain NumPy, float64 by
default; a float32 mode exists only so the benchmark can time the oracle as a
CPU baseline.  For bf16 workloads every intermediate is rounded to bf16 at the
points the pages' PyTorch definitions round it (``rnd = bf16.round_bf16``); the
fp32 workload passes ``rnd = bf16.identity``.

The computation, per sequence b, token t at absolute position p
([70B] "Transformer layer": h = x + Attention(Norm(x)), y = h + FFN(Norm(h))):

  1. xn = R(R(x * r) * g1),  r = (mean(x^2) + eps)^-1/2          RMSNorm
  2. q, k, v = R(xn Wq^T), R(xn Wk^T), R(xn Wv^T)                 projections
  3. q, k rotated pairwise (2i, 2i+1) by p * theta^(-2i/dh), R    RoPE
  4. k, v written to the cache at row p (KV-head size)           KV cache
  5. o_h = R(softmax_j(q_h . k_g(j) / sqrt(dh)) v_g), j <= p,
     g = h // (Hq / Hkv)                                          causal GQA
  6. h = R(x + R(o Wo^T))                                         residual
  7. hn = RMSNorm2(h)
  8. u = R(R(SiLU(R(hn W1^T))) * R(hn W3^T))                      SwiGLU
  9. y = R(h + R(u W2^T))                                         residual

Readings where the pages are silent:
  * bf16 rounding points as above (the unfused PyTorch order of the snippets);
  * a query at absolute position p sees keys 0..p (its own row included);
  * RoPE angles in float64 (the page's listing uses float32 angles);
  * the softmax weights stay unrounded in the oracle.
"""
from __future__ import annotations

import math
from typing import Dict, Optional, Sequence

import numpy as np

from .bf16 import round_bf16, identity


# ---------------------------------------------------------------------------------------------
# RMSNorm
# ---------------------------------------------------------------------------------------------

def rmsnorm(x, g, eps, rnd=round_bf16):
    """RMSNorm over the last axis.

    [70B] "RMSNorm": y = x / sqrt(mean(x^2) + eps) * g, reduction at higher
    precision, the scaled row cast back to the trunk dtype (``type_as``) before
    the gain multiplies it.  [Next] "What's RMSNorm?" gives the same formula with
    eps inside the square root.
    """
    ms = np.mean(x * x, axis=-1, keepdims=True)
    r = 1.0 / np.sqrt(ms + eps)
    return rnd(rnd(x * r) * g)


# ---------------------------------------------------------------------------------------------
# RoPE
# ---------------------------------------------------------------------------------------------

def rope_frequencies(head_dim: int, theta: float) -> np.ndarray:
    """omega_i = theta^(-2i/d_h), i = 0 .. d_h/2 - 1 ([Next] "Why use different
    rotation speeds?").  omega_0 = 1 rad per position."""
    i = np.arange(head_dim // 2, dtype=np.float64)
    return theta ** (-2.0 * i / head_dim)


def rope_frequencies_scaled(head_dim: int, theta: float, factor: float, low_freq_factor: float,
                            high_freq_factor: float, original_context: int) -> np.ndarray:
    """Llama 3.1's long-context adjustment of the base schedule ([Next] "Why use
    different rotation speeds?": the fastest rotations stay as they are, the slowest
    turn ``factor`` times more slowly, a middle range is blended between the two;
    [70B] highlights: "llama3 x8").

    The pages name the three bands but not their edges.  Reading taken: a pair's
    band follows from its wavelength 2 pi / omega_i, measured against the original
    context length: shorter than original_context / high_freq_factor -> unchanged;
    longer than original_context / low_freq_factor -> omega_i / factor; in between,
    omega' = (1 - s) omega_i / factor + s omega_i with
    s = (original_context / wavelength - low_freq_factor) / (high_freq_factor - low_freq_factor),
    which is 1 at the fast edge and 0 at the slow edge (a linear blend in the
    number of turns per original context).  Llama 3.1's released configuration is
    factor 8, low 1, high 4, original context 8192.
    """
    omega = rope_frequencies(head_dim, theta)
    wavelength = 2.0 * math.pi / omega
    fast_edge = original_context / high_freq_factor
    slow_edge = original_context / low_freq_factor
    out = np.empty_like(omega)
    for i, (w, lam) in enumerate(zip(omega, wavelength)):
        if lam < fast_edge:
            out[i] = w
        elif lam > slow_edge:
            out[i] = w / factor
        else:
            s = (original_context / lam - low_freq_factor) / (high_freq_factor - low_freq_factor)
            out[i] = (1.0 - s) * w / factor + s * w
    return out


def rope_angles(positions: Sequence[int], head_dim: int, theta: float, scaling=None) -> np.ndarray:
    """phi[m, i] = m * omega_i ([Next] "What exactly are we rotating?"), float64.
    ``scaling`` = (factor, low_freq_factor, high_freq_factor, original_context)
    selects the long-context schedule of ``rope_frequencies_scaled``."""
    pos = np.asarray(positions, dtype=np.float64)
    omega = rope_frequencies(head_dim, theta) if scaling is None else \
        rope_frequencies_scaled(head_dim, theta, *scaling)
    return np.outer(pos, omega)


def rope_rotate(x: np.ndarray, angles: np.ndarray) -> np.ndarray:
    """Rotate adjacent pairs (x_2i, x_2i+1) of the last axis by angles[..., i].

    [Next] "What exactly are we rotating?": x'_2i = x_2i cos(phi) - x_2i+1 sin(phi),
    x'_2i+1 = x_2i sin(phi) + x_2i+1 cos(phi).  ``angles`` broadcasts against
    x[..., ::2] (for x [H, T, dh] pass [T, dh/2]).
    """
    a = x[..., 0::2]
    b = x[..., 1::2]
    c = np.cos(angles).astype(x.dtype)
    s = np.sin(angles).astype(x.dtype)
    out = np.empty_like(x)
    out[..., 0::2] = a * c - b * s
    out[..., 1::2] = a * s + b * c
    return out


# ---------------------------------------------------------------------------------------------
# attention
# ---------------------------------------------------------------------------------------------

def causal_gqa_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, q_pos: Sequence[int],
                         rnd=round_bf16) -> np.ndarray:
    """Causal grouped-query attention for one sequence.

    q [Hq, Tq, dh] (rotated), k, v [Hkv, Tk, dh] with key j at absolute position j.
    The query at absolute position q_pos[t] sees keys 0..q_pos[t].  Query head h
    reads KV head h // (Hq/Hkv) ([70B] "Grouped-Query Attention": 64 query heads
    in 8 groups share one K/V head each; [Next] Attention notation g(i) = ceil(i/4),
    1-indexed).  Scores are q.k / sqrt(dh) ([Next] "Where does position enter the
    computation?"), the softmax runs over keys ([Next] Attention notation), then
    the weights average the value rows.  Returns merged heads [Tq, Hq*dh].
    """
    hq, tq, dh = q.shape
    hkv, tk, _ = k.shape
    if hq % hkv != 0:
        raise ValueError("query heads must be a multiple of KV heads")
    n_rep = hq // hkv
    qp = np.asarray(q_pos)
    if tk < qp.max() + 1:
        raise ValueError("cache shorter than the latest query position")
    keypos = np.arange(tk)
    masked = keypos[None, :] > qp[:, None]           # [Tq, Tk]
    scale = 1.0 / math.sqrt(dh)
    out = np.empty((tq, hq * dh), dtype=q.dtype)
    for h in range(hq):
        g = h // n_rep
        s = (q[h] @ k[g].T) * scale
        s = np.where(masked, -np.inf, s)
        s = s - s.max(axis=1, keepdims=True)
        p = np.exp(s)
        p = p / p.sum(axis=1, keepdims=True)
        out[:, h * dh:(h + 1) * dh] = rnd(p @ v[g])
    return out


# ---------------------------------------------------------------------------------------------
# SwiGLU
# ---------------------------------------------------------------------------------------------

def silu(z):
    """SiLU(a) = a * sigma(a) = a / (1 + e^-a) ([Next] "What's the SWIGLU block?")."""
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def swiglu_hidden(hn, w_gate, w_up, rnd=round_bf16):
    """u = SiLU(hn W1^T) * (hn W3^T), rounded as the unfused PyTorch expression
    ``F.silu(self.gate(x)) * self.up(x)`` rounds ([70B] "SwiGLU MLP" reference
    implementation; [Next] u = SiLU(a) (.) b)."""
    gate = rnd(hn @ w_gate.T)
    up = rnd(hn @ w_up.T)
    return rnd(rnd(silu(gate)) * up)


# ---------------------------------------------------------------------------------------------
# the block
# ---------------------------------------------------------------------------------------------

def block_forward(x: np.ndarray, w: Dict[str, np.ndarray], g: Dict[str, np.ndarray], dims,
                  k_cache: np.ndarray, v_cache: np.ndarray, start_pos: int,
                  rnd=round_bf16, out_rows: Optional[Sequence[int]] = None, trace: Optional[dict] = None):
    """One decoder block over T new tokens per sequence at positions
    start_pos..start_pos+T-1 (prefill: start_pos = 0; decode: T = 1, start_pos = pos).

    x [B, T, d]; w holds wq, wk, wv, wo, w_gate, w_up, w_down as [out, in]
    (``F.linear`` computes x A^T: [QKV] layers.py excerpt); g holds g_attn, g_ffn.
    k_cache, v_cache [B, Hkv, S_max, dh] hold rows 0..start_pos-1 and are updated
    IN PLACE at rows start_pos..start_pos+T-1 (the cache stores K and V at KV-head
    size, [QKV] Explanation).  ``out_rows`` restricts steps 5-9 to those token
    indices (the cache is still filled for all T).  Returns y [B, len(rows), d].

    ``trace``, if given, receives the values just before their last rounding:
    "y_exact" [B, rows, d], "k_exact" and "v_exact" [B, Hkv, T, dh].  An output
    stored in bf16 cannot be closer to the exact value than half an ulp, so
    parity is measured against these.
    """
    B, T, d = x.shape
    hq, hkv, dh = dims.n_heads, dims.n_kv_heads, dims.head_dim
    rows = np.arange(T) if out_rows is None else np.asarray(out_rows)
    positions = np.arange(start_pos, start_pos + T)
    ang = rope_angles(positions, dh, dims.rope_theta, getattr(dims, "rope_scaling", None))   # [T, dh/2]
    ys = []
    for b in range(B):
        xn = rmsnorm(x[b], g["g_attn"], dims.eps, rnd)
        k = rnd(xn @ w["wk"].T).reshape(T, hkv, dh).transpose(1, 0, 2)
        v_exact = (xn @ w["wv"].T).reshape(T, hkv, dh).transpose(1, 0, 2)
        v = rnd(v_exact)
        k_exact = rope_rotate(k, ang)
        k = rnd(k_exact)
        k_cache[b, :, start_pos:start_pos + T] = k
        v_cache[b, :, start_pos:start_pos + T] = v
        if trace is not None:
            trace.setdefault("k_exact", []).append(k_exact)
            trace.setdefault("v_exact", []).append(v_exact)
        xr = x[b][rows]
        xnr = xn[rows]
        q = rnd(xnr @ w["wq"].T).reshape(len(rows), hq, dh).transpose(1, 0, 2)
        q = rnd(rope_rotate(q, ang[rows]))
        kv_len = start_pos + int(rows.max()) + 1
        o = causal_gqa_attention(q, k_cache[b, :, :kv_len], v_cache[b, :, :kv_len],
                                 positions[rows], rnd)
        h = rnd(xr + rnd(o @ w["wo"].T))
        hn = rmsnorm(h, g["g_ffn"], dims.eps, rnd)
        u = swiglu_hidden(hn, w["w_gate"], w["w_up"], rnd)
        y_exact = h + rnd(u @ w["w_down"].T)
        if trace is not None:
            trace.setdefault("y_exact", []).append(y_exact)
        ys.append(rnd(y_exact))
    if trace is not None:
        for key in ("k_exact", "v_exact", "y_exact"):
            trace[key] = np.stack(trace[key])
    return np.stack(ys)


# ---------------------------------------------------------------------------------------------
# stack head: embedding, final norm, LM head, greedy choice
# ---------------------------------------------------------------------------------------------

def embed(ids: np.ndarray, w_embed: np.ndarray) -> np.ndarray:
    """Row gather from the V x d table, no positional term ([70B] "Token embedding")."""
    return w_embed[np.asarray(ids)]


def lm_head_logits(h_last: np.ndarray, g_final: np.ndarray, w_out: np.ndarray, eps: float,
                   rnd=round_bf16) -> np.ndarray:
    """Final RMSNorm then the bias-free projection to V logits, kept unrounded
    ([Next] "Unembedding": Z = RMSNorm(X) W_out; [70B] "LM head": logits in fp32)."""
    return rmsnorm(h_last, g_final, eps, rnd) @ w_out.T


def greedy(logits: np.ndarray) -> np.ndarray:
    """The most probable token; ties go to the lowest index ([Next] "Top-k and top-p
    sampling": choosing the highest-probability token)."""
    return np.argmax(logits, axis=-1)


def stack_forward(x: np.ndarray, layers, g_final, w_out, dims, caches, start_pos, rnd=round_bf16):
    """L blocks then the head on the last token of each sequence.  ``layers`` is a list
    of (w, g) pairs, ``caches`` a list of (k_cache, v_cache) updated in place.
    Returns (logits [B, V], ids [B])."""
    h = x
    for (w, g), (kc, vc) in zip(layers, caches):
        h = block_forward(h, w, g, dims, kc, vc, start_pos, rnd)
    logits = lm_head_logits(h[:, -1, :], g_final, w_out, dims.eps, rnd)
    return logits, greedy(logits)


__all__ = [
    "rmsnorm", "rope_frequencies", "rope_frequencies_scaled", "rope_angles", "rope_rotate", "causal_gqa_attention",
    "silu", "swiglu_hidden", "block_forward", "embed", "lm_head_logits", "greedy",
    "stack_forward", "round_bf16", "identity",
]
