"""The oracle's bf16 rounding points, pinned against the pages' own module
definitions evaluated by PyTorch on the CPU in bf16.

The pages define the block as PyTorch modules: "Llama 3.1 70B" gives the
DecoderLayer (x + attn(norm1(x)), then x + ffn(norm2(x))), RMSNorm (fp32 scale,
``type_as`` back to the trunk dtype, then the gain), the GQA module (q/k/v
linears, split heads, ``repeat_kv``, scaled dot-product attention with a causal
mask, merged heads, the o linear) and the SwiGLU module (down(silu(gate(x)) *
up(x))); "Llama 3 8B · Prepare Q, K, V" gives ``precompute_freqs_cis`` (fp32
frequencies and angles, unit complex numbers) and the rotation of q and k as
complex pairs.  The code below restates those definitions with torch operators,
so that torch -- not the oracle -- decides where a bf16 value is rounded: every
module output that is a bf16 tensor is rounded once, by torch.

One reading is taken here: torch's CPU kernel for bf16 scaled dot-product
attention rounds its internal scores and weights to bf16 (measured: about a
quarter of its outputs differ from the exact result rounded once), which is a
property of that kernel, not of the operation the page writes down.  The
attention is therefore evaluated in fp32 from the bf16 q, k, v and its output
rounded once to the trunk dtype (the same reading the oracle takes: softmax
weights unrounded, output rounded).

The comparison: the oracle in bf16 mode against this evaluation, on tiny
shapes (B = 2, T <= 12, d = 64, groups of 1, 2 and 4 query heads per KV head).
torch accumulates in fp32 and the oracle in fp64, so a value that lands within
an fp32 rounding error of a bf16 rounding boundary may round the other way;
such flips are rare at these sizes.  Asserted: at least 99% of the elements of
y and of the written cache rows agree bit for bit and every other element is
within one bf16 ulp.  ``test_each_rounding_point_is_seen`` then removes one
rounding call of the oracle at a time (a mutant built from the oracle's source
on the CPU) and checks that this comparison fails for every one of them.
"""
from __future__ import annotations

import ast
import inspect
import math
import types

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import block as ob
from oracle.bf16 import round_bf16
from workloads import BlockDims

BF = torch.bfloat16


# --------------------------------------------------------------------------------- the pages' modules

def rmsnorm_t(x: torch.Tensor, g: torch.Tensor, eps: float) -> torch.Tensor:
    """"Llama 3.1 70B", RMSNorm reference implementation."""
    rms = x.float().pow(2).mean(-1, keepdim=True).add(eps).rsqrt()
    return (x.float() * rms).type_as(x) * g


def freqs_cis_t(dim: int, end: int, theta: float) -> torch.Tensor:
    """"Llama 3 8B · Prepare Q, K, V", model.py excerpt: precompute_freqs_cis."""
    freqs = 1.0 / (theta ** (torch.arange(0, dim, 2)[: (dim // 2)].float() / dim))
    t = torch.arange(end, dtype=torch.float32)
    angles = torch.outer(t, freqs)
    return torch.polar(torch.ones_like(angles), angles)          # complex64 [end, dim/2]


def rotate_t(x: torch.Tensor, fc: torch.Tensor) -> torch.Tensor:
    """Adjacent pairs as complex numbers times e^{i phi}, back to the input dtype.
    x [B, T, H, dh], fc [T, dh/2]."""
    xc = torch.view_as_complex(x.float().reshape(*x.shape[:-1], -1, 2))
    out = torch.view_as_real(xc * fc[None, :, None, :]).flatten(-2)
    return out.type_as(x)


def repeat_kv_t(k: torch.Tensor, n_rep: int) -> torch.Tensor:
    """[B, Hkv, T, dh] -> [B, Hkv * n_rep, T, dh], each KV head repeated over its group."""
    b, hkv, t, dh = k.shape
    return k[:, :, None].expand(b, hkv, n_rep, t, dh).reshape(b, hkv * n_rep, t, dh)


def gqa_t(xn, w, dims: BlockDims, fc, k_cache, v_cache, start_pos):
    """"Llama 3.1 70B", GQA module, with the K/V cache of "Llama 3 8B · Prepare Q,
    K, V" (keys and values stored at KV-head size, repeated after the read)."""
    B, T, _ = xn.shape
    hq, hkv, dh = dims.n_heads, dims.n_kv_heads, dims.head_dim
    q = F.linear(xn, w["wq"]).view(B, T, hq, dh)
    k = F.linear(xn, w["wk"]).view(B, T, hkv, dh)
    v = F.linear(xn, w["wv"]).view(B, T, hkv, dh)
    q = rotate_t(q, fc[start_pos:start_pos + T])
    k = rotate_t(k, fc[start_pos:start_pos + T])
    k_cache[:, :, start_pos:start_pos + T] = k.transpose(1, 2)
    v_cache[:, :, start_pos:start_pos + T] = v.transpose(1, 2)
    L = start_pos + T
    keys = repeat_kv_t(k_cache[:, :, :L], hq // hkv)
    vals = repeat_kv_t(v_cache[:, :, :L], hq // hkv)
    # query t sits at absolute position start_pos + t and sees keys 0 .. start_pos + t
    mask = torch.arange(L)[None, :] <= (start_pos + torch.arange(T))[:, None]
    o = F.scaled_dot_product_attention(q.transpose(1, 2).float(), keys.float(), vals.float(), attn_mask=mask)
    o = o.type_as(xn).transpose(1, 2).reshape(B, T, hq * dh)
    return F.linear(o, w["wo"])


def swiglu_t(hn, w):
    """"Llama 3.1 70B", SwiGLU MLP: down(silu(gate(x)) * up(x))."""
    return F.linear(F.silu(F.linear(hn, w["w_gate"])) * F.linear(hn, w["w_up"]), w["w_down"])


def decoder_layer_t(x, w, g, dims, fc, k_cache, v_cache, start_pos):
    """"Llama 3.1 70B", DecoderLayer: pre-norm, residual adds in the trunk dtype."""
    h = x + gqa_t(rmsnorm_t(x, g["g_attn"], dims.eps), w, dims, fc, k_cache, v_cache, start_pos)
    return h + swiglu_t(rmsnorm_t(h, g["g_ffn"], dims.eps), w)


# --------------------------------------------------------------------------------- inputs

def _inputs(dims: BlockDims, B: int, T: int, seed: int):
    """bf16 weights N(0, 1/sqrt(fan_in)) so that every branch is O(1) next to the
    trunk (each rounding point then moves the result), gains U(0.5, 1.5), x N(0, 1)."""
    gen = torch.Generator().manual_seed(seed)
    shapes = {"wq": (dims.q_dim, dims.d_model), "wk": (dims.kv_dim, dims.d_model),
              "wv": (dims.kv_dim, dims.d_model), "wo": (dims.d_model, dims.q_dim),
              "w_gate": (dims.d_ff, dims.d_model), "w_up": (dims.d_ff, dims.d_model),
              "w_down": (dims.d_model, dims.d_ff)}
    w = {n: (torch.randn(*s, generator=gen) / math.sqrt(s[1])).to(BF) for n, s in shapes.items()}
    g = {n: (torch.rand(dims.d_model, generator=gen) + 0.5).to(BF) for n in ("g_attn", "g_ffn")}
    x = torch.randn(B, T, dims.d_model, generator=gen).to(BF)
    return x, w, g


def _to64(t):
    return t.to(torch.float64).numpy()


def _ulp(v):
    a = np.maximum(np.abs(v), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(a)) - 7)


def agreement(got: np.ndarray, want: np.ndarray):
    """(fraction bit-equal, largest difference in ulps of the reference)."""
    eq = float(np.mean(got == want))
    ulps = float(np.max(np.abs(got - want) / _ulp(want)))
    return eq, ulps


CASES = [
    # (dims, B, prefill T, decode steps)
    (BlockDims(64, 4, 4, 16, 128, rope_theta=500000.0), 2, 12, 0),   # one query head per KV head
    (BlockDims(64, 4, 2, 16, 128, rope_theta=500000.0), 2, 9, 3),    # groups of 2, then decode
    (BlockDims(64, 4, 1, 16, 96, rope_theta=10000.0), 2, 12, 0),     # groups of 4 (one KV head)
]


def run_both(dims, B, T, steps, seed, block_forward):
    """Prefill T tokens then `steps` single-token steps on both sides; returns
    (torch y, oracle y, torch caches, oracle caches) as float64 arrays."""
    n = T + steps
    x, w, g = _inputs(dims, B, n, seed)
    fc = freqs_cis_t(dims.head_dim, n, dims.rope_theta)
    kc_t = torch.zeros(B, dims.n_kv_heads, n, dims.head_dim, dtype=BF)
    vc_t = torch.zeros_like(kc_t)
    ys_t = [decoder_layer_t(x[:, :T], w, g, dims, fc, kc_t, vc_t, 0)]
    for s in range(steps):
        ys_t.append(decoder_layer_t(x[:, T + s:T + s + 1], w, g, dims, fc, kc_t, vc_t, T + s))
    w64 = {k: _to64(v) for k, v in w.items()}
    g64 = {k: _to64(v) for k, v in g.items()}
    kc_o = np.zeros((B, dims.n_kv_heads, n, dims.head_dim))
    vc_o = np.zeros_like(kc_o)
    x64 = _to64(x)
    ys_o = [block_forward(x64[:, :T], w64, g64, dims, kc_o, vc_o, 0, round_bf16)]
    for s in range(steps):
        ys_o.append(block_forward(x64[:, T + s:T + s + 1], w64, g64, dims, kc_o, vc_o, T + s, round_bf16))
    y_t = np.concatenate([_to64(y) for y in ys_t], axis=1)
    y_o = np.concatenate(ys_o, axis=1)
    return y_t, y_o, (_to64(kc_t), _to64(vc_t)), (kc_o, vc_o)


def passes(y_t, y_o, caches_t, caches_o):
    for got, want in ((y_o, y_t), (caches_o[0], caches_t[0]), (caches_o[1], caches_t[1])):
        eq, ulps = agreement(got, want)
        if eq < 0.99 or ulps > 1.0:
            return False
    return True


@pytest.mark.parametrize("case", range(len(CASES)))
def test_oracle_bf16_block_matches_pages_modules_in_torch(case):
    dims, B, T, steps = CASES[case]
    for seed in (0, 1):
        y_t, y_o, c_t, c_o = run_both(dims, B, T, steps, seed, ob.block_forward)
        for name, got, want in (("y", y_o, y_t), ("k cache", c_o[0], c_t[0]), ("v cache", c_o[1], c_t[1])):
            eq, ulps = agreement(got, want)
            assert eq >= 0.99, f"{name}: only {100 * eq:.2f}% bit-equal"
            assert ulps <= 1.0, f"{name}: {ulps:.2f} ulps apart"


# --------------------------------------------------------------------------------- mutants

class _DropRound(ast.NodeTransformer):
    """Replace the index-th call rnd(e) (in source order) by e."""

    def __init__(self, index: int):
        self.index = index
        self.seen = 0

    def visit_Call(self, node):
        self.generic_visit(node)
        if isinstance(node.func, ast.Name) and node.func.id == "rnd" and len(node.args) == 1:
            i = self.seen
            self.seen += 1
            if i == self.index:
                return node.args[0]
        return node


def _rounding_sites():
    tree = ast.parse(inspect.getsource(ob))
    counter = _DropRound(-1)
    counter.visit(tree)
    return counter.seen


def _mutant(index: int):
    tree = ast.parse(inspect.getsource(ob))
    tree = ast.fix_missing_locations(_DropRound(index).visit(tree))
    mod = types.ModuleType(f"oracle_block_mutant_{index}")
    mod.__dict__["__package__"] = "oracle"
    exec(compile(tree, f"<oracle.block without rounding call {index}>", "exec"), mod.__dict__)
    return mod


def test_each_rounding_point_is_seen():
    """Removing any single rnd(...) of the oracle's block (RMSNorm's two roundings,
    the projections, the rotations, the attention output, both residual adds, the
    four SwiGLU roundings, the final output) makes the cross-check fail."""
    n = _rounding_sites()
    assert n >= 16, f"expected at least 16 rounding calls in oracle.block, found {n}"
    dims, B, T, steps = CASES[1]
    for i in range(n):
        m = _mutant(i)
        y_t, y_o, c_t, c_o = run_both(dims, B, T, steps, 0, m.block_forward)
        assert not passes(y_t, y_o, c_t, c_o), f"rounding call {i} of oracle.block can be removed unnoticed"


# --------------------------------------------------------------------------------- the stack head

def test_lm_head_logits_match_pages_head():
    """Final RMSNorm in the trunk dtype, then the bias-free projection h @ W^T with
    fp32 (here fp64) logits ("How Llama 3.1 Generates the Next Token", Unembedding;
    "Llama 3.1 70B", LM head; softmax over the logits is taken in fp32)."""
    gen = torch.Generator().manual_seed(5)
    d, V = 64, 300
    h = torch.randn(3, d, generator=gen).to(BF)
    g = (torch.rand(d, generator=gen) + 0.5).to(BF)
    w = (torch.randn(V, d, generator=gen) / 8).to(BF)
    want = (rmsnorm_t(h, g, 1e-5).double() @ w.double().T).numpy()
    got = ob.lm_head_logits(_to64(h), _to64(g), _to64(w), 1e-5, round_bf16)
    # the normalised rows agree bit for bit except on rare fp32/fp64 rounding flips
    hn_t = _to64(rmsnorm_t(h, g, 1e-5))
    hn_o = ob.rmsnorm(_to64(h), _to64(g), 1e-5, round_bf16)
    eq, ulps = agreement(hn_o, hn_t)
    assert eq >= 0.99 and ulps <= 1.0
    rows_equal = np.all(hn_o == hn_t, axis=-1)
    assert rows_equal.any()
    assert np.allclose(got[rows_equal], want[rows_equal], rtol=1e-12, atol=1e-12)
    # without the trunk-dtype rounding of the norm the logits move well beyond fp64 noise
    unrounded = ob.rmsnorm(_to64(h), _to64(g), 1e-5, lambda a: a) @ _to64(w).T
    assert np.max(np.abs(unrounded - want)) > 1e-6


def test_stack_forward_matches_pages_modules():
    """Two layers then the head on the last token, greedy choice."""
    dims = BlockDims(64, 4, 2, 16, 128)
    B, T, V = 2, 7, 200
    layers_t, layers_o = [], []
    for i in range(2):
        _, w, g = _inputs(dims, 1, 1, 10 + i)
        layers_t.append((w, g))
        layers_o.append(({k: _to64(v) for k, v in w.items()}, {k: _to64(v) for k, v in g.items()}))
    gen = torch.Generator().manual_seed(20)
    x = torch.randn(B, T, dims.d_model, generator=gen).to(BF)
    g_f = (torch.rand(dims.d_model, generator=gen) + 0.5).to(BF)
    w_out = (torch.randn(V, dims.d_model, generator=gen) / 8).to(BF)
    fc = freqs_cis_t(dims.head_dim, T, dims.rope_theta)
    h = x
    for w, g in layers_t:
        kc = torch.zeros(B, dims.n_kv_heads, T, dims.head_dim, dtype=BF)
        h = decoder_layer_t(h, w, g, dims, fc, kc, torch.zeros_like(kc), 0)
    want = (rmsnorm_t(h[:, -1], g_f, dims.eps).double() @ w_out.double().T).numpy()
    caches = [(np.zeros((B, dims.n_kv_heads, T, dims.head_dim)), np.zeros((B, dims.n_kv_heads, T, dims.head_dim)))
              for _ in layers_o]
    logits, ids = ob.stack_forward(_to64(x), layers_o, _to64(g_f), _to64(w_out), dims, caches, 0, round_bf16)
    rel = np.max(np.abs(logits - want)) / np.sqrt(np.mean(want ** 2))
    assert rel < 2e-2
    margin = np.sort(want, axis=-1)
    clear = (margin[:, -1] - margin[:, -2]) > 4 * np.max(np.abs(logits - want))
    assert np.array_equal(ids[clear], np.argmax(want, axis=-1)[clear])
