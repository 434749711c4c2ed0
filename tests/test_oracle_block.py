"""Pins of the oracle's block arithmetic: worked examples the pages print, closed forms,
invariants, special cases that reduce to a library routine (torch CPU), and a scalar
brute-force block on tiny inputs written independently of the vectorised oracle."""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import block as ob
from oracle.bf16 import round_bf16, identity
from workloads import BlockDims

ID = identity


# ------------------------------------------------------------------ RMSNorm

def test_rmsnorm_worked_example(printed):
    ex = printed["rmsnorm_example"]
    for xs, rms in zip(ex["inputs"], ex["rms"]):
        x = np.array(xs, dtype=np.float64)
        assert round(math.sqrt(np.mean(x * x)), 2 if rms < 10 else 1) == rms
        y = ob.rmsnorm(x, np.ones(3), 0.0, ID)
        assert np.allclose(np.round(y, ex["printed_decimals"]), ex["normalized"])


def test_rmsnorm_unit_rms_before_gain_and_gain_per_feature():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((7, 64)) * 3.0
    y = ob.rmsnorm(x, np.ones(64), 1e-5, ID)
    ms = np.mean(x * x, axis=-1)
    assert np.allclose(np.mean(y * y, axis=-1), ms / (ms + 1e-5), rtol=1e-12)
    g = rng.uniform(0.5, 1.5, 64)
    assert np.allclose(ob.rmsnorm(x, g, 1e-5, ID), y * g, rtol=1e-13)
    # scale invariance with eps = 0
    assert np.allclose(ob.rmsnorm(10 * x, g, 0.0, ID), ob.rmsnorm(x, g, 0.0, ID), rtol=1e-13)


def test_rmsnorm_matches_torch_rms_norm():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((5, 96))
    g = rng.uniform(0.5, 1.5, 96)
    want = F.rms_norm(torch.from_numpy(x), (96,), torch.from_numpy(g), eps=1e-5).numpy()
    assert np.allclose(ob.rmsnorm(x, g, 1e-5, ID), want, rtol=1e-13, atol=1e-14)


def test_rmsnorm_bf16_rounding_points():
    # the page's definition evaluated by torch in bf16: (x.float()*r).type_as(x) * g
    gen = torch.Generator().manual_seed(3)
    x = torch.randn(16, 256, generator=gen).to(torch.bfloat16)
    g = (torch.rand(256, generator=gen) + 0.5).to(torch.bfloat16)
    r = x.float().pow(2).mean(-1, keepdim=True).add(1e-5).rsqrt()
    want = ((x.float() * r).to(torch.bfloat16) * g).double().numpy()
    got = ob.rmsnorm(x.double().numpy(), g.double().numpy(), 1e-5, round_bf16)
    # torch reduces in fp32, the oracle in fp64: allow a 1-ulp flip on rare ties
    ulp = np.abs(want) * 2.0 ** -7
    assert np.all(np.abs(got - want) <= ulp + 1e-30)
    assert np.mean(got == want) > 0.99


# ------------------------------------------------------------------ RoPE

def test_rope_frequencies(printed):
    ex = printed["rope_rotation_examples"]
    w = ob.rope_frequencies(ex["head_dim"], ex["theta"])
    assert w.shape == (ex["pairs"],)
    assert w[0] == ex["omega_0_rad_per_position"]
    assert np.all(np.diff(w) < 0)                      # later pairs turn more slowly
    assert math.isclose(w[-1], 500000.0 ** (-126 / 128), rel_tol=1e-14)


def test_rope_worked_examples(printed):
    ex = printed["rope_rotation_examples"]
    q = ob.rope_rotate(np.array([1.0, 0.0]), np.array([math.radians(ex["quarter_turn"]["degrees"])]))
    assert np.allclose(q, ex["quarter_turn"]["output"], atol=1e-15)
    rel = ex["relative"]
    step = math.radians(rel["degrees_per_position"])
    pair = np.array(rel["pair"], dtype=np.float64)
    for c in rel["cases"]:
        qr = ob.rope_rotate(pair, np.array([c["q_pos"] * step]))
        kr = ob.rope_rotate(pair, np.array([c["k_pos"] * step]))
        assert abs(float(qr @ kr) - c["dot"]) < 1e-12
    # moving only the key changes the score (8 vs 2: 180 degrees apart)
    qr = ob.rope_rotate(pair, np.array([8 * step]))
    kr = ob.rope_rotate(pair, np.array([2 * step]))
    assert abs(float(qr @ kr) + 1.0) < 1e-12


def test_rope_invariants():
    rng = np.random.default_rng(4)
    dh, theta = 128, 500000.0
    q = rng.standard_normal(dh)
    k = rng.standard_normal(dh)
    ang = lambda p: ob.rope_angles([p], dh, theta)[0]
    # identity at position 0
    assert np.array_equal(ob.rope_rotate(q, ang(0)), q)
    # each pair keeps its length
    r = ob.rope_rotate(q, ang(777))
    assert np.allclose(r[0::2] ** 2 + r[1::2] ** 2, q[0::2] ** 2 + q[1::2] ** 2, rtol=1e-12)
    # the score depends only on n - m
    s1 = ob.rope_rotate(q, ang(5)) @ ob.rope_rotate(k, ang(2))
    s2 = ob.rope_rotate(q, ang(1005)) @ ob.rope_rotate(k, ang(1002))
    assert math.isclose(s1, s2, rel_tol=1e-9, abs_tol=1e-9)
    # adjacent pairs, not halves: rotating pair 0 touches elements 0 and 1 only
    e0 = np.zeros(dh); e0[0] = 1.0
    out = ob.rope_rotate(e0, np.concatenate([[math.pi / 2], np.zeros(dh // 2 - 1)]))
    assert np.allclose(out[:2], [0, 1], atol=1e-15) and np.all(out[2:] == 0)


def test_rope_matches_complex_multiplication():
    # library pin: view pairs as complex numbers and multiply by e^{i phi}
    rng = np.random.default_rng(5)
    x = rng.standard_normal((3, 9, 64))
    ang = ob.rope_angles(np.arange(100, 109), 64, 500000.0)
    xc = torch.view_as_complex(torch.from_numpy(x).reshape(3, 9, 32, 2).contiguous())
    rot = torch.polar(torch.ones(9, 32, dtype=torch.float64), torch.from_numpy(ang))
    want = torch.view_as_real(xc * rot).reshape(3, 9, 64).numpy()
    assert np.allclose(ob.rope_rotate(x, ang), want, rtol=1e-13, atol=1e-14)


# ------------------------------------------------------------------ attention

def _scalar_attention(q, k, v, q_pos):
    """Brute force with Python floats, one (head, query) at a time."""
    hq, tq, dh = q.shape
    hkv = k.shape[0]
    out = np.zeros((tq, hq * dh))
    for h in range(hq):
        g = (h * hkv) // hq
        for t in range(tq):
            scores = []
            for j in range(q_pos[t] + 1):
                scores.append(sum(q[h, t, c] * k[g, j, c] for c in range(dh)) / math.sqrt(dh))
            mx = max(scores)
            wts = [math.exp(s - mx) for s in scores]
            tot = sum(wts)
            for c in range(dh):
                out[t, h * dh + c] = sum(wts[j] * v[g, j, c] for j in range(len(wts))) / tot
    return out


def test_attention_brute_force_tiny():
    rng = np.random.default_rng(6)
    q = rng.standard_normal((4, 3, 8))
    k = rng.standard_normal((2, 7, 8))
    v = rng.standard_normal((2, 7, 8))
    pos = [4, 5, 6]
    got = ob.causal_gqa_attention(q, k, v, pos, ID)
    assert np.allclose(got, _scalar_attention(q, k, v, pos), rtol=1e-12, atol=1e-13)


def test_attention_position_zero_returns_v0_and_uniform_keys_average():
    rng = np.random.default_rng(7)
    q = rng.standard_normal((2, 1, 16))
    k = rng.standard_normal((1, 5, 16))
    v = rng.standard_normal((1, 5, 16))
    o = ob.causal_gqa_attention(q, k, v, [0], ID)
    assert np.allclose(o.reshape(2, 16), v[0, 0][None, :].repeat(2, 0), rtol=1e-14)
    k_same = np.repeat(k[:, :1], 5, axis=1)
    o = ob.causal_gqa_attention(q, k_same, v, [3], ID)
    assert np.allclose(o.reshape(2, 16), v[0, :4].mean(0)[None, :].repeat(2, 0), rtol=1e-12)


def test_gqa_equals_mha_with_repeated_kv():
    rng = np.random.default_rng(8)
    hq, hkv, T, dh = 8, 2, 6, 16
    q = rng.standard_normal((hq, T, dh))
    k = rng.standard_normal((hkv, T, dh))
    v = rng.standard_normal((hkv, T, dh))
    pos = list(range(T))
    grouped = ob.causal_gqa_attention(q, k, v, pos, ID)
    rep = hq // hkv
    mha = ob.causal_gqa_attention(q, np.repeat(k, rep, axis=0), np.repeat(v, rep, axis=0), pos, ID)
    assert np.allclose(grouped, mha, rtol=1e-13)
    # a wrong grouping (h % Hkv) must disagree: the pin has teeth
    interleaved = ob.causal_gqa_attention(q, np.tile(k, (rep, 1, 1)), np.tile(v, (rep, 1, 1)), pos, ID)
    assert not np.allclose(grouped, interleaved)


@pytest.mark.parametrize("hkv", [1, 2, 8])
def test_attention_matches_torch_sdpa(hkv):
    # library pin: causal SDPA (top-left aligned, queries and keys both from 0),
    # MQA (1), GQA (2) and MHA (8) groupings
    rng = np.random.default_rng(9)
    hq, T, dh = 8, 11, 32
    q = rng.standard_normal((hq, T, dh))
    k = rng.standard_normal((hkv, T, dh))
    v = rng.standard_normal((hkv, T, dh))
    rep = hq // hkv
    kt = torch.from_numpy(np.repeat(k, rep, axis=0))[None]
    vt = torch.from_numpy(np.repeat(v, rep, axis=0))[None]
    want = F.scaled_dot_product_attention(torch.from_numpy(q)[None], kt, vt, is_causal=True)[0]
    want = want.permute(1, 0, 2).reshape(T, hq * dh).numpy()
    got = ob.causal_gqa_attention(q, k, v, list(range(T)), ID)
    assert np.allclose(got, want, rtol=1e-12, atol=1e-13)


# ------------------------------------------------------------------ SwiGLU

def test_silu_closed_forms_and_torch():
    assert ob.silu(np.array(0.0)) == 0.0
    assert math.isclose(float(ob.silu(np.array(1.0))), 1.0 / (1.0 + math.exp(-1.0)), rel_tol=1e-15)
    assert math.isclose(float(ob.silu(np.array(40.0))), 40.0, rel_tol=1e-15)
    assert abs(float(ob.silu(np.array(-800.0)))) == 0.0
    z = np.linspace(-20, 20, 4001)
    assert np.allclose(ob.silu(z), F.silu(torch.from_numpy(z)).numpy(), rtol=1e-14, atol=1e-300)


def test_swiglu_gate_example(printed):
    ex = printed["swiglu_gate_example"]
    # choose branch values whose SiLU is exactly ex["a"]: identity weights and a
    # hidden vector already equal to the pre-activation solving SiLU(z) = a
    a = np.array(ex["a"], dtype=np.float64)
    z = np.array([_silu_inverse(t) for t in a])
    hn = np.concatenate([z, np.array(ex["b"], dtype=np.float64)])[None, :]
    w_gate = np.hstack([np.eye(3), np.zeros((3, 3))])
    w_up = np.hstack([np.zeros((3, 3)), np.eye(3)])
    u = ob.swiglu_hidden(hn, w_gate, w_up, ID)[0]
    assert np.allclose(u, ex["product"], rtol=1e-12, atol=1e-15)


def _silu_inverse(a):
    if a == 0:
        return 0.0
    lo, hi = 0.0, 50.0
    for _ in range(200):
        mid = 0.5 * (lo + hi)
        if mid / (1 + math.exp(-mid)) < a:
            lo = mid
        else:
            hi = mid
    return 0.5 * (lo + hi)


# ------------------------------------------------------------------ the block

def _scalar_block(x, w, g, dims, start):
    """Independent scalar block: Python loops and math.* only, no rounding, one token
    at a time (decode-style) so the KV cache grows step by step."""
    d, hq, hkv, dh, F_ = dims.d_model, dims.n_heads, dims.n_kv_heads, dims.head_dim, dims.d_ff
    T = len(x)
    ks, vs = [], []
    outs = []

    def lin(W, vec):
        return [sum(W[o][i] * vec[i] for i in range(len(vec))) for o in range(len(W))]

    def norm(vec, gain):
        r = 1.0 / math.sqrt(sum(t * t for t in vec) / len(vec) + dims.eps)
        return [vec[i] * r * gain[i] for i in range(len(vec))]

    def rot(vec, p):
        out = list(vec)
        for hbase in range(0, len(vec), dh):
            for i in range(dh // 2):
                ang = p * dims.rope_theta ** (-2.0 * i / dh)
                a, b = vec[hbase + 2 * i], vec[hbase + 2 * i + 1]
                out[hbase + 2 * i] = a * math.cos(ang) - b * math.sin(ang)
                out[hbase + 2 * i + 1] = a * math.sin(ang) + b * math.cos(ang)
        return out

    for t in range(T):
        p = start + t
        xt = list(x[t])
        xn = norm(xt, g["g_attn"])
        q = rot(lin(w["wq"], xn), p)
        ks.append(rot(lin(w["wk"], xn), p))
        vs.append(lin(w["wv"], xn))
        o = []
        for h in range(hq):
            kvh = h // (hq // hkv)
            sc = [sum(q[h * dh + c] * ks[j][kvh * dh + c] for c in range(dh)) / math.sqrt(dh)
                  for j in range(len(ks))]
            m = max(sc)
            e = [math.exp(s - m) for s in sc]
            z = sum(e)
            o += [sum(e[j] * vs[j][kvh * dh + c] for j in range(len(e))) / z for c in range(dh)]
        attn = lin(w["wo"], o)
        hres = [xt[i] + attn[i] for i in range(d)]
        hn = norm(hres, g["g_ffn"])
        a = lin(w["w_gate"], hn)
        b = lin(w["w_up"], hn)
        u = [a[i] / (1 + math.exp(-a[i])) * b[i] for i in range(F_)]
        dn = lin(w["w_down"], u)
        outs.append([hres[i] + dn[i] for i in range(d)])
    return np.array(outs)


def _tiny_inputs(dims, T, seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((1, T, dims.d_model))
    shapes = dims.weight_shapes()
    w = {n: rng.standard_normal(s) * 0.3 for n, s in shapes.items()}
    g = {"g_attn": rng.uniform(0.5, 1.5, dims.d_model), "g_ffn": rng.uniform(0.5, 1.5, dims.d_model)}
    return x, w, g


def test_block_matches_scalar_brute_force():
    dims = BlockDims(d_model=8, n_heads=4, n_kv_heads=2, head_dim=2, d_ff=12, rope_theta=100.0)
    T = 5
    x, w, g = _tiny_inputs(dims, T, 10)
    kc = np.zeros((1, 2, T, 2))
    vc = np.zeros((1, 2, T, 2))
    y = ob.block_forward(x, w, g, dims, kc, vc, 0, ID)[0]
    assert np.allclose(y, _scalar_block(x[0], w, g, dims, 0), rtol=1e-11, atol=1e-12)


def test_block_prefill_then_decode_equals_longer_prefill():
    dims = BlockDims(d_model=16, n_heads=4, n_kv_heads=1, head_dim=4, d_ff=24)
    T = 7
    x, w, g = _tiny_inputs(dims, T, 11)
    kc = np.zeros((1, 1, T, 4)); vc = np.zeros((1, 1, T, 4))
    full = ob.block_forward(x, w, g, dims, kc, vc, 0, ID)
    kc2 = np.zeros_like(kc); vc2 = np.zeros_like(vc)
    part = ob.block_forward(x[:, :4], w, g, dims, kc2, vc2, 0, ID)
    steps = [ob.block_forward(x[:, t:t + 1], w, g, dims, kc2, vc2, t, ID) for t in range(4, T)]
    got = np.concatenate([part] + steps, axis=1)
    assert np.allclose(got, full, rtol=1e-12, atol=1e-13)
    assert np.allclose(kc2, kc) and np.allclose(vc2, vc)
    # sampled rows agree with the full computation
    kc3 = np.zeros_like(kc); vc3 = np.zeros_like(vc)
    rows = ob.block_forward(x, w, g, dims, kc3, vc3, 0, ID, out_rows=[0, 3, 6])
    assert np.allclose(rows[0], full[0, [0, 3, 6]], rtol=1e-12)


def test_block_zero_branches_give_identity():
    # Wo = 0 and W_down = 0: both residual adds return the stream unchanged, bit for bit
    dims = BlockDims(d_model=32, n_heads=2, n_kv_heads=1, head_dim=16, d_ff=48)
    x, w, g = _tiny_inputs(dims, 3, 12)
    x = round_bf16(x)
    w = {k: round_bf16(v) for k, v in w.items()}
    w["wo"] = np.zeros_like(w["wo"])
    w["w_down"] = np.zeros_like(w["w_down"])
    kc = np.zeros((1, 1, 3, 16)); vc = np.zeros((1, 1, 3, 16))
    y = ob.block_forward(x, w, g, dims, kc, vc, 0, round_bf16)
    assert np.array_equal(y, x)


def test_block_cache_rows_written_are_rotated_keys_and_raw_values():
    dims = BlockDims(d_model=16, n_heads=2, n_kv_heads=2, head_dim=8, d_ff=16)
    x, w, g = _tiny_inputs(dims, 3, 13)
    kc = np.full((1, 2, 6, 8), np.nan); vc = np.full((1, 2, 6, 8), np.nan)
    kc[:, :, :2] = 0.5; vc[:, :, :2] = -0.25
    y = ob.block_forward(x[:, :1], w, g, dims, kc, vc, 2, ID)
    assert np.all(np.isfinite(y)) and np.all(np.isnan(kc[:, :, 3:]))
    xn = ob.rmsnorm(x[0, 0], g["g_attn"], dims.eps, ID)
    vrow = (w["wv"] @ xn).reshape(2, 8)
    assert np.allclose(vc[0, :, 2], vrow)
    krow = ob.rope_rotate((w["wk"] @ xn).reshape(2, 8), ob.rope_angles([2], 8, dims.rope_theta)[0])
    assert np.allclose(kc[0, :, 2], krow)


def test_stack_head_greedy_ties_lowest_index():
    logits = np.array([[0.5, 2.0, 2.0, -1.0], [3.0, 3.0, 3.0, 3.0]])
    assert list(ob.greedy(logits)) == [1, 0]
    w_e = np.arange(12, dtype=np.float64).reshape(4, 3)
    assert np.array_equal(ob.embed(np.array([[2, 0]]), w_e), w_e[[2, 0]][None])
