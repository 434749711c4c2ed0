"""GPU parity of the decoder block against the CPU oracle, element by element, at
sizes the oracle finishes in seconds (several tiles, ragged tails), plus the
decode/prefill bit-identity contract, error paths and graph replay."""
import numpy as np
import pytest
import torch

import workloads
from oracle import block as ob
from oracle.bf16 import round_bf16
from tests.blockrun import (BF16_TOL, F32_TOL, check_bf16_output, gpu_block, oracle_weights, rel_err, rnd_for,
                            run_decode, run_prefill)

pytestmark = pytest.mark.gpu

MID = workloads.BlockDims(d_model=2048, n_heads=16, n_kv_heads=4, head_dim=128, d_ff=4096)
# 16 query heads per KV head (the wide-group decode kernel, 8-token prefill tiles)
WIDE = workloads.BlockDims(d_model=2048, n_heads=16, n_kv_heads=1, head_dim=128, d_ff=4096)
# one query head per KV head (128-token prefill tiles)
MHA = workloads.BlockDims(d_model=1024, n_heads=8, n_kv_heads=8, head_dim=128, d_ff=2048)


def _oracle_prefill(inp, T_total, max_seq, trace=None):
    w, g = oracle_weights(inp)
    B = inp.x.shape[0]
    kc = np.zeros((B, inp.dims.n_kv_heads, max_seq, inp.dims.head_dim))
    vc = np.zeros_like(kc)
    x = workloads.to_numpy64(inp.x[:, :T_total])
    y = ob.block_forward(x, w, g, inp.dims, kc, vc, 0, rnd_for(inp.dtype), trace=trace)
    return y, kc, vc


def _prefill_then_decode(inp, T, steps, max_seq):
    """GPU: prefill T tokens, then `steps` decode steps; returns y [B, T+steps, d] and caches."""
    blk, ddb = gpu_block(inp, max_seq)
    dev = torch.device("cuda:0")
    kc = inp.k_cache.to(dev)
    vc = inp.v_cache.to(dev)
    x = inp.x.to(dev)
    ys = [run_prefill(blk, ddb, x[:, :T].contiguous(), kc, vc)]
    for s in range(steps):
        ys.append(run_decode(blk, ddb, x[:, T + s:T + s + 1].contiguous(), kc, vc, T + s))
    torch.cuda.synchronize()
    assert blk.poll_error() == 0
    return torch.cat(ys, dim=1), kc, vc, blk, ddb


@pytest.mark.parametrize("random_gains", [False, True])
def test_tiny_fp32_prefill16_decode4(random_gains):
    """The fp32 workload: d=256, 4/2 heads, head_dim 64, prefill 16 then 4 decode steps."""
    cfg = workloads.TINY_FP32
    T, steps = cfg["prefill_tokens"], cfg["decode_steps"]
    max_seq = T + steps + 4
    inp = workloads.make_block_inputs(cfg["dims"], cfg["batch"], T + steps, dtype=torch.float32,
                                      max_seq=max_seq, random_gains=random_gains)
    y_gpu, kc, vc, _, _ = _prefill_then_decode(inp, T, steps, max_seq)
    y_ref, kref, vref = _oracle_prefill(inp, T + steps, max_seq)
    got = workloads.to_numpy64(y_gpu)
    assert np.all(np.isfinite(got))
    assert rel_err(got, y_ref) <= F32_TOL
    n = T + steps
    assert rel_err(workloads.to_numpy64(kc[:, :, :n]), kref[:, :, :n]) <= F32_TOL
    assert rel_err(workloads.to_numpy64(vc[:, :, :n]), vref[:, :, :n]) <= F32_TOL


def test_tiny_fp32_decode_bit_identical_to_prefill():
    cfg = workloads.TINY_FP32
    T, steps = cfg["prefill_tokens"], cfg["decode_steps"]
    max_seq = 32
    inp = workloads.make_block_inputs(cfg["dims"], 1, T + steps, dtype=torch.float32, max_seq=max_seq)
    y_mix, kc_mix, vc_mix, blk, ddb = _prefill_then_decode(inp, T, steps, max_seq)
    dev = torch.device("cuda:0")
    kc = inp.k_cache.to(dev)
    vc = inp.v_cache.to(dev)
    y_full = run_prefill(blk, ddb, inp.x.to(dev), kc, vc)
    torch.cuda.synchronize()
    assert torch.equal(y_full, y_mix)
    n = T + steps
    assert torch.equal(kc[:, :, :n], kc_mix[:, :, :n]) and torch.equal(vc[:, :, :n], vc_mix[:, :, :n])


@pytest.mark.parametrize("dims,B,T,steps", [(MID, 2, 300, 3), (MID, 1, 129, 2), (MID, 3, 17, 2), (WIDE, 2, 200, 3),
                                             (MHA, 2, 260, 2)], ids=["mid-2x300", "mid-1x129", "mid-3x17",
                                                                     "wide-2x200", "mha-2x260"])
def test_bf16_mid_block_parity(dims, B, T, steps):
    """bf16, 128-wide heads, d=2048 (2 K-segments) and d_ff=4096 (4 K-segments):
    token-tiled prefill (ragged token tiles) and weight-streaming decode; GQA
    groups of 4, 16 and 1 query heads per KV head."""
    max_seq = T + steps + 5
    inp = workloads.make_block_inputs(dims, B, T + steps, max_seq=max_seq, random_gains=True)
    y_gpu, kc, vc, _, _ = _prefill_then_decode(inp, T, steps, max_seq)
    tr = {}
    _oracle_prefill(inp, T + steps, max_seq, trace=tr)
    n = T + steps
    check_bf16_output(workloads.to_numpy64(y_gpu), tr["y_exact"], what="y")
    check_bf16_output(workloads.to_numpy64(kc[:, :, :n]), tr["k_exact"], what="k cache")
    check_bf16_output(workloads.to_numpy64(vc[:, :, :n]), tr["v_exact"], what="v cache")
    # rows past the last written position are untouched (still the NaN poison)
    assert torch.isnan(kc[:, :, n:]).all() and torch.isnan(vc[:, :, n:]).all()


@pytest.mark.parametrize("dims,B,T,steps", [(MID, 2, 300, 3), (MID, 1, 64, 2), (WIDE, 1, 250, 3), (MHA, 2, 130, 2)],
                         ids=["mid-2x300", "mid-1x64", "wide-1x250", "mha-2x130"])
def test_bf16_decode_bit_identical_to_prefill(dims, B, T, steps):
    """Decode rows (weight-streaming projections, split-KV attention) equal the
    prefill rows (token-tiled projections, in-CTA attention fold) bit for bit."""
    max_seq = T + steps + 5
    inp = workloads.make_block_inputs(dims, B, T + steps, max_seq=max_seq)
    y_mix, kc_mix, vc_mix, blk, ddb = _prefill_then_decode(inp, T, steps, max_seq)
    dev = torch.device("cuda:0")
    kc = inp.k_cache.to(dev)
    vc = inp.v_cache.to(dev)
    y_full = run_prefill(blk, ddb, inp.x.to(dev), kc, vc)
    torch.cuda.synchronize()
    n = T + steps
    assert torch.equal(kc[:, :, :n], kc_mix[:, :, :n]) and torch.equal(vc[:, :, :n], vc_mix[:, :, :n])
    assert torch.equal(y_full, y_mix)


def test_bf16_zero_branches_return_input():
    """Wo = 0 and W_down = 0: y = x exactly (both residual adds of zero)."""
    inp = workloads.make_block_inputs(MID, 2, 40, max_seq=48)
    inp.weights["wo"].zero_()
    inp.weights["w_down"].zero_()
    y, _, _, _, _ = _prefill_then_decode(inp, 38, 2, 48)
    assert torch.equal(y.cpu(), inp.x)


def test_decode_devpos_matches_decode_and_graph_replay():
    import dense_decoder_block_gb300 as ddb
    T = 70
    max_seq = 80
    inp = workloads.make_block_inputs(MID, 2, T + 3, max_seq=max_seq)
    y_ref, kc_ref, vc_ref, blk, _ = _prefill_then_decode(inp, T, 3, max_seq)
    dev = torch.device("cuda:0")
    kc = inp.k_cache.to(dev)
    vc = inp.v_cache.to(dev)
    x = inp.x.to(dev)
    run_prefill(blk, ddb, x[:, :T].contiguous(), kc, vc)
    kv = ddb.KVCache(kc, vc)
    pos = torch.tensor([T], dtype=torch.int32, device=dev)
    xin = torch.empty(2, 1, MID.d_model, dtype=torch.bfloat16, device=dev)
    yout = torch.empty_like(xin)
    ws = blk.workspace(2, 1)
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        xin.copy_(x[:, T:T + 1])
        blk.decode_devpos(xin, kv, pos, yout, ws, stream)   # warm-up outside capture
        with torch.cuda.graph(graph, stream=stream):
            blk.decode_devpos(xin, kv, pos, yout, ws, stream)
    torch.cuda.current_stream().wait_stream(stream)
    outs = []
    for s in range(3):
        xin.copy_(x[:, T + s:T + s + 1])
        pos.fill_(T + s)
        graph.replay()
        outs.append(yout.clone())
    torch.cuda.synchronize()
    assert blk.poll_error() == 0
    assert torch.equal(torch.cat(outs, dim=1), y_ref[:, T:T + 3])
    n = T + 3
    assert torch.equal(kc[:, :, :n], kc_ref[:, :, :n])


def test_error_paths():
    import dense_decoder_block_gb300 as ddb
    inp = workloads.make_block_inputs(MID, 1, 4, max_seq=8)
    blk, _ = gpu_block(inp, 8)
    dev = torch.device("cuda:0")
    kc, vc = inp.k_cache.to(dev), inp.v_cache.to(dev)
    kv = ddb.KVCache(kc, vc)
    x = inp.x[:, :1].to(dev)
    y = torch.empty_like(x)
    ws = blk.workspace(1, 1)
    with pytest.raises(ddb.LlamaError) as e:
        blk.decode(x, kv, 8, y, ws)
    assert e.value.code == ddb.LLAMA_ERR_POS_RANGE
    with pytest.raises(ddb.LlamaError) as e:
        blk.decode(x, kv, 0, y, ws[:16])
    assert e.value.code == ddb.LLAMA_ERR_WORKSPACE
    # device-side position check: out of range -> error word, nothing written
    pos = torch.tensor([9], dtype=torch.int32, device=dev)
    before = kc.clone()
    blk.decode_devpos(x, kv, pos, y, ws)
    assert blk.poll_error() == ddb.LLAMA_ERR_POS_RANGE
    assert blk.poll_error() == 0
    assert torch.equal(before.isnan(), kc.isnan()) and torch.equal(before.nan_to_num(), kc.nan_to_num())
    # bad dims
    bad = ddb.llama_block_dims(2048, 16, 5, 128, 4096, 8, 1e-5, 5e5, ddb.LLAMA_BF16)
    with pytest.raises(ddb.LlamaError) as e:
        ddb.llama_block_create(bad, blk.c_w)
    assert e.value.code == ddb.LLAMA_ERR_UNSUPPORTED_DIMS


def test_bounded_wait_expiry_is_reported_and_the_handle_recovers():
    """The failure path of every tensor-core kernel's mbarrier waits, run for real:
    a wait that nothing satisfies gives up after its budget, records
    LLAMA_ERR_DEVICE_TIMEOUT in the handle's error word and returns (no trap, no
    fault); the host reads the code once, and the next decode on the same handle and
    context gives the same bits as before."""
    import time
    import dense_decoder_block_gb300 as ddb
    inp = workloads.make_block_inputs(MID, 2, 1, cache_len=40, max_seq=48)
    blk, _ = gpu_block(inp, 48)
    dev = torch.device("cuda:0")
    kv = ddb.KVCache(inp.k_cache.to(dev), inp.v_cache.to(dev))
    x = inp.x.to(dev)
    y0 = torch.empty_like(x)
    ws = blk.workspace(2, 1)
    blk.decode(x, kv, 40, y0, ws)
    assert blk.poll_error() == 0
    t0 = time.perf_counter()
    blk.selftest_wait_timeout(20_000_000)   # 20 ms
    assert blk.poll_error() == ddb.LLAMA_ERR_DEVICE_TIMEOUT
    waited = time.perf_counter() - t0
    assert 0.015 <= waited < 1.5, waited
    assert blk.poll_error() == 0            # read once, then cleared
    y1 = torch.empty_like(x)
    blk.decode(x, kv, 40, y1, ws)
    assert blk.poll_error() == 0
    assert torch.equal(y0, y1)


def test_rmsnorm_step_matches_oracle():
    import dense_decoder_block_gb300 as ddb
    from oracle.bf16 import round_bf16
    gen = torch.Generator().manual_seed(5)
    x = (torch.randn(37, 4096, generator=gen) * 3).to(torch.bfloat16)
    g = (torch.rand(4096, generator=gen) + 0.5).to(torch.bfloat16)
    dev = torch.device("cuda:0")
    y = torch.empty_like(x, device=dev)
    ddb.llama_rmsnorm(x.to(dev), g.to(dev), y, 37, 4096, 1e-5)
    torch.cuda.synchronize()
    ref = ob.rmsnorm(x.double().numpy(), g.double().numpy(), 1e-5, round_bf16)
    got = y.double().cpu().numpy()
    # fp32 reduction vs fp64: at most one bf16 ulp apart, almost always equal
    assert np.all(np.abs(got - ref) <= np.abs(ref) * 2.0 ** -7 + 1e-30)
    assert np.mean(got == ref) > 0.99


@pytest.mark.parametrize("dims,cuts", [(MID, (0, 100, 229, 240, 300)), (WIDE, (0, 130, 131, 200))],
                         ids=["mid-4-chunks", "wide-3-chunks"])
def test_bf16_chunked_prefill_bit_identical_to_one_prefill(dims, cuts):
    """Prefill in chunks at start positions > 0 (chunks crossing 128-key boundaries;
    chunks of 11 tokens and of one token, whose 22 and 2 rows take the
    weight-streaming projections) gives the same rows and cache, bit for bit, as one
    prefill of all the tokens."""
    B, T = 2, cuts[-1]
    max_seq = T + 5
    inp = workloads.make_block_inputs(dims, B, T, max_seq=max_seq)
    blk, ddb = gpu_block(inp, max_seq)
    dev = torch.device("cuda:0")
    x = inp.x.to(dev)
    kc_full, vc_full = inp.k_cache.to(dev), inp.v_cache.to(dev)
    y_full = run_prefill(blk, ddb, x, kc_full, vc_full)
    kc, vc = inp.k_cache.to(dev), inp.v_cache.to(dev)
    kv = ddb.KVCache(kc, vc)
    ys = []
    for a, b in zip(cuts[:-1], cuts[1:]):
        xc = x[:, a:b].contiguous()
        yc = torch.empty_like(xc)
        blk.prefill_at(xc, kv, a, yc, blk.workspace(B, b - a))
        ys.append(yc)
    torch.cuda.synchronize()
    assert blk.poll_error() == 0
    assert torch.equal(torch.cat(ys, dim=1), y_full)
    assert torch.equal(kc[:, :, :T], kc_full[:, :, :T]) and torch.equal(vc[:, :, :T], vc_full[:, :, :T])
    assert torch.isnan(kc[:, :, T:]).all() and torch.isnan(vc[:, :, T:]).all()
    # the same chunks through the oracle: block_forward at each start position on its
    # own cache ("Llama 3 8B · Prepare Q, K, V", decode mode: the new tokens attend to
    # the cached rows and to themselves)
    w, g = oracle_weights(inp)
    kr = np.zeros((B, dims.n_kv_heads, max_seq, dims.head_dim))
    vr = np.zeros_like(kr)
    x64 = workloads.to_numpy64(inp.x)
    exact, k_ex, v_ex = [], [], []
    for a, b in zip(cuts[:-1], cuts[1:]):
        tr = {}
        ob.block_forward(x64[:, a:b], w, g, dims, kr, vr, a, rnd_for(inp.dtype), trace=tr)
        exact.append(tr["y_exact"])
        k_ex.append(tr["k_exact"])
        v_ex.append(tr["v_exact"])
    check_bf16_output(workloads.to_numpy64(torch.cat(ys, dim=1)), np.concatenate(exact, axis=1),
                      what="chunked prefill y")
    check_bf16_output(workloads.to_numpy64(kc[:, :, :T]), np.concatenate(k_ex, axis=2), what="chunked k cache")
    check_bf16_output(workloads.to_numpy64(vc[:, :, :T]), np.concatenate(v_ex, axis=2), what="chunked v cache")


def test_fp32_chunked_prefill_matches_oracle():
    """The fp32 workload prefilled in two chunks (16 then 4 tokens at position 16)
    against the oracle run the same way (block_forward at start_pos 16 on its cache)."""
    cfg = workloads.TINY_FP32
    T0, T1 = 16, 20
    max_seq = 24
    inp = workloads.make_block_inputs(cfg["dims"], 2, T1, dtype=torch.float32, max_seq=max_seq)
    blk, ddb = gpu_block(inp, max_seq)
    dev = torch.device("cuda:0")
    x = inp.x.to(dev)
    kc, vc = inp.k_cache.to(dev), inp.v_cache.to(dev)
    kv = ddb.KVCache(kc, vc)
    y0 = torch.empty_like(x[:, :T0])
    y1 = torch.empty_like(x[:, T0:T1])
    blk.prefill_at(x[:, :T0].contiguous(), kv, 0, y0, blk.workspace(2, T0))
    blk.prefill_at(x[:, T0:T1].contiguous(), kv, T0, y1, blk.workspace(2, T1 - T0))
    torch.cuda.synchronize()
    assert blk.poll_error() == 0
    w, g = oracle_weights(inp)
    kr = np.zeros((2, cfg["dims"].n_kv_heads, max_seq, cfg["dims"].head_dim))
    vr = np.zeros_like(kr)
    x64 = workloads.to_numpy64(inp.x)
    r0 = ob.block_forward(x64[:, :T0], w, g, cfg["dims"], kr, vr, 0, rnd_for(inp.dtype))
    r1 = ob.block_forward(x64[:, T0:T1], w, g, cfg["dims"], kr, vr, T0, rnd_for(inp.dtype))
    assert rel_err(workloads.to_numpy64(y0), r0) <= F32_TOL
    assert rel_err(workloads.to_numpy64(y1), r1) <= F32_TOL
    assert rel_err(workloads.to_numpy64(kc[:, :, :T1]), kr[:, :, :T1]) <= F32_TOL


def test_chunked_prefill_position_range():
    inp = workloads.make_block_inputs(MID, 1, 8, max_seq=16)
    blk, ddb = gpu_block(inp, 16)
    dev = torch.device("cuda:0")
    x = inp.x.to(dev)
    kv = ddb.KVCache(inp.k_cache.to(dev), inp.v_cache.to(dev))
    y = torch.empty_like(x)
    with pytest.raises(ddb.LlamaError) as ei:
        blk.prefill_at(x, kv, 9, y, blk.workspace(1, 8))   # 9 + 8 > max_seq 16
    assert ei.value.code == -3   # LLAMA_ERR_POS_RANGE
    with pytest.raises(ddb.LlamaError):
        blk.prefill_at(x, kv, -1, y, blk.workspace(1, 8))


def test_host_mapped_x_and_y_match_device_buffers():
    """x read from and y written to pinned host memory by the kernels (through
    llama_device_ptr_of_host) give the same bits as device buffers, in prefill and
    decode; unpinned memory is refused."""
    T, steps, max_seq = 200, 2, 208
    inp = workloads.make_block_inputs(MID, 2, T + steps, max_seq=max_seq)
    y_dev, kc_dev, vc_dev, blk, ddb = _prefill_then_decode(inp, T, steps, max_seq)
    dev = torch.device("cuda:0")
    kc, vc = inp.k_cache.to(dev), inp.v_cache.to(dev)
    kv = ddb.KVCache(kc, vc)
    outs = []
    xh = inp.x[:, :T].contiguous().pin_memory()
    yh = torch.empty_like(xh).pin_memory()
    blk.prefill(ddb.HostMapped(xh), kv, ddb.HostMapped(yh), blk.workspace(2, T))
    torch.cuda.synchronize()
    outs.append(yh.clone())
    for s in range(steps):
        xs = inp.x[:, T + s:T + s + 1].contiguous().pin_memory()
        ys = torch.empty_like(xs).pin_memory()
        blk.decode(ddb.HostMapped(xs), kv, T + s, ddb.HostMapped(ys), blk.workspace(2, 1))
        torch.cuda.synchronize()
        outs.append(ys.clone())
    assert blk.poll_error() == 0
    assert torch.equal(torch.cat(outs, dim=1), y_dev.cpu())
    n = T + steps
    assert torch.equal(kc[:, :, :n], kc_dev[:, :, :n]) and torch.equal(vc[:, :, :n], vc_dev[:, :, :n])
    with pytest.raises(ValueError):
        ddb.HostMapped(torch.empty(4))   # not pinned


# 64 query and 32 KV heads: 128 QKV feature tiles, which the decode projection
# streams in a single K-segment (its epilogue in the projection kernel)
ONESEG = workloads.BlockDims(d_model=8192, n_heads=64, n_kv_heads=32, head_dim=128, d_ff=1024)


@pytest.mark.parametrize("dims,pos", [(MID, [5, 127, 128, 257, 300]), (ONESEG, [3, 130])],
                         ids=["mid-segment-sums", "one-segment-qkv"])
def test_decode_per_sequence_positions_bit_identical_to_prefill(dims, pos):
    """One decode step with a position per sequence (MID: chunk counts 1, 1, 2, 2
    and 3, positions on both sides of chunk edges; its QKV projection adds two
    K-segments, ONESEG's streams one): every sequence's output row and new cache
    row equal the prefill rows at its position bit for bit, cache rows past each
    position are left alone, and an out-of-range position is reported."""
    B, T_all = len(pos), max(pos) + 1
    max_seq = T_all + 4
    inp = workloads.make_block_inputs(dims, B, T_all, max_seq=max_seq)
    blk, ddb = gpu_block(inp, max_seq)
    dev = torch.device("cuda:0")
    kc_pf, vc_pf = inp.k_cache.to(dev), inp.v_cache.to(dev)
    x = inp.x.to(dev)
    y_pf = run_prefill(blk, ddb, x, kc_pf, vc_pf)
    # caches holding only rows 0..pos[b]-1 of each sequence
    kc, vc = kc_pf.clone(), vc_pf.clone()
    for b, p in enumerate(pos):
        kc[b, :, p:] = float("nan")
        vc[b, :, p:] = float("nan")
    x_dec = torch.stack([x[b, p] for b, p in enumerate(pos)]).unsqueeze(1).contiguous()
    pos_seq = torch.tensor(pos, dtype=torch.int32, device=dev)
    y = torch.empty_like(x_dec)
    kv = ddb.KVCache(kc, vc)
    blk.decode_seqpos(x_dec, kv, pos_seq, y, blk.workspace(B, 1))
    torch.cuda.synchronize()
    assert blk.poll_error() == 0
    for b, p in enumerate(pos):
        assert torch.equal(y[b, 0], y_pf[b, p]), f"sequence {b} at {p}"
        assert torch.equal(kc[b, :, p], kc_pf[b, :, p]) and torch.equal(vc[b, :, p], vc_pf[b, :, p])
        assert torch.isnan(kc[b, :, p + 1:]).all() and torch.isnan(vc[b, :, p + 1:]).all()
    # against the oracle: each sequence run alone up to its own position, its row p kept
    w, g = oracle_weights(inp)
    x64 = workloads.to_numpy64(inp.x)
    y_ex, k_ex, v_ex = [], [], []
    for b, p in enumerate(pos):
        kr = np.zeros((1, dims.n_kv_heads, p + 1, dims.head_dim))
        vr = np.zeros_like(kr)
        tr = {}
        ob.block_forward(x64[b:b + 1, :p + 1], w, g, dims, kr, vr, 0, rnd_for(inp.dtype), out_rows=[p], trace=tr)
        y_ex.append(tr["y_exact"][0, 0])
        k_ex.append(tr["k_exact"][0, :, p])
        v_ex.append(tr["v_exact"][0, :, p])
    check_bf16_output(workloads.to_numpy64(y[:, 0]), np.stack(y_ex), what="per-sequence decode y")
    check_bf16_output(workloads.to_numpy64(torch.stack([kc[b, :, p] for b, p in enumerate(pos)])), np.stack(k_ex),
                      what="per-sequence decode k rows")
    check_bf16_output(workloads.to_numpy64(torch.stack([vc[b, :, p] for b, p in enumerate(pos)])), np.stack(v_ex),
                      what="per-sequence decode v rows")
    # a position outside the cache is recorded by the kernels
    bad = torch.tensor([max_seq] + pos[1:], dtype=torch.int32, device=dev)
    blk.decode_seqpos(x_dec, kv, bad, y, blk.workspace(B, 1))
    assert blk.poll_error() == ddb.LLAMA_ERR_POS_RANGE
    assert blk.poll_error() == 0


def test_decode_per_sequence_positions_unsupported_shape():
    """The fp32 workload has no per-sequence decode path: refused up front."""
    inp = workloads.make_block_inputs(workloads.TINY, 2, 4, dtype=torch.float32, max_seq=16)
    blk, ddb = gpu_block(inp, 16)
    dev = torch.device("cuda:0")
    kv = ddb.KVCache(inp.k_cache.to(dev), inp.v_cache.to(dev))
    x = inp.x[:, :1].contiguous().to(dev)
    with pytest.raises(ddb.LlamaError):
        blk.decode_seqpos(x, kv, torch.tensor([1, 2], dtype=torch.int32, device=dev), torch.empty_like(x),
                          blk.workspace(2, 1))


def test_bf16_scaled_rope_matches_oracle():
    """Llama 3.1's long-context RoPE schedule (llama_block_create_scaled): a decode step
    at position 6000 and a 20-token chunk at 6001 on a cache of 6000 rows, against the
    oracle with the same schedule; the slow pairs move far enough at this range that
    the unscaled schedule gives a clearly different result."""
    import dataclasses
    dims = dataclasses.replace(MID, rope_scaling=workloads.LLAMA31_ROPE_SCALING)
    P, T, B = 6000, 20, 2
    max_seq = P + T + 1 + 7
    inp = workloads.make_block_inputs(dims, B, T + 1, cache_len=P, max_seq=max_seq, random_gains=True)
    blk, ddb = gpu_block(inp, max_seq)
    dev = torch.device("cuda:0")
    kc, vc = inp.k_cache.to(dev), inp.v_cache.to(dev)
    kv = ddb.KVCache(kc, vc)
    x = inp.x.to(dev)
    y_dec = run_decode(blk, ddb, x[:, :1].contiguous(), kc, vc, P)
    y_chk = torch.empty_like(x[:, 1:])
    blk.prefill_at(x[:, 1:].contiguous(), kv, P + 1, y_chk, blk.workspace(B, T))
    torch.cuda.synchronize()
    assert blk.poll_error() == 0
    w, g = oracle_weights(inp)
    x64 = workloads.to_numpy64(inp.x)

    def oracle(d):
        kr = workloads.to_numpy64(inp.k_cache).copy()
        vr = workloads.to_numpy64(inp.v_cache).copy()
        t0, t1 = {}, {}
        ob.block_forward(x64[:, :1], w, g, d, kr, vr, P, rnd_for(inp.dtype), trace=t0)
        ob.block_forward(x64[:, 1:], w, g, d, kr, vr, P + 1, rnd_for(inp.dtype), trace=t1)
        return (np.concatenate([t0["y_exact"], t1["y_exact"]], axis=1),
                np.concatenate([t0["k_exact"], t1["k_exact"]], axis=2))

    y_ex, k_ex = oracle(dims)
    got = workloads.to_numpy64(torch.cat([y_dec, y_chk], dim=1))
    check_bf16_output(got, y_ex, what="scaled-RoPE y (decode at 6000, chunk at 6001)")
    check_bf16_output(workloads.to_numpy64(kc[:, :, P:P + T + 1]), k_ex, what="scaled-RoPE k rows")
    _, k_plain = oracle(MID)
    k_got = workloads.to_numpy64(kc[:, :, P:P + T + 1])
    assert rel_err(k_got, round_bf16(k_plain)) > 0.1   # the unscaled schedule is far off
