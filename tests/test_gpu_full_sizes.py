"""GPU parity at the full workload sizes: Llama-3 8B-shaped decode (batch 1/8/32 at
1000 cached positions) and prefill (T = 512, 2048, 8192), Llama-3.1 70B-shaped decode
(batch 16 at 8192 cached positions) and prefill (T = 4096).  Decode checks every
output row; prefill checks sampled rows (first, tile edges, middle, ragged tail) and
every K/V cache row.  The launch configuration is the benchmark's."""
import numpy as np
import pytest
import torch

import workloads
from oracle import block as ob
from oracle.bf16 import round_bf16
from tests.blockrun import check_bf16_output, gpu_block, oracle_weights, run_decode, run_prefill

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def w8b():
    wts = workloads.make_weights(workloads.LLAMA3_8B, weight_std=0.02)
    return wts


@pytest.fixture(scope="module")
def w8b_oracle(w8b):
    to64 = workloads.to_numpy64
    return {k: to64(v) for k, v in w8b[0].items()}, {k: to64(v) for k, v in w8b[1].items()}


def _decode_case(dims, wts, wts64, B, pos, max_seq):
    inp = workloads.make_block_inputs(dims, B, 1, cache_len=pos, max_seq=max_seq, weights=wts)
    blk, ddb = gpu_block(inp, max_seq)
    dev = torch.device("cuda:0")
    kc, vc = inp.k_cache.to(dev), inp.v_cache.to(dev)
    y = run_decode(blk, ddb, inp.x.to(dev), kc, vc, pos)
    torch.cuda.synchronize()
    assert blk.poll_error() == 0
    # kernels per decode step: 8B -- the gate/up pair in one K-segment (epilogue in the
    # projection), QKV, O and down with a reduction each; 70B -- gate/up in two segments
    assert blk.launch_count() == (10 if dims is workloads.LLAMA3_8B else 11)
    # rows past pos were NaN and stay NaN; nothing beyond pos was read (y finite)
    if pos + 1 < max_seq:
        assert torch.isnan(kc[:, :, pos + 1:]).all()
    kc64 = workloads.to_numpy64(inp.k_cache)
    vc64 = workloads.to_numpy64(inp.v_cache)
    tr = {}
    ob.block_forward(workloads.to_numpy64(inp.x), wts64[0], wts64[1], dims, kc64, vc64, pos, round_bf16, trace=tr)
    check_bf16_output(workloads.to_numpy64(y), tr["y_exact"], what=f"decode y B={B} pos={pos}")
    check_bf16_output(workloads.to_numpy64(kc[:, :, pos:pos + 1]), tr["k_exact"], what="decode k row")
    check_bf16_output(workloads.to_numpy64(vc[:, :, pos:pos + 1]), tr["v_exact"], what="decode v row")
    # rows before pos are the caller's and untouched
    assert torch.equal(kc[:, :, :pos].cpu(), inp.k_cache[:, :, :pos])


@pytest.mark.parametrize("B", [1, 8, 32])
def test_decode_8b_pos1000(w8b, w8b_oracle, B):
    _decode_case(workloads.LLAMA3_8B, w8b, w8b_oracle, B, 1000, 1024)


@pytest.mark.parametrize("pos", [0, 1023])
def test_decode_8b_edge_positions(w8b, w8b_oracle, pos):
    _decode_case(workloads.LLAMA3_8B, w8b, w8b_oracle, 2, pos, 1024)


def _sample_rows(T):
    rows = {0, 1, 2, 127, 128, 129, 255, 256, T // 2, T // 2 + 1, T - 3, T - 2, T - 1}
    rng = np.random.default_rng(T)
    rows |= set(rng.integers(0, T, 6).tolist())
    return sorted(r for r in rows if 0 <= r < T)


def _prefill_case(dims, wts, wts64, T, B=1):
    max_seq = T + 64
    inp = workloads.make_block_inputs(dims, B, T, max_seq=max_seq, weights=wts)
    blk, ddb = gpu_block(inp, max_seq)
    dev = torch.device("cuda:0")
    kc, vc = inp.k_cache.to(dev), inp.v_cache.to(dev)
    y = run_prefill(blk, ddb, inp.x.to(dev), kc, vc)
    torch.cuda.synchronize()
    assert blk.poll_error() == 0
    # 8 when the token-tiled projections carry their epilogues; with few tokens the down
    # projection runs its K-segments on separate CTAs and a reduction kernel applies its
    # epilogue (one more)
    assert blk.launch_count() == (9 if T < 1024 else 8)
    rows = _sample_rows(T)
    kc64 = np.zeros((B, dims.n_kv_heads, max_seq, dims.head_dim))
    vc64 = np.zeros_like(kc64)
    tr = {}
    ob.block_forward(workloads.to_numpy64(inp.x), wts64[0], wts64[1], dims, kc64, vc64, 0, round_bf16,
                     out_rows=rows, trace=tr)
    check_bf16_output(workloads.to_numpy64(y[:, rows]), tr["y_exact"], what=f"prefill y T={T} (rows)")
    check_bf16_output(workloads.to_numpy64(kc[:, :, :T]), tr["k_exact"], what=f"prefill k cache T={T}")
    check_bf16_output(workloads.to_numpy64(vc[:, :, :T]), tr["v_exact"], what=f"prefill v cache T={T}")
    assert torch.isnan(kc[:, :, T:]).all()


@pytest.mark.parametrize("T", [512, 2048, 8192])
def test_prefill_8b(w8b, w8b_oracle, T):
    _prefill_case(workloads.LLAMA3_8B, w8b, w8b_oracle, T)


@pytest.fixture(scope="module")
def w70b():
    return workloads.make_weights(workloads.LLAMA31_70B, weight_std=0.01)


@pytest.fixture(scope="module")
def w70b_oracle(w70b):
    to64 = workloads.to_numpy64
    return {k: to64(v) for k, v in w70b[0].items()}, {k: to64(v) for k, v in w70b[1].items()}


def test_decode_70b_b16_pos8192(w70b, w70b_oracle):
    _decode_case(workloads.LLAMA31_70B, w70b, w70b_oracle, 16, 8192, 8192 + 64)


def test_prefill_70b_t4096(w70b, w70b_oracle):
    _prefill_case(workloads.LLAMA31_70B, w70b, w70b_oracle, 4096)
