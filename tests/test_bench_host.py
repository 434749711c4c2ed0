"""Host-side accounting of bench.py (no GPU): the algorithmic bytes a decode step
moves, with one position for the batch and with one position per sequence."""
import os
import sys

import workloads

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def test_decode_bytes_8b_batch32_pos1000():
    """Every weight once (bf16), K and V rows 0..1000 of each (sequence, KV head),
    the new K and V rows, x read and y written."""
    d, f, hq, hkv, dh = 4096, 14336, 32, 8, 128
    weights = d * (hq * dh + 2 * hkv * dh) + hq * dh * d + 3 * d * f + 2 * d
    kv_rows = 2 * 32 * hkv * 1001 * dh
    expect = 2 * (weights + kv_rows + 2 * 32 * hkv * dh + 2 * 32 * d)
    assert bench.decode_step_bytes(workloads.LLAMA3_8B, 32, 1000) == expect == 568082432


def test_per_sequence_bytes_reduce_to_the_uniform_case():
    for dims in (workloads.LLAMA3_8B, workloads.LLAMA31_70B):
        for B, p in ((1, 0), (8, 127), (32, 1000)):
            assert bench.decode_seqpos_bytes(dims, [p] * B) == bench.decode_step_bytes(dims, B, p)


def test_per_sequence_bytes_count_each_sequence_rows():
    dims = workloads.LLAMA3_8B
    a = bench.decode_seqpos_bytes(dims, [10, 20])
    b = bench.decode_seqpos_bytes(dims, [15, 15])
    assert a == b   # the same rows in total
    assert bench.decode_seqpos_bytes(dims, [10, 21]) - a == 2 * 2 * dims.n_kv_heads * dims.head_dim
