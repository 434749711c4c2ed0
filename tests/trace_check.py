"""Run by tests/test_gpu_trace.py in a process of its own: loads the trace build
of the library (libllama_block_trace.so) before anything else loads the product
build, traces decode steps of a small block and prints what it saw as one JSON
line."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads  # noqa: E402
from dense_decoder_block_gb300 import _native  # noqa: E402
from dense_decoder_block_gb300 import build as _build  # noqa: E402


def main():
    _native.load(_build.build(trace=True))
    import dense_decoder_block_gb300 as ddb
    from tests.blockrun import gpu_block
    dims = workloads.BlockDims(d_model=2048, n_heads=16, n_kv_heads=4, head_dim=128, d_ff=4096)
    inp = workloads.make_block_inputs(dims, 4, 1, cache_len=300, max_seq=320)
    blk, _ = gpu_block(inp, 320)
    dev = torch.device("cuda:0")
    kv = ddb.KVCache(inp.k_cache.to(dev), inp.v_cache.to(dev))
    x = inp.x.to(dev)
    ws = blk.workspace(4, 1)
    y0 = torch.empty_like(x)
    blk.decode(x, kv, 300, y0, ws)
    with ddb.Trace(4096, dev) as tr:
        y1 = torch.empty_like(x)
        blk.decode(x, kv, 300, y1, ws)
        torch.cuda.synchronize()
    rec = tr.records()
    y2 = torch.empty_like(x)
    blk.decode(x, kv, 300, y2, ws)      # tracing off again
    torch.cuda.synchronize()
    after_off = int(tr.count.item())
    with ddb.Trace(5, dev) as small:
        blk.decode(x, kv, 300, y2, ws)
        torch.cuda.synchronize()
    srec = small.records()
    ok_times = all(rec["t_start"][i] <= rec["t_end"][i] and
                   (rec["t_release"][i] == 0 or rec["t_start"][i] <= rec["t_release"][i] <= rec["t_end"][i])
                   for i in range(len(rec["kernel"])))
    print(json.dumps({
        "n": len(rec["kernel"]), "claimed": rec["claimed"], "after_off": after_off,
        "kinds": sorted({k & 0xff for k in rec["kernel"]}), "times_ordered": ok_times,
        "max_sm": max(rec["sm"]), "n_sm": torch.cuda.get_device_properties(0).multi_processor_count,
        "same_bits": bool(torch.equal(y0, y1) and torch.equal(y0, y2)), "poll": blk.poll_error(),
        "small_claimed": srec["claimed"], "small_n": len(srec["kernel"])}))


if __name__ == "__main__":
    main()
