"""The per-CTA timeline (llama_trace_begin / llama_trace_end).  The product build
refuses it and carries no tracing code; the trace build (the same sources with
LLAMA_TRACE, run in a process of its own by tests/trace_check.py) writes one
record per CTA of the block's kernels while it is on, none once it is off, drops
what exceeds the capacity, and leaves the block's output bits unchanged."""
import json
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_product_build_refuses_tracing():
    import dense_decoder_block_gb300 as ddb
    ddb.lib()
    with pytest.raises(ddb.LlamaError) as e:
        with ddb.Trace(16, torch.device("cuda:0")):
            pass
    assert e.value.code == ddb.LLAMA_ERR_UNSUPPORTED_DIMS


def test_trace_build_records_each_cta_and_changes_nothing():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "trace_check.py")], capture_output=True,
                       text=True, timeout=900, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-3000:]
    out = json.loads(r.stdout.strip().splitlines()[-1])
    assert out["same_bits"] and out["poll"] == 0
    assert 0 < out["n"] == out["claimed"] <= 4096
    assert out["after_off"] == out["claimed"]
    assert {1, 2, 8, 9} <= set(out["kinds"]) <= {1, 2, 4, 5, 6, 7, 8, 9, 12}
    assert out["times_ordered"]
    assert out["max_sm"] < out["n_sm"]
    assert out["small_claimed"] > 5 and out["small_n"] == 5
