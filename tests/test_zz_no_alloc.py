"""The LM head entry point that allocates nothing (llama_lmhead_argmax_noalloc).

It exists for callers that cannot allocate device memory and so cannot pass a
workspace.  It must give the same logits and token ids as llama_lmhead_argmax,
on the first call in a process and on the calls after it (its scratch array is
shared and keeps the previous call's contents).  This file runs last so that a
failure here does not stop the other GPU tests."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

LOGIT_TOL = 1e-3   # the same bound as the LM head parity test (max|err| / rms)


def _inputs(batch, d, vocab, seed):
    gen = torch.Generator().manual_seed(seed)
    h = torch.randn(batch, d, generator=gen).mul_(2.0).to(torch.bfloat16)
    g = (torch.rand(d, generator=gen) + 0.5).to(torch.bfloat16)
    w = torch.randn(vocab, d, generator=gen).mul_(0.02).to(torch.bfloat16)
    return h, g, w


def _run_with_workspace(ddb, h, g, w, batch, d, vocab):
    dev = h.device
    ids = torch.empty(batch, dtype=torch.int32, device=dev)
    logits = torch.empty(batch, vocab, dtype=torch.float32, device=dev)
    nbytes = ddb.llama_lmhead_workspace_bytes(batch, d, vocab)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    ddb.llama_lmhead_argmax(h, batch, d, g, w, vocab, d, 1e-5, ids, logits, ws, nbytes)
    return ids, logits


def test_noalloc_lmhead_matches_workspace_version_twice():
    import dense_decoder_block_gb300 as ddb
    ddb.lib()
    dev = torch.device("cuda:0")
    d, vocab = 4096, 128256
    for call, (batch, seed) in enumerate([(32, 11), (5, 12)]):   # two calls in a row, different inputs
        h, g, w = (t.to(dev) for t in _inputs(batch, d, vocab, seed))
        ids_ref, logits_ref = _run_with_workspace(ddb, h, g, w, batch, d, vocab)
        ids = torch.full((batch,), -1, dtype=torch.int32, device=dev)
        logits = torch.full((batch, vocab), float("nan"), dtype=torch.float32, device=dev)
        ddb.llama_lmhead_argmax_noalloc(h, batch, d, g, w, vocab, d, 1e-5, ids, logits)
        torch.cuda.synchronize()
        ref = logits_ref.double().cpu().numpy()
        got = logits.double().cpu().numpy()
        rms = np.sqrt(np.mean(ref ** 2))
        assert np.all(np.isfinite(got)), f"call {call}: logits not all written"
        assert np.max(np.abs(got - ref)) / rms <= LOGIT_TOL, f"call {call}"
        assert torch.equal(ids, ids_ref), f"call {call}"


@pytest.mark.parametrize("batch,d,stride,vocab", [(7, 4096, 4096 + 256, 1024), (32, 8192, 8192, 2048)],
                         ids=["rows-strided", "scratch-full"])
def test_noalloc_lmhead_strided_rows_and_full_scratch(batch, d, stride, vocab):
    """Rows read at a stride larger than d_model (one norm launch per row), and the
    largest shape the scratch holds (32 rows of 8192)."""
    import dense_decoder_block_gb300 as ddb
    ddb.lib()
    dev = torch.device("cuda:0")
    h, g, w = (t.to(dev) for t in _inputs(batch, d, vocab, 13))
    hs = torch.zeros(batch, stride, dtype=torch.bfloat16, device=dev)
    hs[:, :d] = h
    ids_ref, logits_ref = _run_with_workspace(ddb, h, g, w, batch, d, vocab)
    ids = torch.full((batch,), -1, dtype=torch.int32, device=dev)
    logits = torch.full((batch, vocab), float("nan"), dtype=torch.float32, device=dev)
    ddb.llama_lmhead_argmax_noalloc(hs, batch, stride, g, w, vocab, d, 1e-5, ids, logits)
    torch.cuda.synchronize()
    assert torch.equal(logits, logits_ref)
    assert torch.equal(ids, ids_ref)


def test_noalloc_lmhead_rejects_sizes_beyond_its_scratch():
    import dense_decoder_block_gb300 as ddb
    ddb.lib()
    dev = torch.device("cuda:0")
    h = torch.zeros(33, 256, dtype=torch.bfloat16, device=dev)
    g = torch.ones(256, dtype=torch.bfloat16, device=dev)
    w = torch.zeros(128, 256, dtype=torch.bfloat16, device=dev)
    ids = torch.empty(33, dtype=torch.int32, device=dev)
    logits = torch.empty(33, 128, dtype=torch.float32, device=dev)
    with pytest.raises(ddb.LlamaError) as e:
        ddb.llama_lmhead_argmax_noalloc(h, 33, 256, g, w, 128, 256, 1e-5, ids, logits)
    assert e.value.code == ddb.LLAMA_ERR_WORKSPACE
    # one row wider than the scratch's 8192 columns
    h = torch.zeros(1, 8320, dtype=torch.bfloat16, device=dev)
    g = torch.ones(8320, dtype=torch.bfloat16, device=dev)
    w = torch.zeros(128, 8320, dtype=torch.bfloat16, device=dev)
    with pytest.raises(ddb.LlamaError) as e:
        ddb.llama_lmhead_argmax_noalloc(h, 1, 8320, g, w, 128, 8320, 1e-5, ids, logits)
    assert e.value.code == ddb.LLAMA_ERR_WORKSPACE
