"""GPU parity of the stack head (token embedding gather; final RMSNorm + LM head +
greedy choice) against the oracle, at the 8B shape (d = 4096, V = 128,256)."""
import numpy as np
import pytest
import torch

import workloads
from oracle import block as ob
from oracle.bf16 import round_bf16

pytestmark = pytest.mark.gpu

LOGIT_TOL = 1e-3   # fp32 logits: max|err| / rms(ref); the oracle accumulates in fp64


def _head_inputs(batch, d=4096, vocab=workloads.VOCAB, seed=7):
    gen = torch.Generator().manual_seed(seed)
    h = torch.randn(batch, d, generator=gen).mul_(2.0).to(torch.bfloat16)
    g = (torch.rand(d, generator=gen) + 0.5).to(torch.bfloat16)
    w = torch.randn(vocab, d, generator=gen).mul_(0.02).to(torch.bfloat16)
    return h, g, w


def _check_ids(ids, logits_ref, tol_abs):
    """Ids must equal the oracle's argmax wherever its top-2 margin exceeds the
    error bound; elsewhere the GPU's id must be within the bound of the max."""
    for b in range(logits_ref.shape[0]):
        row = logits_ref[b]
        top = np.argsort(row)[::-1][:2]
        if row[top[0]] - row[top[1]] > 2 * tol_abs:
            assert ids[b] == top[0]
        else:
            assert row[ids[b]] >= row[top[0]] - 2 * tol_abs


@pytest.mark.parametrize("batch", [1, 4, 32])
def test_lmhead_argmax_matches_oracle(batch):
    import dense_decoder_block_gb300 as ddb
    ddb.lib()
    h, g, w = _head_inputs(batch)
    dev = torch.device("cuda:0")
    hd, gd, wd = h.to(dev), g.to(dev), w.to(dev)
    ids = torch.empty(batch, dtype=torch.int32, device=dev)
    logits = torch.empty(batch, w.shape[0], dtype=torch.float32, device=dev)
    nbytes = ddb.llama_lmhead_workspace_bytes(batch, 4096, w.shape[0])
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    ddb.llama_lmhead_argmax(hd, batch, 4096, gd, wd, w.shape[0], 4096, 1e-5, ids, logits, ws, nbytes)
    torch.cuda.synchronize()
    ref = ob.lm_head_logits(h.double().numpy(), g.double().numpy(), w.double().numpy(), 1e-5, round_bf16)
    got = logits.double().cpu().numpy()
    rms = np.sqrt(np.mean(ref ** 2))
    assert np.max(np.abs(got - ref)) / rms <= LOGIT_TOL
    _check_ids(ids.cpu().numpy(), ref, LOGIT_TOL * rms)
    # the greedy choice is integer work on the kernel's own fp32 logits: exact
    assert np.array_equal(ids.cpu().numpy(), np.argmax(logits.cpu().numpy(), axis=1))


@pytest.mark.parametrize("shift", [1, 4, workloads.VOCAB // 2], ids=["same-thread", "next-thread", "other-slice"])
@pytest.mark.parametrize("offset", [0, 1], ids=["aligned-logits", "unaligned-logits"])
def test_lmhead_argmax_ties_take_the_first_index(shift, offset):
    """Weight rows repeated at a distance `shift` give every logit twice (the
    projection sums each output column in the same order); the id must be the
    first index of the maximum wherever the two copies tie, which puts the
    tie inside one thread's 16-byte load, across neighbouring threads, or across
    the CTAs that split a row.  A logits buffer one float off 16-byte alignment
    takes the scalar loads."""
    import dense_decoder_block_gb300 as ddb
    ddb.lib()
    batch, V = 32, workloads.VOCAB
    h, g, w = _head_inputs(batch, seed=11)
    src = np.arange(V)
    rep = src[(src // shift) % 2 == 1] if shift < V // 2 else src[V // 2:]
    w[rep] = w[rep - shift]
    dev = torch.device("cuda:0")
    ids = torch.empty(batch, dtype=torch.int32, device=dev)
    buf = torch.empty(batch * V + offset, dtype=torch.float32, device=dev)
    logits = buf[offset:].view(batch, V)
    nbytes = ddb.llama_lmhead_workspace_bytes(batch, 4096, V)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    ddb.llama_lmhead_argmax(h.to(dev), batch, 4096, g.to(dev), w.to(dev), V, 4096, 1e-5, ids, logits, ws, nbytes)
    torch.cuda.synchronize()
    lg = logits.cpu().numpy()
    got = ids.cpu().numpy()
    assert np.array_equal(got, np.argmax(lg, axis=1))
    ties = sum(int(np.count_nonzero(lg[b] == lg[b].max()) > 1) for b in range(batch))
    assert ties == batch, f"only {ties} of {batch} rows have their maximum twice"


def test_embed_gather_and_bad_id():
    import dense_decoder_block_gb300 as ddb
    ddb.lib()
    dev = torch.device("cuda:0")
    gen = torch.Generator().manual_seed(3)
    table = torch.randn(1000, 256, generator=gen).to(torch.bfloat16)
    ids = torch.randint(0, 1000, (37,), generator=gen, dtype=torch.int64).to(torch.int32)
    x = torch.empty(37, 256, dtype=torch.bfloat16, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    ddb.llama_embed(ids.to(dev), 37, table.to(dev), 1000, 256, x, err)
    torch.cuda.synchronize()
    assert torch.equal(x.cpu(), torch.from_numpy(ob.embed(ids.numpy(), table.float().numpy())).to(torch.bfloat16))
    assert int(err.item()) == 0
    bad = ids.clone()
    bad[5] = 1000
    ddb.llama_embed(bad.to(dev), 37, table.to(dev), 1000, 256, x, err)
    torch.cuda.synchronize()
    assert int(err.item()) == ddb.LLAMA_ERR_INVALID_ARG
    assert torch.all(x[5].cpu() == 0)
