"""GPU parity of a small decoder stack (token embedding, L blocks, final RMSNorm +
LM head + greedy choice) against the oracle, prefill then teacher-forced decode
steps; and the stack's decode logits bit-identical to a longer prefill's."""
import numpy as np
import pytest
import torch

import workloads
from oracle import block as ob
from tests.parity_log import record_parity

pytestmark = pytest.mark.gpu

# d = 512 (4 query heads, 2 KV heads of 128), d_ff = 1536, 3 layers, vocabulary 1024
SMALL = workloads.BlockDims(d_model=512, n_heads=4, n_kv_heads=2, head_dim=128, d_ff=1536)
LAYERS, VOCAB, B, T, STEPS = 3, 1024, 2, 20, 4
LOGIT_TOL = 2e-2    # max |err| / rms(ref) of the fp32 logits after three bf16 blocks (the bf16 bound)
LOGIT_RMS_TOL = 1e-2


def _stack_inputs():
    layers = [workloads.make_weights(SMALL, weight_std=0.02, seed=100 + i, random_gains=True) for i in range(LAYERS)]
    gen = torch.Generator().manual_seed(11)
    w_embed = torch.randn(VOCAB, SMALL.d_model, generator=gen).to(torch.bfloat16)
    g_final = (torch.rand(SMALL.d_model, generator=gen) + 0.5).to(torch.bfloat16)
    w_out = torch.randn(VOCAB, SMALL.d_model, generator=gen).mul_(0.05).to(torch.bfloat16)
    ids = workloads.make_token_ids(B, T + STEPS, VOCAB, seed=12)
    return layers, w_embed, g_final, w_out, ids


def _gpu_stack(layers, w_embed, g_final, w_out, max_seq):
    import dense_decoder_block_gb300 as ddb
    from dense_decoder_block_gb300.stack import LlamaStack
    ddb.lib()
    dev = torch.device("cuda:0")
    dl = [({k: v.to(dev) for k, v in w.items()}, {k: v.to(dev) for k, v in g.items()}) for w, g in layers]
    st = LlamaStack(SMALL, dl, w_embed.to(dev), g_final.to(dev), w_out.to(dev), batch=B, max_seq=max_seq,
                    prefill_tokens=T + 1)
    return st, dl


def _oracle_hidden(layers, w_embed, ids):
    """h after the L blocks at every position (causal, so position p depends on 0..p only)."""
    to64 = workloads.to_numpy64
    h = ob.embed(ids.numpy(), to64(w_embed))
    n = ids.shape[1]
    for w, g in layers:
        kc = np.zeros((B, SMALL.n_kv_heads, n, SMALL.head_dim))
        vc = np.zeros_like(kc)
        h = ob.block_forward(h, {k: to64(v) for k, v in w.items()}, {k: to64(v) for k, v in g.items()}, SMALL,
                             kc, vc, 0)
    return h


def _check_logits(got, ref, what):
    rms = float(np.sqrt(np.mean(ref ** 2)))
    err = np.abs(got - ref)
    record_parity(f"[parity] {what}: max|err|/rms = {err.max() / rms:.3e}, "
                  f"rms err / rms = {np.sqrt(np.mean(err ** 2)) / rms:.3e}")
    assert np.all(np.isfinite(got))
    assert err.max() <= LOGIT_TOL * rms and np.sqrt(np.mean(err ** 2)) <= LOGIT_RMS_TOL * rms
    return err.max()


def _check_ids(ids, logits_ref, bound):
    """Greedy ids equal the oracle's wherever its top-2 margin exceeds twice the
    error bound; elsewhere the chosen logit is within the bound of the max."""
    for b in range(logits_ref.shape[0]):
        row = logits_ref[b]
        top = np.argsort(row)[::-1][:2]
        if row[top[0]] - row[top[1]] > 2 * bound:
            assert int(ids[b]) == int(top[0])
        else:
            assert row[int(ids[b])] >= row[top[0]] - 2 * bound


def test_stack_prefill_and_teacher_forced_decode_match_oracle():
    layers, w_embed, g_final, w_out, ids = _stack_inputs()
    st, _ = _gpu_stack(layers, w_embed, g_final, w_out, max_seq=T + STEPS + 4)
    dev = torch.device("cuda:0")
    ids_dev = ids.to(dev)
    h_ref = _oracle_hidden(layers, w_embed, ids)
    to64 = workloads.to_numpy64
    head = lambda p: ob.lm_head_logits(h_ref[:, p, :], to64(g_final), to64(w_out), SMALL.eps)

    st.prefill(ids_dev[:, :T].contiguous())
    torch.cuda.synchronize()
    assert st.poll_error() == 0 and int(st.err.item()) == 0
    ref = head(T - 1)
    bound = _check_logits(st.logits.double().cpu().numpy(), ref, "prefill logits")
    _check_ids(st.ids.cpu().numpy(), ref, bound)
    for s in range(STEPS):
        st.ids.copy_(ids_dev[:, T + s])   # teacher forcing: the next input is the given token
        st.decode_step()
        torch.cuda.synchronize()
        assert st.poll_error() == 0 and int(st.pos.item()) == T + s + 1
        ref = head(T + s)
        bound = _check_logits(st.logits.double().cpu().numpy(), ref, f"decode step {s} logits")
        _check_ids(st.ids.cpu().numpy(), ref, bound)


def test_stack_decode_logits_bit_identical_to_prefill():
    """Prefill T tokens then decode token T gives the same logits, bit for bit, as
    prefilling T + 1 tokens (every block's decode row equals its prefill row)."""
    layers, w_embed, g_final, w_out, ids = _stack_inputs()
    st, _ = _gpu_stack(layers, w_embed, g_final, w_out, max_seq=T + 8)
    dev = torch.device("cuda:0")
    ids_dev = ids.to(dev)
    st.prefill(ids_dev[:, :T].contiguous())
    st.ids.copy_(ids_dev[:, T])
    st.decode_step()
    torch.cuda.synchronize()
    logits_dec, ids_dec = st.logits.clone(), st.ids.clone()
    st.prefill(ids_dev[:, :T + 1].contiguous())
    torch.cuda.synchronize()
    assert st.poll_error() == 0
    assert torch.equal(st.logits, logits_dec) and torch.equal(st.ids, ids_dec)


def test_stack_decode_replays_as_a_graph():
    """decode_step captured once in a CUDA graph and replayed gives the same ids and
    logits as eager steps (the position lives on the device)."""
    layers, w_embed, g_final, w_out, ids = _stack_inputs()
    st, _ = _gpu_stack(layers, w_embed, g_final, w_out, max_seq=T + 2 * STEPS + 8)
    dev = torch.device("cuda:0")
    ids_dev = ids.to(dev)
    st.prefill(ids_dev[:, :T].contiguous())
    eager = []
    for _ in range(STEPS):
        st.decode_step()
        eager.append((st.ids.clone(), st.logits.clone()))
    # again from the same prefill, now through a captured graph
    st.prefill(ids_dev[:, :T].contiguous())
    torch.cuda.synchronize()
    ids0, pos0 = st.ids.clone(), st.pos.clone()
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        st.decode_step(side)              # warm-up outside the capture
        torch.cuda.synchronize()
        st.ids.copy_(ids0)
        st.pos.copy_(pos0)
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=side):
            st.decode_step(side)
    torch.cuda.synchronize()
    st.ids.copy_(ids0)
    st.pos.copy_(pos0)
    torch.cuda.synchronize()
    for k in range(STEPS):
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(st.ids, eager[k][0]) and torch.equal(st.logits, eager[k][1])
    assert int(st.pos.item()) == T + STEPS and st.poll_error() == 0
