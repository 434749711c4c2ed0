"""A decoder-only stack sequenced from the library's calls.

"How Llama 3.1 Generates the Next Token" (the transformer blocks, Unembedding,
Sampling) and "Llama 3.1 70B" (Token embedding, Transformer layer, LM head):
token ids are embedded, pass through L decoder blocks, and the last position's
hidden state goes through the final RMSNorm and the LM head; the next id is the
greedy choice.  Every arithmetic step runs in the library's kernels
(llama_embed, llama_block_prefill / llama_block_decode_devpos,
llama_lmhead_argmax); this module only orders the calls and owns the per-layer
KV caches and the scratch buffers, all allocated once.
"""
from __future__ import annotations

import contextlib
from typing import Callable, Dict, List, Optional, Sequence, Tuple

import torch

from . import (KVCache, LlamaBlock, llama_embed, llama_lmhead_argmax, llama_lmhead_workspace_bytes)


class LlamaStack:
    """L blocks of one shape plus embedding and head, for `batch` sequences of up to
    `max_seq` positions.  Weights are borrowed (device tensors, [out, in] bf16)."""

    def __init__(self, dims, layers: Sequence[Tuple[Dict[str, torch.Tensor], Dict[str, torch.Tensor]]],
                 w_embed: torch.Tensor, g_final: torch.Tensor, w_out: torch.Tensor, batch: int, max_seq: int,
                 prefill_tokens: int):
        dev = w_embed.device
        dt = w_embed.dtype
        self.dims, self.batch, self.max_seq, self.prefill_tokens = dims, batch, max_seq, prefill_tokens
        self.vocab = w_embed.shape[0]
        self.w_embed, self.g_final, self.w_out = w_embed, g_final, w_out
        self.blocks: List[LlamaBlock] = [LlamaBlock(dims, w, g, max_seq) for w, g in layers]
        shape = (batch, dims.n_kv_heads, max_seq, dims.head_dim)
        self.caches: List[KVCache] = [KVCache(torch.zeros(shape, dtype=dt, device=dev),
                                              torch.zeros(shape, dtype=dt, device=dev)) for _ in layers]
        ws_bytes = max(self.blocks[0].workspace_bytes(batch, prefill_tokens), self.blocks[0].workspace_bytes(batch, 1))
        self.ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
        # activations ping-pong between two flat buffers large enough for the prefill
        self.act = [torch.empty(batch * prefill_tokens * dims.d_model, dtype=dt, device=dev) for _ in range(2)]
        self.head_ws = torch.empty(llama_lmhead_workspace_bytes(batch, dims.d_model, self.vocab), dtype=torch.uint8,
                                   device=dev)
        self.logits = torch.empty(batch, self.vocab, dtype=torch.float32, device=dev)
        self.ids = torch.zeros(batch, dtype=torch.int32, device=dev)   # the chosen ids (decode feeds them back)
        self.pos = torch.zeros(1, dtype=torch.int32, device=dev)       # the decode position, on the device
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)       # out-of-range ids from llama_embed

    @staticmethod
    def _on(stream):
        # the position counter is updated on the stream the library calls were issued on
        return torch.cuda.stream(stream) if stream is not None else contextlib.nullcontext()

    def _acts(self, T: int):
        n = self.batch * T * self.dims.d_model
        return [a[:n].view(self.batch, T, self.dims.d_model) for a in self.act]

    def _head(self, x: torch.Tensor, T: int, stream) -> None:
        # the last position of each sequence: rows T-1, 2T-1, ... of x [B, T, d], i.e.
        # B rows T * d elements apart starting at row T-1
        last = x.view(-1)[(T - 1) * self.dims.d_model:]
        llama_lmhead_argmax(last, self.batch, T * self.dims.d_model, self.g_final, self.w_out, self.vocab,
                            self.dims.d_model, self.dims.eps, self.ids, self.logits, self.head_ws,
                            self.head_ws.numel(), stream)

    def prefill(self, ids: torch.Tensor, stream: Optional[torch.cuda.Stream] = None,
                on_layer: Optional[Callable[[int, torch.Tensor], None]] = None) -> None:
        """ids [B, T] int32 on the device, positions 0..T-1.  Leaves the logits of the
        last position in self.logits, the greedy ids in self.ids, and self.pos = T.
        ``on_layer(l, h)``, if given, sees the embedding (l = -1) and each block's
        output h [B, T, d] as soon as its call is enqueued (for inspection)."""
        B, T = ids.shape
        assert B == self.batch and T <= self.prefill_tokens
        x, y = self._acts(T)
        llama_embed(ids, B * T, self.w_embed, self.vocab, self.dims.d_model, x, self.err, stream)
        if on_layer:
            on_layer(-1, x)
        for l, (blk, kv) in enumerate(zip(self.blocks, self.caches)):
            blk.prefill(x, kv, y, self.ws, stream)
            if on_layer:
                on_layer(l, y)
            x, y = y, x
        self._head(x, T, stream)
        with self._on(stream):
            self.pos.fill_(T)

    def decode_step(self, stream: Optional[torch.cuda.Stream] = None,
                    on_layer: Optional[Callable[[int, torch.Tensor], None]] = None) -> None:
        """One token for every sequence at position self.pos (on the device): embeds
        self.ids, runs the blocks, writes the next ids into self.ids and advances
        self.pos.  Capturable in a CUDA graph (nothing is read on the host) when
        ``on_layer`` (as in prefill) is not given."""
        x, y = self._acts(1)
        llama_embed(self.ids, self.batch, self.w_embed, self.vocab, self.dims.d_model, x, self.err, stream)
        if on_layer:
            on_layer(-1, x)
        for l, (blk, kv) in enumerate(zip(self.blocks, self.caches)):
            blk.decode_devpos(x, kv, self.pos, y, self.ws, stream)
            if on_layer:
                on_layer(l, y)
            x, y = y, x
        self._head(x, 1, stream)
        with self._on(stream):
            self.pos.add_(1)

    def poll_error(self) -> int:
        for blk in self.blocks:
            rc = blk.poll_error()
            if rc:
                return rc
        return 0
