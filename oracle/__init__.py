"""CPU oracle for the Llama-3-style pre-norm decoder block.

TEST INFRASTRUCTURE ONLY.  Nothing in the product package
(``dense_decoder_block_gb300``) imports, links or runs anything here; only
``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` do.  The oracle shares no code with the CUDA path.

Modules
  bf16    round-to-nearest-even to bfloat16, emulated in float64/float32.
  shapes  parameter, d_ff and FLOP counting from a model config.
  block   the block itself: RMSNorm, Q/K/V projections, RoPE, causal GQA
          attention over a KV cache, O projection, residual adds, SwiGLU FFN;
          plus the 32-layer stack head (embedding, final norm, LM head,
          greedy choice).

Every function cites the passage of the pages it follows, by page title and
section.  The pages are:
  [70B]   "Llama 3.1 70B" (ainfra.dev LLM architecture diagram)
  [Block] "Inside a Transformer Block: FFN, the Residual Stream, and Normalization"
  [Next]  "How Llama 3.1 Generates the Next Token"
  [QKV]   "Llama 3 8B · Prepare Q, K, V" (decode mode, P = 1,000)
"""
from . import bf16, shapes, block  # noqa: F401
