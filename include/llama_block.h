/*
 * llama_block.h — C ABI of the GB300 (sm_103a) Llama-3-style decoder block library.
 *
 * One pre-norm decoder block, forward pass only, in causal prefill and in
 * KV-cached decode:
 *
 *     h = x + Attn(RMSNorm_1(x))          y = h + SwiGLU_FFN(RMSNorm_2(h))
 *
 * as defined by "Llama 3.1 70B" (ainfra.dev LLM architecture diagram:
 * Transformer layer, RMSNorm, Grouped-Query Attention, Residual add, SwiGLU
 * MLP), "How Llama 3.1 Generates the Next Token" (The transformer blocks,
 * What's RMSNorm?, What's the SWIGLU block?, RoPE) and "Llama 3 8B · Prepare
 * Q, K, V" (decode mode: Q/K/V projections, RoPE, K and V cached at KV-head
 * size).
 *
 * Conventions shared by every entry point
 *   - All pointers to tensors are DEVICE pointers owned by the caller; the
 *     library never frees them.  Weights are borrowed by the handle and must
 *     outlive it.  Nothing is copied.
 *   - Matrices are row-major [out, in] (torch.nn.Linear's storage: y = x W^T).
 *   - Activations are row-major [B, T, d_model].  The KV cache is two
 *     buffers K, V of shape [batch, n_kv_heads, max_seq, head_dim].
 *   - Element type is bf16 (LLAMA_BF16) or fp32 (LLAMA_F32) throughout one
 *     handle; token ids are int32.
 *   - Device pointers must be 16-byte aligned; every row length in bytes must
 *     be a multiple of 16.
 *   - Work is enqueued on the caller's stream (a cudaStream_t passed as
 *     void*; NULL = legacy default stream).  No host synchronisation, no
 *     device allocation and no device-wide barrier happens inside
 *     prefill/decode, so they may be captured into a CUDA graph.
 *   - Every function returns LLAMA_OK (0) or a negative LLAMA_ERR_* code;
 *     nothing throws across the ABI.  llama_block_last_error() returns a
 *     message for the last failure on that handle.
 */
#ifndef LLAMA_BLOCK_H_
#define LLAMA_BLOCK_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define LLAMA_OK 0
#define LLAMA_ERR_INVALID_ARG (-1)      /* null / misaligned pointer, bad size */
#define LLAMA_ERR_UNSUPPORTED_DIMS (-2) /* dims outside what the kernels implement */
#define LLAMA_ERR_POS_RANGE (-3)        /* position outside [0, max_seq) */
#define LLAMA_ERR_WORKSPACE (-4)        /* workspace missing or too small */
#define LLAMA_ERR_CUDA (-5)             /* a CUDA runtime call failed */
#define LLAMA_ERR_DEVICE_TIMEOUT (-6)   /* a bounded device-side wait expired */

typedef enum { LLAMA_F32 = 0, LLAMA_BF16 = 1 } llama_dtype;

/* Block shape.  n_heads query heads share n_kv_heads K/V heads in groups of
 * n_heads / n_kv_heads ("Llama 3.1 70B", Grouped-Query Attention).  eps sits
 * inside the square root of RMSNorm; rope_theta is the RoPE base (omega_i =
 * theta^(-2i/head_dim), "How Llama 3.1 Generates the Next Token", Why use
 * different rotation speeds?).  max_seq bounds positions and sizes the
 * cos/sin table built at create.
 * bf16 handles need head_dim == 128 and d_model, d_ff multiples of 128;
 * fp32 handles accept head_dim in {32, 64, 128} and d_model, d_ff multiples
 * of 4. */
typedef struct {
    int32_t d_model, n_heads, n_kv_heads, head_dim, d_ff, max_seq;
    float eps, rope_theta;
    int32_t dtype; /* llama_dtype */
} llama_block_dims;

/* Device pointers, element type = dims.dtype.
 *   g_attn, g_ffn   [d_model]                 RMSNorm gains
 *   wq              [n_heads*head_dim, d]     wk, wv [n_kv_heads*head_dim, d]
 *   wo              [d, n_heads*head_dim]
 *   w_gate, w_up    [d_ff, d]                 w_down [d, d_ff]
 * ("How Llama 3.1 Generates the Next Token", Weight dimensions, transposed to
 * [out, in] as in "Llama 3 8B · Prepare Q, K, V", layers.py excerpt.) */
typedef struct {
    const void *g_attn, *wq, *wk, *wv, *wo, *g_ffn, *w_gate, *w_up, *w_down;
} llama_block_weights;

/* K and V rows are stored after RoPE (K) at KV-head size ("Llama 3 8B ·
 * Prepare Q, K, V", Explanation).  batch and max_seq describe the buffers;
 * max_seq may differ from the handle's but positions must fit both. */
typedef struct {
    void *k, *v;
    int32_t batch, max_seq;
} llama_kv_cache;

typedef struct llama_block_s* llama_block;

/* Validate dims, borrow weight pointers, build the TMA descriptors over the
 * weights and upload the fp32 cos/sin table [max_seq, head_dim/2] (computed
 * in fp64 on the host).  This is the only call that allocates device memory
 * (the table and a 4-byte error word).  On success *out holds the handle. */
int llama_block_create(const llama_block_dims* dims, const llama_block_weights* w, llama_block* out);

/* Llama 3.1's long-context RoPE schedule ("How Llama 3.1 Generates the Next
 * Token", Why use different rotation speeds?: the fastest rotations unchanged,
 * the slowest slowed by a factor, a middle range blended; "Llama 3.1 70B",
 * highlights: llama3 x8).  Pair i turns omega_i = rope_theta^(-2i/head_dim)
 * radians per position in the base schedule; with wavelength 2 pi / omega_i:
 *   wavelength < original_max_pos / high_freq_factor  ->  omega_i (unchanged)
 *   wavelength > original_max_pos / low_freq_factor   ->  omega_i / factor
 *   otherwise  (1 - s) omega_i / factor + s omega_i,
 *              s = (original_max_pos / wavelength - low_freq_factor)
 *                  / (high_freq_factor - low_freq_factor).
 * The pages give the factor (8) but not the band edges; Llama 3.1's released
 * configuration is factor 8, low 1, high 4, original_max_pos 8192.  Requires
 * factor >= 1, 0 < low_freq_factor < high_freq_factor, original_max_pos > 0. */
typedef struct {
    float factor, low_freq_factor, high_freq_factor;
    int32_t original_max_pos;
} llama_rope_scaling;

/* llama_block_create with the long-context RoPE schedule above in the handle's
 * cos/sin table (scaling = NULL: the base schedule, same as
 * llama_block_create).  Only the table differs; every call on the handle then
 * rotates q and k with the scaled angles.  LLAMA_ERR_INVALID_ARG for scaling
 * values outside the ranges above. */
int llama_block_create_scaled(const llama_block_dims* dims, const llama_block_weights* w,
                              const llama_rope_scaling* scaling, llama_block* out);

/* Free the handle's table, error word and host state.  NULL is a no-op. */
void llama_block_destroy(llama_block blk);

/* Bytes of device workspace that prefill (tokens = T) or decode (tokens = 1)
 * needs for batch B.  Returns 0 for invalid arguments. */
size_t llama_block_workspace_bytes(llama_block blk, int batch, int tokens);

/* Where a call's intermediates sit in its workspace, for inspection after the
 * call (stage-by-stage checks, callers that reuse a stage's output).  For a
 * call with this batch and tokens (tokens = 1: decode), offsets[i] receives the
 * byte offset from the workspace start of
 *   [0] xn  = RMSNorm_1(x)                    [batch*tokens, d_model]
 *   [1] q   after RoPE                        [batch*tokens, n_heads*head_dim]
 *   [2] o   attention output, heads merged    [batch*tokens, n_heads*head_dim]
 *   [3] h   = x + o Wo^T                      [batch*tokens, d_model]
 *   [4] hn  = RMSNorm_2(h)                    [batch*tokens, d_model]
 *   [5] u   = SiLU(hn W_gate^T) * (hn W_up^T) [batch*tokens, d_ff]
 * row-major, element type dims.dtype ("Llama 3.1 70B", Transformer layer: the
 * steps of the block in order).  n must be at least LLAMA_BLOCK_INTERMEDIATES.
 * Returns LLAMA_BLOCK_INTERMEDIATES, or LLAMA_ERR_INVALID_ARG. */
#define LLAMA_BLOCK_INTERMEDIATES 6
int llama_block_workspace_offsets(llama_block blk, int batch, int tokens, size_t* offsets, int n);

/* Causal prefill of T tokens per sequence at positions 0..T-1.
 *   x  [batch, T, d]   input residual stream
 *   y  [batch, T, d]   output; may alias x
 *   kv cache rows 0..T-1 of sequences 0..batch-1 are overwritten with the
 *      rotated keys and the values.
 * Attention follows "Llama 3.1 70B", Grouped-Query Attention (scaled dot
 * product, causal, 1/sqrt(head_dim)); the query at position p sees keys 0..p. */
int llama_block_prefill(llama_block blk, const void* x, int batch, int tokens, const llama_kv_cache* kv, void* y,
                        void* workspace, size_t workspace_bytes, void* stream);

/* Prefill of `tokens` new tokens per sequence at positions start_pos ..
 * start_pos + tokens - 1 on a cache that already holds the earlier tokens
 * (prefill in chunks).  kv rows 0 .. start_pos - 1 must hold their keys and
 * values; rows start_pos .. start_pos + tokens - 1 are written; the query at
 * position p sees keys 0..p.  llama_block_prefill is this call with
 * start_pos = 0.  Each row equals, bit for bit, the same row of one prefill of
 * all start_pos + tokens tokens.  start_pos + tokens must not exceed max_seq
 * (LLAMA_ERR_POS_RANGE otherwise). */
int llama_block_prefill_at(llama_block blk, const void* x, int batch, int tokens, int start_pos,
                           const llama_kv_cache* kv, void* y, void* workspace, size_t workspace_bytes, void* stream);

/* One decode step at position pos for every sequence of the batch.
 *   x [batch, 1, d] in, y [batch, 1, d] out (may alias x).
 *   kv rows 0..pos-1 must hold the cached keys/values; row pos is written;
 *   attention reads keys 0..pos (L = pos + 1, "Llama 3 8B · Prepare Q, K, V",
 *   decode mode) and nothing beyond.
 * The result for position pos is bit-identical to row pos of a prefill of
 * the same tokens (both paths share one reduction schedule). */
int llama_block_decode(llama_block blk, const void* x, int batch, const llama_kv_cache* kv, int pos, void* y,
                       void* workspace, size_t workspace_bytes, void* stream);

/* Same as llama_block_decode with the position read on the device from
 * *pos_dev (int32) when the kernels run, so one captured CUDA graph can be
 * replayed for successive positions.  The value must lie in [0, max_seq);
 * a value outside that range makes the kernels record LLAMA_ERR_POS_RANGE in
 * the handle's error word (read it with llama_block_poll_error); no cache row
 * is written and y is left undefined. */
int llama_block_decode_devpos(llama_block blk, const void* x, int batch, const llama_kv_cache* kv,
                              const int32_t* pos_dev, void* y, void* workspace, size_t workspace_bytes,
                              void* stream);

/* One decode step with a position per sequence: sequence b sits at position
 * pos_seq[b] (int32, device memory, read by the kernels when they run, so a
 * captured graph can be replayed as the positions move).  Sequence b reads its
 * cache rows 0..pos_seq[b] and writes row pos_seq[b]; its result equals, bit for
 * bit, what llama_block_decode at that position gives for it.  Each value must lie
 * in [0, max_seq): otherwise the kernels record LLAMA_ERR_POS_RANGE in the error
 * word, write no cache row and leave y undefined.  Supported for bf16 handles
 * with at most 8 query heads per KV head and batch <= 32; otherwise
 * LLAMA_ERR_UNSUPPORTED_DIMS. */
int llama_block_decode_seqpos(llama_block blk, const void* x, int batch, const llama_kv_cache* kv,
                              const int32_t* pos_seq, void* y, void* workspace, size_t workspace_bytes,
                              void* stream);

/* Synchronise `stream`, read and clear the handle's device error word.
 * Returns LLAMA_OK or the code a kernel recorded (LLAMA_ERR_DEVICE_TIMEOUT,
 * LLAMA_ERR_POS_RANGE). */
int llama_block_poll_error(llama_block blk, void* stream);

/* Per-CTA timeline of the block's kernels (RMSNorm, the projections, their
 * reductions, RoPE, attention and its combine), in the trace build of the
 * library (libllama_block_trace.so, the same sources compiled with
 * LLAMA_TRACE); the product library returns LLAMA_ERR_UNSUPPORTED_DIMS from
 * llama_trace_begin and carries no tracing code in its kernels.  Between
 * llama_trace_begin and llama_trace_end every CTA of those kernels claims one
 * record with an atomic
 * increment of *count and, while the index is below `capacity`, writes four
 * uint64 words at records[4 * index]:
 *   [0] kernel id (bits 0..7: 1 RMSNorm, 2 weight-streaming projection, 3
 *       token-tiled projection, 4..7 the QKV / residual / SwiGLU / residual +
 *       RMSNorm reductions, 8 decode attention, 9 its combine, 10 prefill
 *       attention, 11 RoPE, 12 wide-group decode attention; bits 8..11 the
 *       projection's epilogue: 0 QKV, 1 residual, 2 SwiGLU, 4 logits; bit 12
 *       a token-tiled projection whose K-segments run on separate CTAs),
 *       bits 16..31 the SM, bits 32..63 the CTA's linear index;
 *   [1] %globaltimer (ns) when the CTA started;
 *   [2] when its grid-dependency wait returned (0 if that CTA's recording
 *       thread does not wait);
 *   [3] when the CTA's thread 0 finished.
 * records (capacity x 32 bytes) and count (zeroed by the caller) are device
 * memory owned by the caller and must stay valid until llama_trace_end.  The
 * setting is process-wide and applies to kernels that run after the call
 * (graph replays included); with it on, each CTA reads it from the constant
 * bank at its start (a traced step runs about 3 us longer).  Returns LLAMA_OK,
 * LLAMA_ERR_INVALID_ARG, LLAMA_ERR_CUDA or (product build)
 * LLAMA_ERR_UNSUPPORTED_DIMS. */
int llama_trace_begin(unsigned long long* records, unsigned int* count, unsigned int capacity);
int llama_trace_end(void);

/* Failure-path self-test.  Launches on `stream` one warp that waits, through the
 * same bounded mbarrier wait every tensor-core kernel of the library uses, on a
 * barrier nothing arrives on.  After budget_ns nanoseconds (0 or more than 2 s:
 * the kernels' own 2 s budget) the wait gives up, records
 * LLAMA_ERR_DEVICE_TIMEOUT in the handle's error word and the kernel returns:
 * llama_block_poll_error then reports it, and the handle and the CUDA context stay
 * usable.  Returns LLAMA_OK once the launch is queued. */
int llama_block_selftest_wait_timeout(llama_block blk, unsigned long long budget_ns, void* stream);

/* Message of the last failure on this handle ("" if none).  Valid until the
 * next call on the handle. */
const char* llama_block_last_error(llama_block blk);

/* Stage timing.  events = NULL disables it; otherwise an array of 8 cudaEvent_t
 * (passed as void*) that every later prefill/decode on this handle records on
 * its stream: events[i] before stage i and events[7] after the last, for the
 * stages RMSNorm_1, QKV+RoPE+append, attention, O+residual, RMSNorm_2,
 * gate/up+SwiGLU, down+residual.  The array is borrowed until disabled. */
#define LLAMA_BLOCK_STAGES 7
int llama_block_set_stage_events(llama_block blk, void* const* events, int n_events);

/* Number of kernels the last successful prefill/decode call on this handle
 * enqueued (0 before the first call, after a failed call, or for NULL).  It
 * depends on the shape (the K-segment schedule fixed at create decides which
 * projections need a reduction kernel) and on the call (decode or prefill). */
int llama_block_launch_count(llama_block blk);

/* Device address of pinned host memory (cudaHostAlloc / cudaHostRegister; with
 * unified addressing every such allocation is mapped).  x and y of prefill and
 * decode may be given this way: the kernels then read x from and write y to host
 * memory directly (over NVLink-C2C on a Grace host), with no copy calls around
 * the block.  Only x and y take host memory: weights, the cache and the
 * workspace are read by TMA and must be device memory.  *dev = NULL and
 * LLAMA_ERR_INVALID_ARG if `host` is not pinned and mapped. */
int llama_device_ptr_of_host(const void* host, void** dev);

/* ---------------------------------------------------------------------------
 * Stack head (32-layer generation loop): embedding gather, final RMSNorm,
 * LM head with greedy choice.  bf16 only.
 * ------------------------------------------------------------------------- */

/* x[n, :] = w_embed[ids[n], :] for n < n_tokens ("Llama 3.1 70B", Token
 * embedding: a row gather, no positional term).  ids int32 in [0, vocab);
 * an id outside that range writes a zero row and records
 * LLAMA_ERR_INVALID_ARG in *err_dev (may be NULL). */
int llama_embed(const int32_t* ids, int n_tokens, const void* w_embed, int vocab, int d_model, void* x,
                int32_t* err_dev, void* stream);

/* ids[b] = argmax_v (RMSNorm_final(h[b]) . w_out[v]), fp32 logits, ties to the
 * lowest index ("How Llama 3.1 Generates the Next Token", Unembedding and
 * Sampling: greedy choice).  h [batch, d_model] (stride h_stride elements
 * between rows), g_final [d_model], w_out [vocab, d_model].  logits, if not
 * NULL, receives [batch, vocab] fp32.  workspace: llama_lmhead_workspace_bytes
 * (it also holds the call's device error word).  Every wait inside the kernels
 * is bounded; if one expires, ids[b] receives LLAMA_ERR_DEVICE_TIMEOUT (a
 * negative value, never a token id) for every row and the logits are undefined. */
size_t llama_lmhead_workspace_bytes(int batch, int d_model, int vocab);
int llama_lmhead_argmax(const void* h, int batch, int h_stride, const void* g_final, const void* w_out, int vocab,
                        int d_model, float eps, int32_t* ids, float* logits, void* workspace,
                        size_t workspace_bytes, void* stream);

/* Same result as llama_lmhead_argmax, for callers that cannot allocate device
 * memory (no workspace to pass: code running where cudaMalloc is not allowed or
 * must not happen on the hot path).  There is no counterpart on the pages; it is
 * a deployment variant.  The normalised rows live in a library-owned device
 * array of 32 x 8192 bf16 (512 KiB), held by every GPU that loads the library
 * until the process exits; batch > 32 or d_model > 8192 returns
 * LLAMA_ERR_WORKSPACE.  logits [batch, vocab] fp32 is required (it is an
 * output).  Nothing is allocated.  The first call on a device looks up the
 * array's device address (with that device current) and caches it: make that
 * first call before any stream capture.  Every call shares the one array, which
 * keeps the last call's rows; calls that overlap on the GPU (other streams,
 * other threads) race on it.  The cached address belongs to the device's
 * context: after cudaDeviceReset (or a reset of the primary context) the
 * library must be reloaded before this call is used again.  A device wait that
 * expires is reported as in llama_lmhead_argmax: ids[b] =
 * LLAMA_ERR_DEVICE_TIMEOUT (the error word is a second library-owned device
 * int, cleared by every call). */
int llama_lmhead_argmax_noalloc(const void* h, int batch, int h_stride, const void* g_final, const void* w_out,
                                int vocab, int d_model, float eps, int32_t* ids, float* logits, void* stream);

/* Next-token sampling from fp32 logits [batch, vocab] ("How Llama 3.1
 * Generates the Next Token", Temperature, Softmax, Top-k and top-p sampling):
 * divide by the temperature, softmax over the whole vocabulary, keep the top_k
 * most probable tokens and the smallest set of most probable tokens whose
 * probability reaches top_p (both restrictions: the smaller set), renormalise,
 * and draw: with the kept tokens in order of decreasing logit (equal logits by
 * increasing index), ids[b] is the first token whose cumulative renormalised
 * probability exceeds uniforms[b] (device fp32 in [0, 1), one per row, supplied
 * by the caller; values outside are clamped).  temperature = 0 or top_k = 1
 * gives the greedy choice (first maximum); top_k = 0 means no top-k limit and
 * top_p = 1 no top-p limit.  Weights e^{(z - max)/T} are computed in fp32 and
 * summed exactly in 2^-40 fixed point, top_p and the uniforms are taken to 24
 * bits: the result does not depend on thread scheduling.  Logits must be finite
 * (-inf allowed, weight zero).  Requires temperature >= 0, top_k >= 0,
 * 0 < top_p <= 1, 1 <= vocab <= 2^20, batch <= 65535; otherwise
 * LLAMA_ERR_INVALID_ARG.  No workspace, nothing allocated. */
int llama_sample(const float* logits, int batch, int vocab, float temperature, int top_k, float top_p,
                 const float* uniforms, int32_t* ids, void* stream);

/* ---------------------------------------------------------------------------
 * Step-level entry points (the block's individual steps, for unit tests and
 * for callers that compose their own schedule).  Same conventions as above.
 * ------------------------------------------------------------------------- */

/* y = bf16(bf16(x * r) * g), r = 1/sqrt(mean(x^2) + eps) per row
 * ("Llama 3.1 70B", RMSNorm reference implementation).  rows x d. */
int llama_rmsnorm(const void* x, const void* g, void* y, int rows, int d, float eps, int dtype, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* LLAMA_BLOCK_H_ */
