// Host-side interfaces between the library's translation units (not public ABI).
#pragma once
#include <string>

#include "common.cuh"

namespace llama {

enum EpiKind : int {
    EPI_QKV = 0,     // RoPE on q/k tiles, q -> workspace, k/v -> cache rows
    EPI_RESID = 1,   // y = bf16(resid + bf16(acc))
    EPI_SWIGLU = 2,  // y = bf16(bf16(silu(bf16(gate))) * bf16(up)), two accumulators
    EPI_PLAIN = 3,   // y = bf16(acc)
    EPI_LOGITS = 4,  // y_f32 = acc
};

// Everything the GEMM epilogue needs.  Device pointers.
struct GemmEpi {
    int kind = EPI_PLAIN;
    bf16* out = nullptr;          // [M, F] (QKV: q [M, n_heads*128])
    const bf16* resid = nullptr;  // [M, F]
    float* out_f32 = nullptr;     // [M, F]
    // QKV / RoPE / cache append
    bf16* kc = nullptr;
    bf16* vc = nullptr;
    int n_heads = 0, n_kv_heads = 0, kv_seq = 0;   // cache row stride = kv_seq * 128
    int tokens_per_seq = 1;                         // token n -> (n / T, n % T)
    int start_pos = 0;                              // position of token t = base + t
    const int* pos_dev = nullptr;                   // if set, base = *pos_dev
    const int* pos_seq = nullptr;                   // decode (T = 1): token n at position pos_seq[n]
    int max_pos = 0;                                // positions must be < max_pos
    const float* cos_tab = nullptr;                 // [max_pos, 64]
    const float* sin_tab = nullptr;
    bool rope_later = false;                        // QKV: store q, k unrotated (launch_rope_inplace follows)
    int* err = nullptr;
};

// One projection: Y[M, F] = X[M, K] . W^T with W given as up to three row
// blocks (wq / wk / wv) or as the gate/up pair (dual).
struct GemmProblem {
    int M = 0, F = 0, K = 0;
    int seg_kb = 0;              // k-blocks (64 elements) per K-segment; 0 = kSegK / 64
    const CUtensorMap* a_maps[3] = {nullptr, nullptr, nullptr};   // host copies, [rows, K] bf16
    int n_maps = 1;
    bool dual = false;           // a_maps[0] = gate, a_maps[1] = up, F = d_ff
    const bf16* x = nullptr;     // [M, K] bf16, row stride K
};

enum GemmPath : int { PATH_AUTO = 0, PATH_TOKEN_TILED = 1, PATH_WEIGHT_STREAM = 2 };

// Scratch for the weight-streaming path: fp32 segment results [seg][acc][M][F].
size_t gemm_partial_bytes(const GemmProblem& p, int path);
int pick_gemm_path(const GemmProblem& p, int path);
int gemm_num_segments(const GemmProblem& p);
// True when the projection leaves segment results for a reduction kernel
// (weight-streaming schedule with more than one K-segment, or the token-tiled
// schedule in split mode).
bool gemm_needs_reduce(const GemmProblem& p, int path);
// True when a token-tiled projection runs its K-segments on separate CTAs (few
// tokens: its whole tiles would leave most SMs idle).
bool gemm_tt_split(const GemmProblem& p, int path);
// K-segment length (in 64-element k-blocks) for a projection of n_tiles feature
// tiles and total_kb k-blocks: the fewest segments whose units fill 70-100% of
// the n_sm SMs in one wave; failing that, the one that minimises the
// weight-streaming makespan, at least 8 k-blocks per segment.
int choose_seg_kb(int n_tiles, int total_kb, int n_sm);
// SMs of the current device (looked up once per device).
int device_sm_count();
// Runs setup(kern) once per (kernel, device) -- function attributes such as the
// dynamic shared-memory limit apply to the device that was current when they were
// set -- under a process-wide lock, so concurrent first calls do not race.  A
// failed setup is not recorded and runs again on the next call.
cudaError_t kernel_setup_once(const void* kern, cudaError_t (*setup)(const void* kern));
// Setup of a row-wise kernel that uses little or no shared memory: prefer the
// largest shared-memory carveout, so that an SM running its CTAs can take the CTAs
// of the projection or attention launched behind it without reconfiguring.
cudaError_t setup_prefer_shared(const void* kern);

cudaError_t launch_gemm(const GemmProblem& p, const GemmEpi& e, int path, float* partial, cudaStream_t s);

// Segment reductions (decode): add each output's segments in ascending order and
// apply the projection's epilogue (kind = EPI_QKV, EPI_RESID or EPI_SWIGLU).
struct ReduceArgs {
    const float* partial = nullptr;
    int n_segs = 0, M = 0, F = 0;
    GemmEpi e;
};
cudaError_t launch_reduce(const ReduceArgs& r, int kind, cudaStream_t s);
// Residual epilogue followed by RMSNorm of each row (d = F), writing h (e.out) and hn.
bool reduce_resid_norm_supported(int d);
cudaError_t launch_reduce_resid_norm(const ReduceArgs& r, const void* gain, void* hn, float eps, cudaStream_t s);

// Whole-K dot products per CTA (no segment split), weight-streaming, M <= 32.
// For outputs that have no token-tiled counterpart (the LM head logits).
cudaError_t launch_gemm_single_segment(const GemmProblem& p, const GemmEpi& e, cudaStream_t s);

// 2-D bf16 TMA descriptor, 128-byte swizzle, box = [box_rows, 64].
bool make_tmap_bf16(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                    std::string* why);

// ---------------------------------------------------------------- other kernels
cudaError_t launch_rmsnorm(const void* x, const void* g, void* y, int rows, int d, float eps, int dtype,
                           cudaStream_t s);

// Attention (SIMT).  q, o [M, Hq*dh]; caches [Bc, Hkv, kv_seq, dh].
struct AttnArgs {
    const void* q = nullptr;
    void* o = nullptr;
    const void* kc = nullptr;
    const void* vc = nullptr;
    int batch = 0, tokens = 0;          // M = batch * tokens
    int n_heads = 0, n_kv_heads = 0, head_dim = 0, kv_seq = 0;
    int start_pos = 0;
    const int* pos_dev = nullptr;
    const int* pos_seq = nullptr;       // decode: sequence b at position pos_seq[b] (device)
    int max_pos = 0;
    int dtype = LLAMA_BF16;
    float* partial = nullptr;           // decode: [B, Hkv, n_chunks, n_rep, head_dim + 4]
    int n_chunks = 0;                   // decode: chunk slots per (b, kv head)
    int* err = nullptr;
};
size_t attn_decode_partial_bytes(int batch, int n_kv_heads, int n_chunks, int n_rep, int head_dim);
cudaError_t launch_attention_prefill(const AttnArgs& a, cudaStream_t s);   // CUDA cores
cudaError_t launch_attention_decode(const AttnArgs& a, cudaStream_t s);    // CUDA cores, + combine
// Ascending fold of the decode chunk partials into o (shared by both decode kernels).
cudaError_t launch_attention_combine(const AttnArgs& a, cudaStream_t s);
// Tensor-core attention (bf16, head_dim 128, n_heads / n_kv_heads dividing 128).
bool attention_tc_supported(int n_heads, int n_kv_heads, int head_dim);
cudaError_t launch_attention_tc_prefill(const AttnArgs& a, cudaStream_t s);
cudaError_t launch_attention_tc_decode(const AttnArgs& a, int chunks_per_cta, cudaStream_t s);

// RoPE in place on the bf16 q rows [M, n_heads * 128] and on the cache rows of
// the M tokens (token n = (b, t) at position base + t, base = *pos_dev or
// start_pos): what the QKV epilogue does when it stores q and k unrotated.
cudaError_t launch_rope_inplace(void* q, void* kc, int M, int T, int n_heads, int n_kv_heads, int kv_seq,
                                int start_pos, const int* pos_dev, int max_pos, const float* cos_tab,
                                const float* sin_tab, int* err, cudaStream_t s);

// fp32 SIMT block pieces
cudaError_t launch_linear_f32(const float* x, const float* w, const float* w2, const float* resid, float* y, int M,
                              int F, int K, int mode, cudaStream_t s);   // mode 0 plain, 1 resid, 2 swiglu
cudaError_t launch_rope_append_f32(const float* qkv_q, const float* qkv_k, const float* qkv_v, float* q_out,
                                   float* kc, float* vc, int M, int T, int n_heads, int n_kv_heads, int head_dim,
                                   int kv_seq, int start_pos, const int* pos_dev, int max_pos,
                                   const float* cos_tab, const float* sin_tab, int* err, cudaStream_t s);

// stack head
cudaError_t launch_embed(const int32_t* ids, int n, const void* w, int vocab, int d, void* x, int32_t* err,
                         cudaStream_t s);
// ids[r] = argmax of logits row r, or *err when err is set and nonzero.
// Per-CTA timeline: the control word of each translation unit with traced kernels.
cudaError_t trace_set_norm(const TraceCtl& c);
cudaError_t trace_set_gemm_ws(const TraceCtl& c);
cudaError_t trace_set_gemm_tt(const TraceCtl& c);
cudaError_t trace_set_reduce(const TraceCtl& c);
cudaError_t trace_set_attn_tc(const TraceCtl& c);
cudaError_t trace_set_attn_simt(const TraceCtl& c);

// Failure-path self-test: a bounded wait that nothing satisfies (records LLAMA_ERR_DEVICE_TIMEOUT in *err).
cudaError_t launch_expire_wait(int* err, unsigned long long budget_ns, cudaStream_t s);
cudaError_t launch_argmax_rows(const float* logits, int rows, int vocab, int32_t* ids, const int* err,
                               cudaStream_t s);

// Next-token sampling: one CTA per row of fp32 logits [batch, vocab].
cudaError_t launch_sample(const float* logits, int batch, int vocab, float temperature, int top_k, float top_p,
                          const float* uniforms, int32_t* ids, cudaStream_t s);

}  // namespace llama
