// The C ABI: handle management, argument validation, workspace layout and the
// per-call schedule of kernels for prefill and decode.
#include <cmath>
#include <cstdio>
#include <cstring>
#include <new>
#include <string>
#include <vector>

#include "internal.h"

using namespace llama;

struct llama_block_s {
    llama_block_dims dims{};
    llama_block_weights w{};
    CUtensorMap m_wq, m_wk, m_wv, m_wo, m_wg, m_wu, m_wd;
    float* cos_tab = nullptr;   // [max_seq, 64]
    float* sin_tab = nullptr;
    int* err_dev = nullptr;
    int last_launches = 0;      // kernels enqueued by the last prefill/decode call
    int device = 0;
    std::string last_error;
    cudaEvent_t stage_events[LLAMA_BLOCK_STAGES + 1] = {};
    bool timing = false;
    // K-segment length (64-element k-blocks) of each projection: QKV, O, gate/up, down.
    // Fixed at create and shared by prefill and decode (it is part of the arithmetic).
    int seg_kb[4] = {0, 0, 0, 0};
};

namespace {

constexpr size_t kAlign = 1024;

size_t align_up(size_t v) { return (v + kAlign - 1) & ~(kAlign - 1); }
bool aligned16(const void* p) { return ((uintptr_t)p & 15) == 0; }

int fail(llama_block b, int code, const std::string& msg) {
    if (b) b->last_error = msg;
    return code;
}

int cuda_fail(llama_block b, cudaError_t e, const char* where) {
    return fail(b, LLAMA_ERR_CUDA, std::string(where) + ": " + cudaGetErrorString(e));
}

// Workspace carve-up for one call.
struct Ws {
    void* xn = nullptr;
    void* q = nullptr;
    void* o = nullptr;
    void* h = nullptr;
    void* hn = nullptr;
    void* u = nullptr;
    void* k_raw = nullptr;   // fp32 path only
    void* v_raw = nullptr;
    void* q_raw = nullptr;
    float* gemm_partial = nullptr;
    float* attn_partial = nullptr;
    size_t total = 0;
};

int attn_chunk_slots(const llama_block_dims& d) { return (d.max_seq + kAttnChunk - 1) / kAttnChunk; }

GemmProblem problem_qkv(const llama_block_s* b, int M, const void* x) {
    GemmProblem p;
    p.M = M;
    p.F = (b->dims.n_heads + 2 * b->dims.n_kv_heads) * b->dims.head_dim;
    p.K = b->dims.d_model;
    p.a_maps[0] = &b->m_wq;
    p.a_maps[1] = &b->m_wk;
    p.a_maps[2] = &b->m_wv;
    p.n_maps = 3;
    p.seg_kb = b->seg_kb[0];
    p.x = (const bf16*)x;
    return p;
}
GemmProblem problem_o(const llama_block_s* b, int M, const void* x) {
    GemmProblem p;
    p.M = M;
    p.F = b->dims.d_model;
    p.K = b->dims.n_heads * b->dims.head_dim;
    p.a_maps[0] = &b->m_wo;
    p.seg_kb = b->seg_kb[1];
    p.x = (const bf16*)x;
    return p;
}
GemmProblem problem_gateup(const llama_block_s* b, int M, const void* x) {
    GemmProblem p;
    p.M = M;
    p.F = b->dims.d_ff;
    p.K = b->dims.d_model;
    p.a_maps[0] = &b->m_wg;
    p.a_maps[1] = &b->m_wu;
    p.n_maps = 2;
    p.dual = true;
    p.seg_kb = b->seg_kb[2];
    p.x = (const bf16*)x;
    return p;
}
GemmProblem problem_down(const llama_block_s* b, int M, const void* x) {
    GemmProblem p;
    p.M = M;
    p.F = b->dims.d_model;
    p.K = b->dims.d_ff;
    p.a_maps[0] = &b->m_wd;
    p.seg_kb = b->seg_kb[3];
    p.x = (const bf16*)x;
    return p;
}

Ws layout(const llama_block_s* b, int B, int T, uint8_t* base, bool decode) {
    const auto& d = b->dims;
    const size_t M = (size_t)B * T;
    const size_t es = d.dtype == LLAMA_BF16 ? 2 : 4;
    const size_t qd = (size_t)d.n_heads * d.head_dim, kvd = (size_t)d.n_kv_heads * d.head_dim;
    Ws w;
    size_t off = 0;
    auto take = [&](size_t bytes) -> void* {
        void* p = base ? base + off : nullptr;
        off += align_up(bytes);
        return p;
    };
    w.xn = take(M * d.d_model * es);
    w.q = take(M * qd * es);
    w.o = take(M * qd * es);
    w.h = take(M * d.d_model * es);
    w.hn = take(M * d.d_model * es);
    w.u = take(M * d.d_ff * es);
    if (d.dtype == LLAMA_F32) {
        w.q_raw = take(M * qd * es);
        w.k_raw = take(M * kvd * es);
        w.v_raw = take(M * kvd * es);
    } else {
        size_t part = 0;
        const GemmProblem ps[4] = {problem_qkv(b, (int)M, nullptr), problem_o(b, (int)M, nullptr),
                                   problem_gateup(b, (int)M, nullptr), problem_down(b, (int)M, nullptr)};
        for (const auto& p : ps) part = std::max(part, gemm_partial_bytes(p, PATH_AUTO));
        w.gemm_partial = (float*)take(part);
    }
    if (decode) {
        const int n_rep = d.n_heads / d.n_kv_heads;
        w.attn_partial = (float*)take(attn_decode_partial_bytes(B, d.n_kv_heads, attn_chunk_slots(d), n_rep,
                                                                d.head_dim));
    }
    w.total = off;
    return w;
}

int check_kv(llama_block b, const llama_kv_cache* kv, int batch, int last_pos) {
    if (!kv || !kv->k || !kv->v) return fail(b, LLAMA_ERR_INVALID_ARG, "kv cache pointers are null");
    if (!aligned16(kv->k) || !aligned16(kv->v)) return fail(b, LLAMA_ERR_INVALID_ARG, "kv cache not 16-byte aligned");
    if (kv->batch < batch) return fail(b, LLAMA_ERR_INVALID_ARG, "kv cache batch smaller than the call's batch");
    if (kv->max_seq <= 0) return fail(b, LLAMA_ERR_INVALID_ARG, "kv cache max_seq must be positive");
    if (last_pos >= kv->max_seq || last_pos >= b->dims.max_seq)
        return fail(b, LLAMA_ERR_POS_RANGE, "position beyond the cache or the handle's max_seq");
    return LLAMA_OK;
}

// The block's schedule, shared by prefill (T tokens at 0..T-1) and decode
// (T = 1 at `pos`, or at *pos_dev).
int run_block(llama_block b, const void* x, int B, int T, const llama_kv_cache* kv, int start_pos,
              const int32_t* pos_dev, void* y, void* ws, size_t ws_bytes, void* stream_v, bool decode,
              const int32_t* pos_seq = nullptr) {
    const auto& d = b->dims;
    cudaStream_t s = (cudaStream_t)stream_v;
    const int M = B * T;
    if (M == 0) return LLAMA_OK;
    Ws w = layout(b, B, T, nullptr, decode);
    if (!ws || ws_bytes < w.total)
        return fail(b, LLAMA_ERR_WORKSPACE, "workspace too small: need " + std::to_string(w.total) + " bytes");
    if (!aligned16(ws)) return fail(b, LLAMA_ERR_INVALID_ARG, "workspace not 16-byte aligned");
    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess) return fail(b, LLAMA_ERR_CUDA, "cudaGetDevice failed");
    if (cur != b->device) return fail(b, LLAMA_ERR_INVALID_ARG, "the handle's device is not the current device");
    w = layout(b, B, T, (uint8_t*)ws, decode);
    const int max_pos = std::min(d.max_seq, kv->max_seq);
    cudaError_t e;
    // kernels enqueued by this call (each launcher below issues one; decode attention two)
    int n_launch = 0;
    b->last_launches = 0;
#define LLAMA_TRY(call, where)                          \
    do {                                                \
        e = (call);                                     \
        if (e != cudaSuccess) return cuda_fail(b, e, where); \
        ++n_launch;                                     \
    } while (0)
    int stage = 0;
    cudaStreamCaptureStatus capturing = cudaStreamCaptureStatusNone;
    if (b->timing) cudaStreamIsCapturing(s, &capturing);
    auto mark = [&]() {
        // inside stream capture an external record becomes a timing event node of the graph
        if (b->timing && stage <= LLAMA_BLOCK_STAGES)
            cudaEventRecordWithFlags(b->stage_events[stage], s,
                                     capturing == cudaStreamCaptureStatusActive ? cudaEventRecordExternal : 0);
        ++stage;
    };

    AttnArgs at;
    at.q = w.q;
    at.o = w.o;
    at.kc = kv->k;
    at.vc = kv->v;
    at.batch = B;
    at.tokens = T;
    at.n_heads = d.n_heads;
    at.n_kv_heads = d.n_kv_heads;
    at.head_dim = d.head_dim;
    at.kv_seq = kv->max_seq;
    at.start_pos = start_pos;
    at.pos_dev = pos_dev;
    at.pos_seq = pos_seq;
    at.max_pos = max_pos;
    at.dtype = d.dtype;
    at.partial = w.attn_partial;
    at.n_chunks = attn_chunk_slots(d);
    at.err = b->err_dev;

    if (d.dtype == LLAMA_BF16) {
        // Projections with a weight-streaming schedule leave fp32 segment results that a
        // reduction kernel adds (ascending) before the same epilogue the token-tiled
        // schedule fuses.
        auto reduce = [&](const GemmProblem& p, const GemmEpi& ep, int kind) -> cudaError_t {
            ReduceArgs r;
            r.partial = w.gemm_partial;
            r.n_segs = gemm_num_segments(p);
            r.M = p.M;
            r.F = p.F;
            r.e = ep;
            return launch_reduce(r, kind, s);
        };
        // 1. RMSNorm_1
        mark();
        LLAMA_TRY(launch_rmsnorm(x, b->w.g_attn, w.xn, M, d.d_model, d.eps, d.dtype, s), "rmsnorm_1");
        // 2. QKV projection + RoPE + KV append
        mark();
        GemmEpi eq;
        eq.kind = EPI_QKV;
        eq.out = (bf16*)w.q;
        eq.kc = (bf16*)kv->k;
        eq.vc = (bf16*)kv->v;
        eq.n_heads = d.n_heads;
        eq.n_kv_heads = d.n_kv_heads;
        eq.kv_seq = kv->max_seq;
        eq.tokens_per_seq = T;
        eq.start_pos = start_pos;
        eq.pos_dev = pos_dev;
        eq.pos_seq = pos_seq;
        eq.max_pos = max_pos;
        eq.cos_tab = b->cos_tab;
        eq.sin_tab = b->sin_tab;
        eq.err = b->err_dev;
        const GemmProblem pq = problem_qkv(b, M, w.xn);
        // The token-tiled (prefill) QKV stores q and k unrotated and a vectorised
        // kernel rotates them in place: the per-column table loads of a fused RoPE
        // kept that projection's epilogue warps behind its MMAs.
        eq.rope_later = pick_gemm_path(pq, PATH_AUTO) == PATH_TOKEN_TILED && !gemm_tt_split(pq, PATH_AUTO);
        LLAMA_TRY(launch_gemm(pq, eq, PATH_AUTO, w.gemm_partial, s), "qkv");
        if (eq.rope_later)
            LLAMA_TRY(launch_rope_inplace(w.q, kv->k, M, T, d.n_heads, d.n_kv_heads, kv->max_seq, start_pos, pos_dev,
                                          max_pos, b->cos_tab, b->sin_tab, b->err_dev, s),
                      "qkv_rope");
        if (gemm_needs_reduce(pq, PATH_AUTO)) LLAMA_TRY(reduce(pq, eq, EPI_QKV), "qkv_reduce");
        // 3. attention (tensor cores when the group size divides 128; one choice per handle)
        mark();
        if (attention_tc_supported(d.n_heads, d.n_kv_heads, d.head_dim)) {
            if (decode) {
                LLAMA_TRY(launch_attention_tc_decode(at, 0, s), "attention_decode");
                ++n_launch;   // and its combine
            } else {
                LLAMA_TRY(launch_attention_tc_prefill(at, s), "attention_prefill");
            }
        } else {
            if (decode) {
                LLAMA_TRY(launch_attention_decode(at, s), "attention_decode");
                ++n_launch;   // and its combine
            } else {
                LLAMA_TRY(launch_attention_prefill(at, s), "attention_prefill");
            }
        }
        // 4. O projection + residual -> h, 5. RMSNorm_2 -> hn
        mark();
        GemmEpi eo;
        eo.kind = EPI_RESID;
        eo.out = (bf16*)w.h;
        eo.resid = (const bf16*)x;
        eo.err = b->err_dev;
        const GemmProblem po = problem_o(b, M, w.o);
        LLAMA_TRY(launch_gemm(po, eo, PATH_AUTO, w.gemm_partial, s), "o_proj");
        const bool o_red = gemm_needs_reduce(po, PATH_AUTO);
        if (o_red && reduce_resid_norm_supported(d.d_model)) {
            ReduceArgs r;
            r.partial = w.gemm_partial;
            r.n_segs = gemm_num_segments(po);
            r.M = po.M;
            r.F = po.F;
            r.e = eo;
            mark();
            LLAMA_TRY(launch_reduce_resid_norm(r, b->w.g_ffn, w.hn, d.eps, s), "o_reduce_rmsnorm_2");
        } else {
            if (o_red) LLAMA_TRY(reduce(po, eo, EPI_RESID), "o_reduce");
            mark();
            LLAMA_TRY(launch_rmsnorm(w.h, b->w.g_ffn, w.hn, M, d.d_model, d.eps, d.dtype, s), "rmsnorm_2");
        }
        // 6. gate/up + SwiGLU
        mark();
        GemmEpi eg;
        eg.kind = EPI_SWIGLU;
        eg.out = (bf16*)w.u;
        eg.err = b->err_dev;
        const GemmProblem pg = problem_gateup(b, M, w.hn);
        LLAMA_TRY(launch_gemm(pg, eg, PATH_AUTO, w.gemm_partial, s), "gate_up");
        if (gemm_needs_reduce(pg, PATH_AUTO)) LLAMA_TRY(reduce(pg, eg, EPI_SWIGLU), "gate_up_reduce");
        // 7. down + residual -> y
        mark();
        GemmEpi ed;
        ed.kind = EPI_RESID;
        ed.out = (bf16*)y;
        ed.resid = (const bf16*)w.h;
        ed.err = b->err_dev;
        const GemmProblem pd = problem_down(b, M, w.u);
        LLAMA_TRY(launch_gemm(pd, ed, PATH_AUTO, w.gemm_partial, s), "down");
        if (gemm_needs_reduce(pd, PATH_AUTO)) LLAMA_TRY(reduce(pd, ed, EPI_RESID), "down_reduce");
        mark();
    } else {
        const int qd = d.n_heads * d.head_dim, kvd = d.n_kv_heads * d.head_dim;
        const float* xf = (const float*)x;
        LLAMA_TRY(launch_rmsnorm(x, b->w.g_attn, w.xn, M, d.d_model, d.eps, d.dtype, s), "rmsnorm_1");
        LLAMA_TRY(launch_linear_f32((const float*)w.xn, (const float*)b->w.wq, nullptr, nullptr, (float*)w.q_raw, M,
                                    qd, d.d_model, 0, s),
                  "q_proj");
        LLAMA_TRY(launch_linear_f32((const float*)w.xn, (const float*)b->w.wk, nullptr, nullptr, (float*)w.k_raw, M,
                                    kvd, d.d_model, 0, s),
                  "k_proj");
        LLAMA_TRY(launch_linear_f32((const float*)w.xn, (const float*)b->w.wv, nullptr, nullptr, (float*)w.v_raw, M,
                                    kvd, d.d_model, 0, s),
                  "v_proj");
        LLAMA_TRY(launch_rope_append_f32((const float*)w.q_raw, (const float*)w.k_raw, (const float*)w.v_raw,
                                         (float*)w.q, (float*)kv->k, (float*)kv->v, M, T, d.n_heads, d.n_kv_heads,
                                         d.head_dim, kv->max_seq, start_pos, pos_dev, max_pos, b->cos_tab,
                                         b->sin_tab, b->err_dev, s),
                  "rope_append");
        if (decode) {
            LLAMA_TRY(launch_attention_decode(at, s), "attention_decode");
            ++n_launch;   // and its combine
        } else {
            LLAMA_TRY(launch_attention_prefill(at, s), "attention_prefill");
        }
        LLAMA_TRY(launch_linear_f32((const float*)w.o, (const float*)b->w.wo, nullptr, xf, (float*)w.h, M, d.d_model,
                                    qd, 1, s),
                  "o_proj");
        LLAMA_TRY(launch_rmsnorm(w.h, b->w.g_ffn, w.hn, M, d.d_model, d.eps, d.dtype, s), "rmsnorm_2");
        LLAMA_TRY(launch_linear_f32((const float*)w.hn, (const float*)b->w.w_gate, (const float*)b->w.w_up, nullptr,
                                    (float*)w.u, M, d.d_ff, d.d_model, 2, s),
                  "gate_up");
        LLAMA_TRY(launch_linear_f32((const float*)w.u, (const float*)b->w.w_down, nullptr, (const float*)w.h,
                                    (float*)y, M, d.d_model, d.d_ff, 1, s),
                  "down");
    }
#undef LLAMA_TRY
    b->last_launches = n_launch;
    return LLAMA_OK;
}

int validate_dims(const llama_block_dims* d, std::string* why) {
    if (!d) { *why = "dims is null"; return LLAMA_ERR_INVALID_ARG; }
    if (d->d_model <= 0 || d->n_heads <= 0 || d->n_kv_heads <= 0 || d->head_dim <= 0 || d->d_ff <= 0 ||
        d->max_seq <= 0) {
        *why = "dims must be positive";
        return LLAMA_ERR_INVALID_ARG;
    }
    if (!(d->eps >= 0.f) || !(d->rope_theta > 0.f)) {
        *why = "eps must be >= 0 and rope_theta > 0";
        return LLAMA_ERR_INVALID_ARG;
    }
    if (d->n_heads % d->n_kv_heads != 0) {
        *why = "n_heads must be a multiple of n_kv_heads";
        return LLAMA_ERR_UNSUPPORTED_DIMS;
    }
    if (d->n_heads / d->n_kv_heads > 64) {
        *why = "at most 64 query heads per KV head";
        return LLAMA_ERR_UNSUPPORTED_DIMS;
    }
    if (d->dtype == LLAMA_BF16) {
        if (d->head_dim != 128 || d->d_model % 128 != 0 || d->d_ff % 128 != 0) {
            *why = "bf16 blocks need head_dim 128 and d_model, d_ff multiples of 128";
            return LLAMA_ERR_UNSUPPORTED_DIMS;
        }
    } else if (d->dtype == LLAMA_F32) {
        if ((d->head_dim != 32 && d->head_dim != 64 && d->head_dim != 128) || d->d_model % 4 || d->d_ff % 4) {
            *why = "fp32 blocks need head_dim in {32, 64, 128} and d_model, d_ff multiples of 4";
            return LLAMA_ERR_UNSUPPORTED_DIMS;
        }
    } else {
        *why = "dtype must be LLAMA_F32 or LLAMA_BF16";
        return LLAMA_ERR_INVALID_ARG;
    }
    if (d->max_seq > (1 << 24)) {
        *why = "max_seq too large";
        return LLAMA_ERR_UNSUPPORTED_DIMS;
    }
    return LLAMA_OK;
}

}  // namespace

// ======================================================================== ABI

namespace {
// Radians per position of RoPE pair i: theta^(-2i/head_dim), or Llama 3.1's
// long-context schedule (fast band unchanged, slow band / factor, blend between),
// in fp64.
double rope_omega(const llama_block_dims& d, const llama_rope_scaling* sc, int i) {
    const double omega = std::pow((double)d.rope_theta, -2.0 * i / d.head_dim);
    if (!sc) return omega;
    const double pi = 3.14159265358979323846;
    const double wavelength = 2.0 * pi / omega;
    const double fast_edge = (double)sc->original_max_pos / sc->high_freq_factor;
    const double slow_edge = (double)sc->original_max_pos / sc->low_freq_factor;
    if (wavelength < fast_edge) return omega;
    if (wavelength > slow_edge) return omega / sc->factor;
    const double s = ((double)sc->original_max_pos / wavelength - sc->low_freq_factor) /
                     ((double)sc->high_freq_factor - sc->low_freq_factor);
    return (1.0 - s) * omega / sc->factor + s * omega;
}
}  // namespace

extern "C" int llama_block_create(const llama_block_dims* dims, const llama_block_weights* w, llama_block* out) {
    return llama_block_create_scaled(dims, w, nullptr, out);
}

extern "C" int llama_block_create_scaled(const llama_block_dims* dims, const llama_block_weights* w,
                                         const llama_rope_scaling* scaling, llama_block* out) {
    if (!out) return LLAMA_ERR_INVALID_ARG;
    *out = nullptr;
    std::string why;
    int rc = validate_dims(dims, &why);
    if (rc != LLAMA_OK) return rc;
    if (!w) return LLAMA_ERR_INVALID_ARG;
    if (scaling && !(scaling->factor >= 1.f && scaling->low_freq_factor > 0.f &&
                     scaling->high_freq_factor > scaling->low_freq_factor && scaling->original_max_pos > 0))
        return LLAMA_ERR_INVALID_ARG;
    const void* ptrs[9] = {w->g_attn, w->wq, w->wk, w->wv, w->wo, w->g_ffn, w->w_gate, w->w_up, w->w_down};
    for (const void* p : ptrs)
        if (!p || !aligned16(p)) return LLAMA_ERR_INVALID_ARG;
    llama_block b = new (std::nothrow) llama_block_s();
    if (!b) return LLAMA_ERR_INVALID_ARG;
    b->dims = *dims;
    b->w = *w;
    cudaGetDevice(&b->device);
    const auto& d = b->dims;
    if (d.dtype == LLAMA_BF16) {
        const uint64_t qd = (uint64_t)d.n_heads * d.head_dim, kvd = (uint64_t)d.n_kv_heads * d.head_dim;
        bool ok = make_tmap_bf16(&b->m_wq, w->wq, qd, d.d_model, 128, &why) &&
                  make_tmap_bf16(&b->m_wk, w->wk, kvd, d.d_model, 128, &why) &&
                  make_tmap_bf16(&b->m_wv, w->wv, kvd, d.d_model, 128, &why) &&
                  make_tmap_bf16(&b->m_wo, w->wo, d.d_model, qd, 128, &why) &&
                  make_tmap_bf16(&b->m_wg, w->w_gate, d.d_ff, d.d_model, 128, &why) &&
                  make_tmap_bf16(&b->m_wu, w->w_up, d.d_ff, d.d_model, 128, &why) &&
                  make_tmap_bf16(&b->m_wd, w->w_down, d.d_model, d.d_ff, 128, &why);
        if (!ok) {
            delete b;
            return LLAMA_ERR_CUDA;
        }
        const int n_sm = device_sm_count();
        const int qkv_tiles = (d.n_heads + 2 * d.n_kv_heads) * d.head_dim / 128;
        b->seg_kb[0] = choose_seg_kb(qkv_tiles, d.d_model / 64, n_sm);
        b->seg_kb[1] = choose_seg_kb(d.d_model / 128, d.n_heads * d.head_dim / 64, n_sm);
        b->seg_kb[2] = choose_seg_kb(d.d_ff / 128, d.d_model / 64, n_sm);
        b->seg_kb[3] = choose_seg_kb(d.d_model / 128, d.d_ff / 64, n_sm);
    }
    // cos/sin of p * omega_i, computed in fp64, stored fp32, padded to 64 pairs
    const size_t n = (size_t)d.max_seq * kRopeMaxPairs;
    std::vector<float> hc(n, 1.f), hs(n, 0.f);
    std::vector<double> omega(d.head_dim / 2);
    for (int i = 0; i < d.head_dim / 2; ++i) omega[i] = rope_omega(d, scaling, i);
    for (int p = 0; p < d.max_seq; ++p)
        for (int i = 0; i < d.head_dim / 2; ++i) {
            const double ang = (double)p * omega[i];
            hc[(size_t)p * kRopeMaxPairs + i] = (float)std::cos(ang);
            hs[(size_t)p * kRopeMaxPairs + i] = (float)std::sin(ang);
        }
    if (cudaMalloc(&b->cos_tab, n * sizeof(float)) != cudaSuccess ||
        cudaMalloc(&b->sin_tab, n * sizeof(float)) != cudaSuccess ||
        cudaMalloc(&b->err_dev, sizeof(int)) != cudaSuccess ||
        cudaMemcpy(b->cos_tab, hc.data(), n * sizeof(float), cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMemcpy(b->sin_tab, hs.data(), n * sizeof(float), cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMemset(b->err_dev, 0, sizeof(int)) != cudaSuccess) {
        llama_block_destroy(b);
        return LLAMA_ERR_CUDA;
    }
    *out = b;
    return LLAMA_OK;
}

extern "C" void llama_block_destroy(llama_block b) {
    if (!b) return;
    if (b->cos_tab) cudaFree(b->cos_tab);
    if (b->sin_tab) cudaFree(b->sin_tab);
    if (b->err_dev) cudaFree(b->err_dev);
    delete b;
}

extern "C" size_t llama_block_workspace_bytes(llama_block b, int batch, int tokens) {
    if (!b || batch <= 0 || tokens <= 0) return 0;
    // decode needs the attention partials; prefill does not
    return layout(b, batch, tokens, nullptr, tokens == 1).total;
}

extern "C" int llama_block_workspace_offsets(llama_block b, int batch, int tokens, size_t* offsets, int n) {
    if (!b || batch <= 0 || tokens <= 0 || !offsets || n < LLAMA_BLOCK_INTERMEDIATES) return LLAMA_ERR_INVALID_ARG;
    uint8_t* const base = (uint8_t*)(uintptr_t)kAlign;   // any aligned base: offsets are base-relative
    const Ws w = layout(b, batch, tokens, base, tokens == 1);
    const void* at[LLAMA_BLOCK_INTERMEDIATES] = {w.xn, w.q, w.o, w.h, w.hn, w.u};
    for (int i = 0; i < LLAMA_BLOCK_INTERMEDIATES; ++i) offsets[i] = (size_t)((const uint8_t*)at[i] - base);
    return LLAMA_BLOCK_INTERMEDIATES;
}

extern "C" int llama_block_prefill(llama_block b, const void* x, int batch, int tokens, const llama_kv_cache* kv,
                                   void* y, void* ws, size_t ws_bytes, void* stream) {
    if (!b) return LLAMA_ERR_INVALID_ARG;
    if (batch < 0 || tokens < 0) return fail(b, LLAMA_ERR_INVALID_ARG, "negative batch or tokens");
    if (batch == 0 || tokens == 0) return LLAMA_OK;
    if (!x || !y || !aligned16(x) || !aligned16(y))
        return fail(b, LLAMA_ERR_INVALID_ARG, "x / y null or not 16-byte aligned");
    int rc = check_kv(b, kv, batch, tokens - 1);
    if (rc != LLAMA_OK) return rc;
    return run_block(b, x, batch, tokens, kv, 0, nullptr, y, ws, ws_bytes, stream, false);
}

extern "C" int llama_block_prefill_at(llama_block b, const void* x, int batch, int tokens, int start_pos,
                                      const llama_kv_cache* kv, void* y, void* ws, size_t ws_bytes, void* stream) {
    if (!b) return LLAMA_ERR_INVALID_ARG;
    if (batch < 0 || tokens < 0) return fail(b, LLAMA_ERR_INVALID_ARG, "negative batch or tokens");
    if (start_pos < 0) return fail(b, LLAMA_ERR_POS_RANGE, "negative start position");
    if (batch == 0 || tokens == 0) return LLAMA_OK;
    if (!x || !y || !aligned16(x) || !aligned16(y))
        return fail(b, LLAMA_ERR_INVALID_ARG, "x / y null or not 16-byte aligned");
    if ((long)start_pos + tokens > b->dims.max_seq) return fail(b, LLAMA_ERR_POS_RANGE, "start_pos + tokens > max_seq");
    int rc = check_kv(b, kv, batch, start_pos + tokens - 1);
    if (rc != LLAMA_OK) return rc;
    return run_block(b, x, batch, tokens, kv, start_pos, nullptr, y, ws, ws_bytes, stream, false);
}

extern "C" int llama_block_decode(llama_block b, const void* x, int batch, const llama_kv_cache* kv, int pos,
                                  void* y, void* ws, size_t ws_bytes, void* stream) {
    if (!b) return LLAMA_ERR_INVALID_ARG;
    if (batch < 0) return fail(b, LLAMA_ERR_INVALID_ARG, "negative batch");
    if (batch == 0) return LLAMA_OK;
    if (!x || !y || !aligned16(x) || !aligned16(y))
        return fail(b, LLAMA_ERR_INVALID_ARG, "x / y null or not 16-byte aligned");
    if (pos < 0) return fail(b, LLAMA_ERR_POS_RANGE, "negative position");
    int rc = check_kv(b, kv, batch, pos);
    if (rc != LLAMA_OK) return rc;
    return run_block(b, x, batch, 1, kv, pos, nullptr, y, ws, ws_bytes, stream, true);
}

extern "C" int llama_block_decode_devpos(llama_block b, const void* x, int batch, const llama_kv_cache* kv,
                                         const int32_t* pos_dev, void* y, void* ws, size_t ws_bytes, void* stream) {
    if (!b) return LLAMA_ERR_INVALID_ARG;
    if (batch < 0) return fail(b, LLAMA_ERR_INVALID_ARG, "negative batch");
    if (batch == 0) return LLAMA_OK;
    if (!x || !y || !pos_dev || !aligned16(x) || !aligned16(y))
        return fail(b, LLAMA_ERR_INVALID_ARG, "x / y / pos_dev null or x / y not 16-byte aligned");
    int rc = check_kv(b, kv, batch, 0);
    if (rc != LLAMA_OK) return rc;
    return run_block(b, x, batch, 1, kv, 0, pos_dev, y, ws, ws_bytes, stream, true);
}

extern "C" int llama_block_decode_seqpos(llama_block b, const void* x, int batch, const llama_kv_cache* kv,
                                         const int32_t* pos_seq, void* y, void* ws, size_t ws_bytes, void* stream) {
    if (!b) return LLAMA_ERR_INVALID_ARG;
    if (batch < 0) return fail(b, LLAMA_ERR_INVALID_ARG, "negative batch");
    if (batch == 0) return LLAMA_OK;
    if (!x || !y || !pos_seq || !aligned16(x) || !aligned16(y))
        return fail(b, LLAMA_ERR_INVALID_ARG, "x / y / pos_seq null or x / y not 16-byte aligned");
    const auto& d = b->dims;
    // The per-sequence positions reach the QKV projection's epilogue (RoPE, cache
    // row), the weight-streaming decode attention and the combine: bf16, up to 8
    // query heads per KV head, at most 32 sequences (the weight-streaming schedule).
    if (d.dtype != LLAMA_BF16 || !attention_tc_supported(d.n_heads, d.n_kv_heads, d.head_dim) ||
        d.n_heads / d.n_kv_heads > 8 || batch > 32)
        return fail(b, LLAMA_ERR_UNSUPPORTED_DIMS, "per-sequence positions need the bf16 weight-streaming decode path");
    int rc = check_kv(b, kv, batch, 0);
    if (rc != LLAMA_OK) return rc;
    return run_block(b, x, batch, 1, kv, 0, nullptr, y, ws, ws_bytes, stream, true, pos_seq);
}

extern "C" int llama_block_poll_error(llama_block b, void* stream) {
    if (!b) return LLAMA_ERR_INVALID_ARG;
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(b, e, "stream synchronize");
    int v = 0;
    e = cudaMemcpy(&v, b->err_dev, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(b, e, "error word read");
    if (v != 0) {
        cudaMemset(b->err_dev, 0, sizeof(int));
        return fail(b, v, "a kernel reported error " + std::to_string(v));
    }
    return LLAMA_OK;
}

#ifdef LLAMA_TRACE
static int trace_set_all(const TraceCtl& c) {
    for (auto set : {trace_set_norm, trace_set_gemm_ws, trace_set_gemm_tt, trace_set_reduce, trace_set_attn_tc,
                     trace_set_attn_simt})
        if (set(c) != cudaSuccess) return LLAMA_ERR_CUDA;
    return LLAMA_OK;
}

extern "C" int llama_trace_begin(unsigned long long* records, unsigned int* count, unsigned int capacity) {
    if (!records || !count || capacity == 0) return LLAMA_ERR_INVALID_ARG;
    return trace_set_all(TraceCtl{records, count, capacity});
}

extern "C" int llama_trace_end(void) { return trace_set_all(TraceCtl{nullptr, nullptr, 0}); }
#else
// the product build records nothing
extern "C" int llama_trace_begin(unsigned long long*, unsigned int*, unsigned int) { return LLAMA_ERR_UNSUPPORTED_DIMS; }
extern "C" int llama_trace_end(void) { return LLAMA_OK; }
#endif

extern "C" int llama_block_selftest_wait_timeout(llama_block b, unsigned long long budget_ns, void* stream) {
    if (!b) return LLAMA_ERR_INVALID_ARG;
    if (budget_ns == 0 || budget_ns > 2000000000ull) budget_ns = 2000000000ull;
    cudaError_t e = launch_expire_wait(b->err_dev, budget_ns, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(b, e, "wait self-test launch");
    return LLAMA_OK;
}

extern "C" const char* llama_block_last_error(llama_block b) { return b ? b->last_error.c_str() : ""; }

extern "C" int llama_block_set_stage_events(llama_block b, void* const* events, int n_events) {
    if (!b) return LLAMA_ERR_INVALID_ARG;
    if (!events) {
        b->timing = false;
        return LLAMA_OK;
    }
    if (n_events != LLAMA_BLOCK_STAGES + 1) return fail(b, LLAMA_ERR_INVALID_ARG, "need LLAMA_BLOCK_STAGES + 1 events");
    for (int i = 0; i < n_events; ++i) {
        if (!events[i]) return fail(b, LLAMA_ERR_INVALID_ARG, "null event");
        b->stage_events[i] = (cudaEvent_t)events[i];
    }
    b->timing = true;
    return LLAMA_OK;
}

extern "C" int llama_block_launch_count(llama_block b) { return b ? b->last_launches : 0; }

extern "C" int llama_device_ptr_of_host(const void* host, void** dev) {
    if (!host || !dev) return LLAMA_ERR_INVALID_ARG;
    *dev = nullptr;
    void* p = nullptr;
    if (cudaHostGetDevicePointer(&p, const_cast<void*>(host), 0) != cudaSuccess) {
        cudaGetLastError();   // not pinned and mapped: clear the error, report it
        return LLAMA_ERR_INVALID_ARG;
    }
    *dev = p;
    return LLAMA_OK;
}

extern "C" int llama_rmsnorm(const void* x, const void* g, void* y, int rows, int d, float eps, int dtype,
                             void* stream) {
    if (rows < 0 || d <= 0) return LLAMA_ERR_INVALID_ARG;
    if (rows == 0) return LLAMA_OK;
    if (!x || !g || !y) return LLAMA_ERR_INVALID_ARG;
    if (dtype != LLAMA_BF16 && dtype != LLAMA_F32) return LLAMA_ERR_INVALID_ARG;
    return launch_rmsnorm(x, g, y, rows, d, eps, dtype, (cudaStream_t)stream) == cudaSuccess
               ? LLAMA_OK
               : LLAMA_ERR_CUDA;
}

extern "C" int llama_embed(const int32_t* ids, int n_tokens, const void* w_embed, int vocab, int d_model, void* x,
                           int32_t* err_dev, void* stream) {
    if (n_tokens < 0 || vocab <= 0 || d_model <= 0 || (d_model * 2) % 16) return LLAMA_ERR_INVALID_ARG;
    if (n_tokens == 0) return LLAMA_OK;
    if (!ids || !w_embed || !x || !aligned16(w_embed) || !aligned16(x)) return LLAMA_ERR_INVALID_ARG;
    return launch_embed(ids, n_tokens, w_embed, vocab, d_model, x, err_dev, (cudaStream_t)stream) == cudaSuccess
               ? LLAMA_OK
               : LLAMA_ERR_CUDA;
}

namespace {
struct HeadWs {
    void* hn;
    float* logits;
    int* err;   // set by an expired wait of the projection, reported through ids
    size_t total;
};
HeadWs head_layout(int batch, int d_model, int vocab, uint8_t* base, bool own_logits) {
    HeadWs w{};
    size_t off = 0;
    auto take = [&](size_t bytes) -> void* {
        void* p = base ? base + off : nullptr;
        off += align_up(bytes);
        return p;
    };
    w.hn = take((size_t)batch * d_model * 2);
    w.logits = own_logits ? (float*)take((size_t)batch * vocab * sizeof(float)) : nullptr;
    w.err = (int*)take(sizeof(int));
    w.total = off;
    return w;
}
}  // namespace

extern "C" size_t llama_lmhead_workspace_bytes(int batch, int d_model, int vocab) {
    if (batch <= 0 || d_model <= 0 || vocab <= 0) return 0;
    return head_layout(batch, d_model, vocab, nullptr, true).total;
}

extern "C" int llama_lmhead_argmax(const void* h, int batch, int h_stride, const void* g_final, const void* w_out,
                                   int vocab, int d_model, float eps, int32_t* ids, float* logits, void* ws,
                                   size_t ws_bytes, void* stream) {
    if (batch < 0 || vocab <= 0 || d_model <= 0 || d_model % 128 || vocab % 128) return LLAMA_ERR_INVALID_ARG;
    if (batch == 0) return LLAMA_OK;
    if (batch > 32 || !h || !g_final || !w_out || !ids || h_stride < d_model) return LLAMA_ERR_INVALID_ARG;
    const HeadWs need = head_layout(batch, d_model, vocab, nullptr, true);
    if (!ws || ws_bytes < need.total) return LLAMA_ERR_WORKSPACE;
    HeadWs w = head_layout(batch, d_model, vocab, (uint8_t*)ws, true);
    float* lg = logits ? logits : w.logits;
    cudaStream_t s = (cudaStream_t)stream;
    if (cudaMemsetAsync(w.err, 0, sizeof(int), s) != cudaSuccess) return LLAMA_ERR_CUDA;
    // final RMSNorm of the selected rows (row stride h_stride), one row at a time is
    // avoided by a strided view: the norm kernel reads rows of length d at stride d,
    // so copy-free only when h_stride == d_model.
    if (h_stride != d_model) {
        for (int r = 0; r < batch; ++r)
            if (launch_rmsnorm((const uint8_t*)h + (size_t)r * h_stride * 2, g_final, (uint8_t*)w.hn + (size_t)r * d_model * 2,
                               1, d_model, eps, LLAMA_BF16, s) != cudaSuccess)
                return LLAMA_ERR_CUDA;
    } else if (launch_rmsnorm(h, g_final, w.hn, batch, d_model, eps, LLAMA_BF16, s) != cudaSuccess) {
        return LLAMA_ERR_CUDA;
    }
    CUtensorMap mw;
    std::string why;
    if (!make_tmap_bf16(&mw, w_out, vocab, d_model, 128, &why)) return LLAMA_ERR_INVALID_ARG;
    GemmProblem p;
    p.M = batch;
    p.F = vocab;
    p.K = d_model;
    p.a_maps[0] = &mw;
    p.x = (const bf16*)w.hn;
    GemmEpi e;
    e.kind = EPI_LOGITS;
    e.out_f32 = lg;
    e.err = w.err;
    // one K segment per CTA: logits need no prefill counterpart, so each CTA owns whole dot products
    if (launch_gemm_single_segment(p, e, s) != cudaSuccess) return LLAMA_ERR_CUDA;
    if (launch_argmax_rows(lg, batch, vocab, ids, w.err, s) != cudaSuccess) return LLAMA_ERR_CUDA;
    return LLAMA_OK;
}

extern "C" int llama_sample(const float* logits, int batch, int vocab, float temperature, int top_k, float top_p,
                            const float* uniforms, int32_t* ids, void* stream) {
    if (batch < 0 || vocab <= 0 || vocab > (1 << 20) || batch > 65535) return LLAMA_ERR_INVALID_ARG;
    if (!(temperature >= 0.f) || std::isinf(temperature) || top_k < 0 || !(top_p > 0.f && top_p <= 1.f))
        return LLAMA_ERR_INVALID_ARG;
    if (batch == 0) return LLAMA_OK;
    if (!logits || !uniforms || !ids) return LLAMA_ERR_INVALID_ARG;
    return launch_sample(logits, batch, vocab, temperature, top_k, top_p, uniforms, ids, (cudaStream_t)stream) ==
                   cudaSuccess
               ? LLAMA_OK
               : LLAMA_ERR_CUDA;
}
