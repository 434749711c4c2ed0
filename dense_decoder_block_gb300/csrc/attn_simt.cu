// Causal GQA attention on CUDA cores, prefill and decode, with one shared
// reduction schedule.
//
// "Llama 3.1 70B", Grouped-Query Attention: scores q.k / sqrt(d_h), causal,
// softmax over keys, weights average V; query head h reads KV head
// h / (n_heads / n_kv_heads).  "Llama 3 8B · Prepare Q, K, V" (decode mode):
// K and V are cached at KV-head size and read once per group.
//
// Schedule.  Keys are cut into chunks of kAttnChunk = 128.  For one query row
// and one chunk a warp computes the chunk partial (m, l, o): m the chunk's max
// score (log2 domain), l = sum 2^(s - m), o = sum 2^(s - m) v.  Chunks are
// folded in ascending order from chunk 0.  The prefill kernel folds in
// registers as it walks the chunks; the decode kernel writes each chunk's
// partial to the workspace (split over CTAs) and the combine kernel folds them
// in the same order with the same function, so a decode row is bit-identical
// to the prefill row at the same position.  Keys past the query's position are
// neither scored nor loaded.
#include <cfloat>

#include "attn_fold.cuh"
#include "internal.h"

namespace llama {

namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kRowsMax = 64;    // query rows per prefill CTA (n_rep * tokens)
constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ void ptx_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void ptx_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ float to_f(bf16 v) { return __bfloat162float(v); }
__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ void from_f(bf16* p, float v) { *p = __float2bfloat16_rn(v); }
__device__ __forceinline__ void from_f(float* p, float v) { *p = v; }

template <typename T, int DH>
struct Tile {
    static constexpr int VEC = 16 / sizeof(T);          // elements per 16-byte vector
    static constexpr int LD = DH + VEC;                  // padded row stride (elements)
    static constexpr int DPL = DH / 32;                  // output dims per lane
};

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, bool valid) {
    const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
    const int src = valid ? 16 : 0;   // 0 -> zero fill, nothing read
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(s), "l"(gmem), "r"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

// Load keys [key0, key0 + 128) of one (sequence, kv head) into smem; keys above
// last_key are zero-filled without touching global memory.
template <typename T, int DH>
__device__ __forceinline__ void load_chunk(T* Ks, T* Vs, const T* kc, const T* vc, size_t head_base, int key0,
                                           int last_key) {
    using TL = Tile<T, DH>;
    constexpr int VPR = DH / TL::VEC;   // vectors per row
    for (int v = threadIdx.x; v < kAttnChunk * VPR; v += kThreads) {
        const int j = v / VPR, c = (v % VPR) * TL::VEC;
        const int key = key0 + j;
        const bool ok = key <= last_key;
        const size_t g = head_base + (size_t)(ok ? key : 0) * DH + c;
        cp_async16(Ks + j * TL::LD + c, kc + g, ok);
        cp_async16(Vs + j * TL::LD + c, vc + g, ok);
    }
    cp_async_wait_all();
}

// One warp: the partial of one query row (fp32 in smem) over one chunk.
// jmax = last key index inside the chunk this row may see (0..127).
template <typename T, int DH>
__device__ __forceinline__ void chunk_partial(const float* q, const T* Ks, const T* Vs, int jmax, float scale_log2,
                                              float& m_out, float& l_out, float (&o)[DH / 32]) {
    using TL = Tile<T, DH>;
    const int lane = threadIdx.x & 31;
    float s[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int j = lane + 32 * i;
        if (j <= jmax) {
            const T* kr = Ks + j * TL::LD;
            float acc = 0.f;
#pragma unroll 4
            for (int d = 0; d < DH; d += TL::VEC) {
                T kv[TL::VEC];
                *reinterpret_cast<uint4*>(kv) = *reinterpret_cast<const uint4*>(kr + d);
#pragma unroll
                for (int e = 0; e < TL::VEC; ++e) acc = __fmaf_rn(q[d + e], to_f(kv[e]), acc);
            }
            s[i] = __fmul_rn(acc, scale_log2);
        } else {
            s[i] = -INFINITY;
        }
    }
    float mx = fmaxf(fmaxf(s[0], s[1]), fmaxf(s[2], s[3]));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, off));
    float p[4];
    float l = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        p[i] = (lane + 32 * i <= jmax) ? exp2f(__fsub_rn(s[i], mx)) : 0.f;
        l = __fadd_rn(l, p[i]);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) l = __fadd_rn(l, __shfl_xor_sync(kFull, l, off));
    l = __shfl_sync(kFull, l, 0);
#pragma unroll
    for (int e = 0; e < TL::DPL; ++e) o[e] = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if (32 * i > jmax) break;
#pragma unroll 8
        for (int jj = 0; jj < 32; ++jj) {
            const int j = 32 * i + jj;
            if (j > jmax) break;
            const float pj = __shfl_sync(kFull, p[i], jj);
            const T* vr = Vs + j * TL::LD + lane * TL::DPL;
#pragma unroll
            for (int e = 0; e < TL::DPL; ++e) o[e] = __fmaf_rn(pj, to_f(vr[e]), o[e]);
        }
    }
    m_out = mx;
    l_out = l;
}

struct AttnK {
    const void* q;
    void* o;
    const void* kc;
    const void* vc;
    int batch, tokens, n_heads, n_kv_heads, kv_seq, start_pos, max_pos;
    const int* pos_dev;
    const int* pos_seq;   // decode combine: sequence b at position pos_seq[b]
    float scale_log2;
    float* partial;
    int n_chunks;
    int tq;    // prefill: tokens per CTA
    int* err;
};

__device__ __forceinline__ int base_position(const AttnK& a) { return a.pos_dev ? *a.pos_dev : a.start_pos; }

// ----------------------------------------------------------------------------- prefill
template <typename T, int DH>
__global__ void __launch_bounds__(kThreads) k_attn_prefill(const AttnK a) {
    using TL = Tile<T, DH>;
    constexpr int DPL = TL::DPL;
    constexpr int RPW = kRowsMax / kWarps;
    extern __shared__ __align__(16) uint8_t smem_raw[];
    T* Ks = reinterpret_cast<T*>(smem_raw);
    T* Vs = Ks + kAttnChunk * TL::LD;
    float* qs = reinterpret_cast<float*>(Vs + kAttnChunk * TL::LD);

    ptx_wait();
    if (threadIdx.x == 0) ptx_launch_dependents();
    const int g = blockIdx.y, b = blockIdx.z;
    const int n_rep = a.n_heads / a.n_kv_heads;
    const int t0 = blockIdx.x * a.tq;
    const int rows = n_rep * a.tq;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int base = base_position(a);
    const int t_last = min(t0 + a.tq, a.tokens) - 1;
    if (base < 0 || base + t_last >= a.max_pos) {
        if (threadIdx.x == 0) record_error(a.err, LLAMA_ERR_POS_RANGE);
        return;
    }
    const int pos_last = base + t_last;
    const T* q = reinterpret_cast<const T*>(a.q);
    const size_t qld = (size_t)a.n_heads * DH;
    for (int i = threadIdx.x; i < rows * DH; i += kThreads) {
        const int r = i / DH, d = i % DH;
        const int t = t0 + r / n_rep, h = g * n_rep + r % n_rep;
        qs[i] = (t < a.tokens) ? to_f(q[((size_t)b * a.tokens + t) * qld + (size_t)h * DH + d]) : 0.f;
    }
    float M[RPW], L[RPW], O[RPW][DPL];
    const size_t head_base = ((size_t)b * a.n_kv_heads + g) * a.kv_seq * DH;
    const int n_chunks = pos_last / kAttnChunk + 1;
    for (int c = 0; c < n_chunks; ++c) {
        __syncthreads();
        load_chunk<T, DH>(Ks, Vs, reinterpret_cast<const T*>(a.kc), reinterpret_cast<const T*>(a.vc), head_base,
                          c * kAttnChunk, pos_last);
        __syncthreads();
#pragma unroll
        for (int rr = 0; rr < RPW; ++rr) {
            const int r = warp + kWarps * rr;
            if (r >= rows) break;
            const int t = t0 + r / n_rep;
            if (t >= a.tokens) continue;
            const int pos = base + t;
            if (c * kAttnChunk > pos) continue;
            const int jmax = min(kAttnChunk - 1, pos - c * kAttnChunk);
            float m, l, o[DPL];
            chunk_partial<T, DH>(qs + r * DH, Ks, Vs, jmax, a.scale_log2, m, l, o);
            if (c == 0) {
                M[rr] = m;
                L[rr] = l;
#pragma unroll
                for (int e = 0; e < DPL; ++e) O[rr][e] = o[e];
            } else {
                fold<DPL>(M[rr], L[rr], O[rr], m, l, o);
            }
        }
    }
    T* out = reinterpret_cast<T*>(a.o);
#pragma unroll
    for (int rr = 0; rr < RPW; ++rr) {
        const int r = warp + kWarps * rr;
        if (r >= rows) break;
        const int t = t0 + r / n_rep;
        if (t >= a.tokens) continue;
        const int h = g * n_rep + r % n_rep;
        T* dst = out + ((size_t)b * a.tokens + t) * qld + (size_t)h * DH + lane * DPL;
        const float inv_l = __frcp_rn(L[rr]);
#pragma unroll
        for (int e = 0; e < DPL; ++e) from_f(dst + e, __fmul_rn(O[rr][e], inv_l));
    }
}

// ----------------------------------------------------------------------------- decode
template <typename T, int DH>
__global__ void __launch_bounds__(kThreads) k_attn_decode_chunks(const AttnK a) {
    using TL = Tile<T, DH>;
    constexpr int DPL = TL::DPL;
    extern __shared__ __align__(16) uint8_t smem_raw[];
    T* Ks = reinterpret_cast<T*>(smem_raw);
    T* Vs = Ks + kAttnChunk * TL::LD;
    float* qs = reinterpret_cast<float*>(Vs + kAttnChunk * TL::LD);

    ptx_wait();
    if (threadIdx.x == 0) ptx_launch_dependents();
    const int c = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int n_rep = a.n_heads / a.n_kv_heads;
    const int pos = base_position(a);
    if (pos < 0 || pos >= a.max_pos) {
        if (threadIdx.x == 0 && c == 0 && g == 0 && b == 0) record_error(a.err, LLAMA_ERR_POS_RANGE);
        return;
    }
    if (c * kAttnChunk > pos) return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const T* q = reinterpret_cast<const T*>(a.q);
    const size_t qld = (size_t)a.n_heads * DH;
    for (int i = threadIdx.x; i < n_rep * DH; i += kThreads) {
        const int r = i / DH, d = i % DH;
        qs[i] = to_f(q[(size_t)b * qld + (size_t)(g * n_rep + r) * DH + d]);
    }
    const size_t head_base = ((size_t)b * a.n_kv_heads + g) * a.kv_seq * DH;
    load_chunk<T, DH>(Ks, Vs, reinterpret_cast<const T*>(a.kc), reinterpret_cast<const T*>(a.vc), head_base,
                      c * kAttnChunk, pos);
    __syncthreads();
    const int jmax = min(kAttnChunk - 1, pos - c * kAttnChunk);
    for (int r = warp; r < n_rep; r += kWarps) {
        float m, l, o[DPL];
        chunk_partial<T, DH>(qs + r * DH, Ks, Vs, jmax, a.scale_log2, m, l, o);
        float* dst = a.partial + ((((size_t)b * a.n_kv_heads + g) * a.n_chunks + c) * n_rep + r) * part_stride(DH);
#pragma unroll
        for (int e = 0; e < DPL; ++e) dst[lane * DPL + e] = o[e];
        if (lane == 0) {
            dst[DH] = m;
            dst[DH + 1] = l;
        }
    }
}

template <typename T, int DH>
__global__ void __launch_bounds__(32) k_attn_decode_combine(const AttnK a) {
    TRACE(const unsigned long long tr0 = trace_stamp();)
    const int h = blockIdx.x, b = blockIdx.y, lane = threadIdx.x;
    // The position is set before the step, never by the kernels this one overlaps.
    const int pos = a.pos_seq ? a.pos_seq[b] : base_position(a);
    // The O projection after this kernel reads only its weights before its own wait:
    // it may launch at once and take the SMs as the attention CTAs leave them.
    if (threadIdx.x == 0) ptx_launch_dependents();
    ptx_wait();
    TRACE(const unsigned long long tr1 = trace_stamp();)
    const int n_rep = a.n_heads / a.n_kv_heads;
    const int g = h / n_rep, r = h % n_rep;
    if (pos < 0 || pos >= a.max_pos) return;
    const float* base = a.partial + (((size_t)b * a.n_kv_heads + g) * a.n_chunks * n_rep + r) * part_stride(DH);
    T* dst = reinterpret_cast<T*>(a.o) + (size_t)b * a.n_heads * DH + (size_t)h * DH;
    fold_row<T, DH>(base, (size_t)n_rep * part_stride(DH), pos / kAttnChunk + 1, lane, dst);
    TRACE(trace_cta(TR_ATTN_COMBINE, tr0, tr1);)
}

template <typename T, int DH>
size_t smem_bytes(int rows) {
    return 2 * (size_t)kAttnChunk * Tile<T, DH>::LD * sizeof(T) + (size_t)rows * DH * sizeof(float);
}

AttnK make_k(const AttnArgs& a) {
    AttnK k{};
    k.q = a.q;
    k.o = a.o;
    k.kc = a.kc;
    k.vc = a.vc;
    k.batch = a.batch;
    k.tokens = a.tokens;
    k.n_heads = a.n_heads;
    k.n_kv_heads = a.n_kv_heads;
    k.kv_seq = a.kv_seq;
    k.start_pos = a.start_pos;
    k.max_pos = a.max_pos;
    k.pos_dev = a.pos_dev;
    k.pos_seq = a.pos_seq;
    k.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)a.head_dim));
    k.partial = a.partial;
    k.n_chunks = a.n_chunks;
    k.err = a.err;
    return k;
}

template <typename T, int DH>
cudaError_t combine_launch(const AttnK& k, cudaStream_t s) {
    auto kern = k_attn_decode_combine<T, DH>;
    cudaError_t r = kernel_setup_once((const void*)kern, setup_prefer_shared);
    if (r != cudaSuccess) return r;
    return launch_pdl(kern, dim3(k.n_heads, k.batch), dim3(32), 0, s, k);
}

template <typename T, int DH>
cudaError_t prefill_impl(const AttnArgs& a, cudaStream_t s) {
    AttnK k = make_k(a);
    const int n_rep = a.n_heads / a.n_kv_heads;
    k.tq = kRowsMax / n_rep;
    if (k.tq < 1) return cudaErrorInvalidValue;
    const size_t sm = smem_bytes<T, DH>(kRowsMax);
    auto kern = k_attn_prefill<T, DH>;
    cudaError_t r = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (r != cudaSuccess) return r;
    dim3 grid((a.tokens + k.tq - 1) / k.tq, a.n_kv_heads, a.batch);
    return launch_pdl(kern, grid, dim3(kThreads), sm, s, k);
}

template <typename T, int DH>
cudaError_t decode_impl(const AttnArgs& a, cudaStream_t s) {
    AttnK k = make_k(a);
    const int n_rep = a.n_heads / a.n_kv_heads;
    const size_t sm = smem_bytes<T, DH>(n_rep);
    auto kern = k_attn_decode_chunks<T, DH>;
    cudaError_t r = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (r != cudaSuccess) return r;
    dim3 grid(a.n_chunks, a.n_kv_heads, a.batch);
    r = launch_pdl(kern, grid, dim3(kThreads), sm, s, k);
    if (r != cudaSuccess) return r;
    return combine_launch<T, DH>(k, s);
}

template <typename T, int DH>
cudaError_t combine_impl(const AttnArgs& a, cudaStream_t s) {
    return combine_launch<T, DH>(make_k(a), s);
}

}  // namespace

LLAMA_TRACE_UNIT(attn_simt)

size_t attn_decode_partial_bytes(int batch, int n_kv_heads, int n_chunks, int n_rep, int head_dim) {
    return (size_t)batch * n_kv_heads * n_chunks * n_rep * part_stride(head_dim) * sizeof(float);
}

cudaError_t launch_attention_combine(const AttnArgs& a, cudaStream_t s) {
    if (a.batch <= 0) return cudaSuccess;
    if (a.dtype == LLAMA_BF16) {
        if (a.head_dim == 128) return combine_impl<bf16, 128>(a, s);
        return cudaErrorInvalidValue;
    }
    switch (a.head_dim) {
        case 32: return combine_impl<float, 32>(a, s);
        case 64: return combine_impl<float, 64>(a, s);
        case 128: return combine_impl<float, 128>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_attention_prefill(const AttnArgs& a, cudaStream_t s) {
    if (a.batch <= 0 || a.tokens <= 0) return cudaSuccess;
    if (a.dtype == LLAMA_BF16) {
        if (a.head_dim == 128) return prefill_impl<bf16, 128>(a, s);
        return cudaErrorInvalidValue;
    }
    switch (a.head_dim) {
        case 32: return prefill_impl<float, 32>(a, s);
        case 64: return prefill_impl<float, 64>(a, s);
        case 128: return prefill_impl<float, 128>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_attention_decode(const AttnArgs& a, cudaStream_t s) {
    if (a.batch <= 0) return cudaSuccess;
    if (a.dtype == LLAMA_BF16) {
        if (a.head_dim == 128) return decode_impl<bf16, 128>(a, s);
        return cudaErrorInvalidValue;
    }
    switch (a.head_dim) {
        case 32: return decode_impl<float, 32>(a, s);
        case 64: return decode_impl<float, 64>(a, s);
        case 128: return decode_impl<float, 128>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace llama
