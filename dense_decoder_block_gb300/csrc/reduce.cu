// Decode-side segment reductions of the weight-streaming projections.
//
// The persistent projection kernel (gemm_ws.cuh) leaves one fp32 result per
// K-segment, laid out [segment][accumulator][token][feature].  Each kernel here
// adds an output's segments in ascending order -- the order of the token-tiled
// kernel's running sum -- and applies that projection's epilogue with the same
// device functions, so decode rows equal prefill rows bit for bit:
//   qkv:    bf16 round, RoPE on q/k pairs, q -> workspace, k/v -> cache row
//   resid:  y = bf16(x + bf16(sum))
//   swiglu: u = bf16(bf16(silu(bf16(gate))) * bf16(up))
//   resid + RMSNorm: h as resid, then hn = RMSNorm(h) with the 256-thread tree
// All loads of one output are issued before its additions (one round trip).
#include "internal.h"

namespace llama {

namespace {

constexpr int kThreads = 256;
constexpr int kBatch = 16;   // segments loaded per round trip

__device__ __forceinline__ void griddep() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Ascending sum over segments of 4 consecutive fp32 values at `off`.
__device__ __forceinline__ float4 seg_sum4(const float* part, size_t seg_stride, int n_segs, size_t off) {
    float4 s = __ldcg(reinterpret_cast<const float4*>(part + off));
    for (int s0 = 1; s0 < n_segs; s0 += kBatch) {
        float4 v[kBatch];
#pragma unroll
        for (int i = 0; i < kBatch; ++i)
            if (s0 + i < n_segs) v[i] = __ldcg(reinterpret_cast<const float4*>(part + (size_t)(s0 + i) * seg_stride + off));
#pragma unroll
        for (int i = 0; i < kBatch; ++i)
            if (s0 + i < n_segs) {
                s.x = __fadd_rn(s.x, v[i].x);
                s.y = __fadd_rn(s.y, v[i].y);
                s.z = __fadd_rn(s.z, v[i].z);
                s.w = __fadd_rn(s.w, v[i].w);
            }
    }
    return s;
}

__device__ __forceinline__ void store4(bf16* dst, float a, float b, float c, float d) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(a, b);
    __nv_bfloat162 hi = __floats2bfloat162_rn(c, d);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&lo);
    u.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(dst) = u;
}

__device__ __forceinline__ float4 load4_bf16(const bf16* src) {
    const uint2 u = *reinterpret_cast<const uint2*>(src);
    const __nv_bfloat162 lo = *reinterpret_cast<const __nv_bfloat162*>(&u.x);
    const __nv_bfloat162 hi = *reinterpret_cast<const __nv_bfloat162*>(&u.y);
    return make_float4(__low2float(lo), __high2float(lo), __low2float(hi), __high2float(hi));
}

__global__ void __launch_bounds__(kThreads) k_reduce_qkv(const ReduceArgs r) {
    griddep();
    const int F4 = r.F / 4;
    const int idx = blockIdx.x * kThreads + threadIdx.x;
    if (idx >= r.M * F4) return;
    const int n = idx / F4, f0 = (idx - n * F4) * 4;
    const float4 s = seg_sum4(r.partial, (size_t)r.M * r.F, r.n_segs, (size_t)n * r.F + f0);
    const GemmEpi& e = r.e;
    const int tile = f0 / 128, row0 = f0 % 128;
    int kind, head;
    if (tile < e.n_heads) { kind = 0; head = tile; }
    else if (tile < e.n_heads + e.n_kv_heads) { kind = 1; head = tile - e.n_heads; }
    else { kind = 2; head = tile - e.n_heads - e.n_kv_heads; }
    const int T = e.tokens_per_seq;
    const int b = n / T, t = n - b * T;
    const int pos = (e.pos_dev ? *e.pos_dev : e.start_pos) + t;
    if (pos < 0 || pos >= e.max_pos) {
        record_error(e.err, LLAMA_ERR_POS_RANGE);
        return;
    }
    float v0 = bf16_round(s.x), v1 = bf16_round(s.y), v2 = bf16_round(s.z), v3 = bf16_round(s.w);
    if (kind < 2) {
        const int i0 = row0 >> 1;
        const float c0 = __ldg(e.cos_tab + (size_t)pos * kRopeMaxPairs + i0);
        const float s0 = __ldg(e.sin_tab + (size_t)pos * kRopeMaxPairs + i0);
        const float c1 = __ldg(e.cos_tab + (size_t)pos * kRopeMaxPairs + i0 + 1);
        const float s1 = __ldg(e.sin_tab + (size_t)pos * kRopeMaxPairs + i0 + 1);
        const float r0 = rope_rotate_elem(v0, v1, c0, s0, false), r1 = rope_rotate_elem(v1, v0, c0, s0, true);
        const float r2 = rope_rotate_elem(v2, v3, c1, s1, false), r3 = rope_rotate_elem(v3, v2, c1, s1, true);
        v0 = r0; v1 = r1; v2 = r2; v3 = r3;
    }
    bf16* dst;
    if (kind == 0) dst = e.out + (size_t)n * (e.n_heads * 128) + head * 128 + row0;
    else dst = ((kind == 1) ? e.kc : e.vc) + (((size_t)b * e.n_kv_heads + head) * e.kv_seq + pos) * 128 + row0;
    store4(dst, v0, v1, v2, v3);
}

__global__ void __launch_bounds__(kThreads) k_reduce_resid(const ReduceArgs r) {
    griddep();
    const int F4 = r.F / 4;
    const int idx = blockIdx.x * kThreads + threadIdx.x;
    if (idx >= r.M * F4) return;
    const int n = idx / F4, f0 = (idx - n * F4) * 4;
    const size_t off = (size_t)n * r.F + f0;
    const float4 s = seg_sum4(r.partial, (size_t)r.M * r.F, r.n_segs, off);
    const float4 x = load4_bf16(r.e.resid + off);
    store4(r.e.out + off, epi_resid(x.x, s.x), epi_resid(x.y, s.y), epi_resid(x.z, s.z), epi_resid(x.w, s.w));
}

__global__ void __launch_bounds__(kThreads) k_reduce_swiglu(const ReduceArgs r) {
    griddep();
    const int F4 = r.F / 4;
    const int idx = blockIdx.x * kThreads + threadIdx.x;
    if (idx >= r.M * F4) return;
    const int n = idx / F4, f0 = (idx - n * F4) * 4;
    const size_t off = (size_t)n * r.F + f0;
    const size_t plane = (size_t)r.M * r.F;                  // [seg][gate|up][M][F]
    const float4 g = seg_sum4(r.partial, 2 * plane, r.n_segs, off);
    const float4 u = seg_sum4(r.partial, 2 * plane, r.n_segs, plane + off);
    store4(r.e.out + off, epi_swiglu(g.x, u.x), epi_swiglu(g.y, u.y), epi_swiglu(g.z, u.z), epi_swiglu(g.w, u.w));
}

// One CTA per token row: h = resid epilogue, then RMSNorm(h) with the same element
// ownership (i = tid + 256 e) and tree as the standalone RMSNorm kernel.
template <int EPT>
__global__ void __launch_bounds__(kThreads) k_reduce_resid_norm(const ReduceArgs r, const bf16* __restrict__ gain,
                                                                bf16* __restrict__ hn, float eps) {
    __shared__ float red[8];
    griddep();
    const int n = blockIdx.x, tid = threadIdx.x;
    const int d = r.F;
    const size_t plane = (size_t)r.M * r.F;
    const size_t row = (size_t)n * d;
    constexpr int SB = (64 / EPT) > 0 ? (64 / EPT) : 1;   // segments per load batch
    float acc[EPT];
    {
        float v[EPT];
#pragma unroll
        for (int e = 0; e < EPT; ++e) acc[e] = __ldcg(r.partial + row + tid + 256 * e);
        for (int s0 = 1; s0 < r.n_segs; s0 += SB) {
            float w[SB][EPT];
#pragma unroll
            for (int i = 0; i < SB; ++i)
                if (s0 + i < r.n_segs)
#pragma unroll
                    for (int e = 0; e < EPT; ++e) w[i][e] = __ldcg(r.partial + (size_t)(s0 + i) * plane + row + tid + 256 * e);
#pragma unroll
            for (int i = 0; i < SB; ++i)
                if (s0 + i < r.n_segs)
#pragma unroll
                    for (int e = 0; e < EPT; ++e) acc[e] = __fadd_rn(acc[e], w[i][e]);
        }
        (void)v;
    }
    float h[EPT];
    float ss = 0.f;
#pragma unroll
    for (int e = 0; e < EPT; ++e) {
        const int i = tid + 256 * e;
        const bf16 hb = __float2bfloat16_rn(epi_resid(__bfloat162float(r.e.resid[row + i]), acc[e]));
        r.e.out[row + i] = hb;
        h[e] = __bfloat162float(hb);
        ss = __fmaf_rn(h[e], h[e], ss);
    }
    const float scale = rms_scale(rms_tree_256(ss, red), d, eps);
#pragma unroll
    for (int e = 0; e < EPT; ++e) {
        const int i = tid + 256 * e;
        const float xs = bf16_round(__fmul_rn(h[e], scale));
        hn[row + i] = __float2bfloat16_rn(__fmul_rn(xs, __bfloat162float(gain[i])));
    }
}

dim3 grid4(const ReduceArgs& r) { return dim3((unsigned)(((size_t)r.M * (r.F / 4) + kThreads - 1) / kThreads)); }

}  // namespace

cudaError_t launch_reduce(const ReduceArgs& r, int kind, cudaStream_t s) {
    if (r.M <= 0) return cudaSuccess;
    if (r.F % 4) return cudaErrorInvalidValue;
    switch (kind) {
        case EPI_QKV: return launch_pdl(k_reduce_qkv, grid4(r), dim3(kThreads), 0, s, r);
        case EPI_RESID: return launch_pdl(k_reduce_resid, grid4(r), dim3(kThreads), 0, s, r);
        case EPI_SWIGLU: return launch_pdl(k_reduce_swiglu, grid4(r), dim3(kThreads), 0, s, r);
        default: return cudaErrorInvalidValue;
    }
}

bool reduce_resid_norm_supported(int d) {
    return d % 256 == 0 && (d / 256 == 1 || d / 256 == 2 || d / 256 == 4 || d / 256 == 8 || d / 256 == 16 ||
                            d / 256 == 32);
}

cudaError_t launch_reduce_resid_norm(const ReduceArgs& r, const void* gain, void* hn, float eps, cudaStream_t s) {
    if (r.M <= 0) return cudaSuccess;
    const dim3 g(r.M), b(kThreads);
    switch (r.F / 256) {
        case 1: return launch_pdl(k_reduce_resid_norm<1>, g, b, 0, s, r, (const bf16*)gain, (bf16*)hn, eps);
        case 2: return launch_pdl(k_reduce_resid_norm<2>, g, b, 0, s, r, (const bf16*)gain, (bf16*)hn, eps);
        case 4: return launch_pdl(k_reduce_resid_norm<4>, g, b, 0, s, r, (const bf16*)gain, (bf16*)hn, eps);
        case 8: return launch_pdl(k_reduce_resid_norm<8>, g, b, 0, s, r, (const bf16*)gain, (bf16*)hn, eps);
        case 16: return launch_pdl(k_reduce_resid_norm<16>, g, b, 0, s, r, (const bf16*)gain, (bf16*)hn, eps);
        case 32: return launch_pdl(k_reduce_resid_norm<32>, g, b, 0, s, r, (const bf16*)gain, (bf16*)hn, eps);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace llama
