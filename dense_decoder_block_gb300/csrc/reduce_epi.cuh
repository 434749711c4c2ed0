// The epilogues of the segment reductions (reduce.cu), on 4 consecutive features
// of one token.  They apply the element functions of common.cuh that the
// projection kernels' fused epilogues apply, so a reduced decode output has the
// same bits as the token-tiled prefill kernel's.
#pragma once
#include "common.cuh"
#include "internal.h"

namespace llama {

__device__ __forceinline__ void add4(float4& s, const float4& v) {
    s.x = __fadd_rn(s.x, v.x);
    s.y = __fadd_rn(s.y, v.y);
    s.z = __fadd_rn(s.z, v.z);
    s.w = __fadd_rn(s.w, v.w);
}

// Ascending sums over segments of 4 consecutive fp32 values at off (and at off2
// when PAIR): the loads of a batch of NB segments are all issued before its adds.
// The sums start at -0, and -0 + x == x for every fp32 x, so each equals
// ((s0 + s1) + s2) + ... exactly.
template <bool PAIR, int NB>
__device__ __forceinline__ void seg_sum4(const float* part, size_t seg_stride, int n_segs, size_t off, size_t off2,
                                         float4& s, float4& s2) {
    s = make_float4(-0.f, -0.f, -0.f, -0.f);
    s2 = s;
    for (int s0 = 0; s0 < n_segs; s0 += NB) {
        float4 v[NB], w[NB];
#pragma unroll
        for (int i = 0; i < NB; ++i)
            if (s0 + i < n_segs) {
                v[i] = __ldcg(reinterpret_cast<const float4*>(part + (size_t)(s0 + i) * seg_stride + off));
                if (PAIR) w[i] = __ldcg(reinterpret_cast<const float4*>(part + (size_t)(s0 + i) * seg_stride + off2));
            }
#pragma unroll
        for (int i = 0; i < NB; ++i)
            if (s0 + i < n_segs) {
                add4(s, v[i]);
                if (PAIR) add4(s2, w[i]);
            }
    }
}

__device__ __forceinline__ void store4_bf16(bf16* dst, float a, float b, float c, float d) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(a, b);
    __nv_bfloat162 hi = __floats2bfloat162_rn(c, d);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&lo);
    u.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(dst) = u;
}

// Through L2 (__ldcg): the values may have been written by an earlier kernel of the
// step that ran on another SM.
__device__ __forceinline__ float4 load4_bf16(const bf16* src) {
    const uint2 u = __ldcg(reinterpret_cast<const uint2*>(src));
    const __nv_bfloat162 lo = *reinterpret_cast<const __nv_bfloat162*>(&u.x);
    const __nv_bfloat162 hi = *reinterpret_cast<const __nv_bfloat162*>(&u.y);
    return make_float4(__low2float(lo), __high2float(lo), __low2float(hi), __high2float(hi));
}

// QKV: bf16 round, RoPE on q/k pairs, q -> workspace, k/v -> the cache row of the
// token's position.  f0 = first of the 4 features (a multiple of 4), n = token.
// The work splits in two: epi4_qkv_prepare reads only what the step's earlier
// kernels do not write (the position, the RoPE tables) and may run before
// griddepcontrol.wait; epi4_qkv_apply takes the segment sum.
struct Qkv4 {
    bf16* dst;              // null: position out of range (error recorded)
    float c0, s0, c1, s1;   // rotation of the pairs (f0, f0+1), (f0+2, f0+3); unused for v
    bool rope;
};

__device__ __forceinline__ Qkv4 epi4_qkv_prepare(const GemmEpi& e, int n, int f0) {
    Qkv4 p{};
    const int tile = f0 / 128, row0 = f0 % 128;
    int kind, head;
    if (tile < e.n_heads) { kind = 0; head = tile; }
    else if (tile < e.n_heads + e.n_kv_heads) { kind = 1; head = tile - e.n_heads; }
    else { kind = 2; head = tile - e.n_heads - e.n_kv_heads; }
    const int T = e.tokens_per_seq;
    const int b = n / T, t = n - b * T;
    const int pos = e.pos_seq ? e.pos_seq[b] : (e.pos_dev ? *e.pos_dev : e.start_pos) + t;   // pos_seq: T = 1
    if (pos < 0 || pos >= e.max_pos) {
        record_error(e.err, LLAMA_ERR_POS_RANGE);
        p.dst = nullptr;
        return p;
    }
    p.rope = kind < 2;
    if (p.rope) {
        const int i0 = row0 >> 1;
        p.c0 = __ldg(e.cos_tab + (size_t)pos * kRopeMaxPairs + i0);
        p.s0 = __ldg(e.sin_tab + (size_t)pos * kRopeMaxPairs + i0);
        p.c1 = __ldg(e.cos_tab + (size_t)pos * kRopeMaxPairs + i0 + 1);
        p.s1 = __ldg(e.sin_tab + (size_t)pos * kRopeMaxPairs + i0 + 1);
    }
    if (kind == 0) p.dst = e.out + (size_t)n * (e.n_heads * 128) + head * 128 + row0;
    else p.dst = ((kind == 1) ? e.kc : e.vc) + (((size_t)b * e.n_kv_heads + head) * e.kv_seq + pos) * 128 + row0;
    return p;
}

__device__ __forceinline__ void epi4_qkv_apply(const Qkv4& p, float4 s) {
    if (p.dst == nullptr) return;
    float v0 = bf16_round(s.x), v1 = bf16_round(s.y), v2 = bf16_round(s.z), v3 = bf16_round(s.w);
    if (p.rope) {
        const float r0 = rope_rotate_elem(v0, v1, p.c0, p.s0, false), r1 = rope_rotate_elem(v1, v0, p.c0, p.s0, true);
        const float r2 = rope_rotate_elem(v2, v3, p.c1, p.s1, false), r3 = rope_rotate_elem(v3, v2, p.c1, p.s1, true);
        v0 = r0; v1 = r1; v2 = r2; v3 = r3;
    }
    store4_bf16(p.dst, v0, v1, v2, v3);
}

// y = bf16(x + bf16(sum)), [M, F] row-major; x (the residual) was loaded by the caller
__device__ __forceinline__ void epi4_resid(const GemmEpi& e, int F, int n, int f0, float4 x, float4 s) {
    const size_t off = (size_t)n * F + f0;
    store4_bf16(e.out + off, epi_resid(x.x, s.x), epi_resid(x.y, s.y), epi_resid(x.z, s.z), epi_resid(x.w, s.w));
}

// u = bf16(bf16(silu(bf16(gate))) * bf16(up))
__device__ __forceinline__ void epi4_swiglu(const GemmEpi& e, int F, int n, int f0, float4 g, float4 u) {
    store4_bf16(e.out + (size_t)n * F + f0, epi_swiglu(g.x, u.x), epi_swiglu(g.y, u.y), epi_swiglu(g.z, u.z),
                epi_swiglu(g.w, u.w));
}

}  // namespace llama
