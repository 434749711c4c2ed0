// The ascending fold of attention chunk partials: the CUDA-core prefill kernel
// folds with it as it walks the chunks, and the decode combine kernel folds the
// stored partials of both decode kernels with it, so decode rows carry the same
// bits as the prefill rows (the tensor-core prefill kernel's fold warps apply
// the same formula).
//
// "Llama 3.1 70B", Grouped-Query Attention (softmax over the keys, weights
// average V), computed per chunk of keys: a chunk partial is (m, l, o) with m
// the chunk's scaled max score (log2 domain), l = sum 2^(s - m) and
// o = sum 2^(s - m) v.  Folding chunk c into the running (M, L, O):
//   M' = max(M, m), L' = L 2^(M - M') + l 2^(m - M'), O' likewise;
// the row's output is O / L, computed as O * (1 / L).
//
// Partial layout: [sequence][KV head][chunk slot][query row of the group][head_dim + 4]
// floats, o first, then m and l.
#pragma once
#include "common.cuh"

namespace llama {

// Fold the partial (m, l, o) of the next chunk into the running state (M, L, O).
template <int DPL>
__device__ __forceinline__ void fold(float& M, float& L, float (&O)[DPL], float m, float l, const float (&o)[DPL]) {
    const float Mn = fmaxf(M, m);
    const float a = exp2f(__fsub_rn(M, Mn));
    const float b = exp2f(__fsub_rn(m, Mn));
    L = __fmaf_rn(L, a, __fmul_rn(l, b));
#pragma unroll
    for (int e = 0; e < DPL; ++e) O[e] = __fmaf_rn(O[e], a, __fmul_rn(o[e], b));
    M = Mn;
}

// One chunk partial's DPL values of this lane (16-, 8- or 4-byte loads through L2:
// the partials were written by other CTAs).
template <int DPL>
__device__ __forceinline__ void ld_part(const float* p, float (&o)[DPL]) {
    if constexpr (DPL == 4) {
        const float4 v = __ldcg(reinterpret_cast<const float4*>(p));
        o[0] = v.x; o[1] = v.y; o[2] = v.z; o[3] = v.w;
    } else if constexpr (DPL == 2) {
        const float2 v = __ldcg(reinterpret_cast<const float2*>(p));
        o[0] = v.x; o[1] = v.y;
    } else {
#pragma unroll
        for (int e = 0; e < DPL; ++e) o[e] = __ldcg(p + e);
    }
}

__device__ __forceinline__ void store_out(bf16* p, float v) { *p = __float2bfloat16_rn(v); }
__device__ __forceinline__ void store_out(float* p, float v) { *p = v; }

// One warp folds the n_chunks partials of one query row (chunk 0 at `base`, the
// next ones cstride floats apart) and writes the row's head_dim outputs to dst;
// lane owns dims lane*DPL .. lane*DPL + DPL-1.  The loads of a batch of chunks are
// issued before its folds (one memory round trip per batch).
template <typename T, int DH>
__device__ __forceinline__ void fold_row(const float* base, size_t cstride, int n_chunks, int lane, T* dst) {
    constexpr int DPL = DH / 32;
    constexpr int kCB = 8;
    float M = 0.f, L = 0.f, O[DPL];
#pragma unroll
    for (int e = 0; e < DPL; ++e) O[e] = 0.f;
    for (int c0 = 0; c0 < n_chunks; c0 += kCB) {
        float o[kCB][DPL], m[kCB], l[kCB];
#pragma unroll
        for (int i = 0; i < kCB; ++i)
            if (c0 + i < n_chunks) {
                const float* p = base + (size_t)(c0 + i) * cstride;
                ld_part<DPL>(p + lane * DPL, o[i]);
                const float2 ml = __ldcg(reinterpret_cast<const float2*>(p + DH));
                m[i] = ml.x;
                l[i] = ml.y;
            }
#pragma unroll
        for (int i = 0; i < kCB; ++i) {
            if (c0 + i >= n_chunks) break;
            if (c0 + i == 0) {
                M = m[0];
                L = l[0];
#pragma unroll
                for (int e = 0; e < DPL; ++e) O[e] = o[0][e];
            } else {
                fold<DPL>(M, L, O, m[i], l[i], o[i]);
            }
        }
    }
    const float inv_l = __frcp_rn(L);
#pragma unroll
    for (int e = 0; e < DPL; ++e) store_out(dst + lane * DPL + e, __fmul_rn(O[e], inv_l));
}

}  // namespace llama
