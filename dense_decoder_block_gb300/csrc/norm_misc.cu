// RMSNorm, the fp32 (CUDA-core) projection path, embedding gather and row argmax.
#include <cfloat>

#include "internal.h"

namespace llama {

namespace {

constexpr int kNormThreads = 256;

__device__ __forceinline__ float to_f(bf16 v) { return __bfloat162float(v); }
__device__ __forceinline__ float to_f(float v) { return v; }

// "Llama 3.1 70B", RMSNorm reference implementation: fp32 mean of squares,
// eps inside the square root, the scaled row cast to the trunk dtype before the
// gain multiplies it.  One CTA per row; the sum of squares uses one fixed tree
// (thread-sequential, warp butterfly read at lane 0, warps in ascending order),
// the same for every caller, so prefill and decode rows agree bit for bit.
template <typename T>
__global__ void __launch_bounds__(kNormThreads) k_rmsnorm(const T* __restrict__ x, const T* __restrict__ g,
                                                          T* __restrict__ y, int d, float eps, unsigned* zero,
                                                          int n_zero) {
    __shared__ float red[kNormThreads / 32];
    __shared__ float s_scale;
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int row = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (blockIdx.x == 0 && zero)
        for (int i = tid; i < n_zero; i += kNormThreads) zero[i] = 0u;
    const T* xr = x + (size_t)row * d;
    float ss = 0.f;
    for (int i = tid; i < d; i += kNormThreads) {
        const float v = to_f(xr[i]);
        ss = __fmaf_rn(v, v, ss);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, off));
    if (lane == 0) red[warp] = ss;
    __syncthreads();
    if (tid == 0) {
        float t = red[0];
        for (int w = 1; w < kNormThreads / 32; ++w) t = __fadd_rn(t, red[w]);
        s_scale = rms_scale(t, d, eps);
    }
    __syncthreads();
    const float r = s_scale;
    T* yr = y + (size_t)row * d;
    for (int i = tid; i < d; i += kNormThreads) {
        const float v = to_f(xr[i]);
        if constexpr (sizeof(T) == 2) {
            const float xs = bf16_round(__fmul_rn(v, r));
            yr[i] = __float2bfloat16_rn(__fmul_rn(xs, to_f(g[i])));
        } else {
            yr[i] = __fmul_rn(__fmul_rn(v, r), to_f(g[i]));
        }
    }
}

// fp32 projection: one thread per output, ascending K (the same order for any M).
__global__ void k_linear_f32(const float* __restrict__ x, const float* __restrict__ w,
                             const float* __restrict__ w2, const float* __restrict__ resid, float* __restrict__ y,
                             int M, int F, int K, int mode) {
    const int f = blockIdx.x * blockDim.x + threadIdx.x;
    const int n = blockIdx.y;
    if (f >= F || n >= M) return;
    const float* xr = x + (size_t)n * K;
    const float* wr = w + (size_t)f * K;
    float acc = 0.f;
    for (int k = 0; k < K; ++k) acc = __fmaf_rn(xr[k], wr[k], acc);
    const size_t idx = (size_t)n * F + f;
    if (mode == 0) {
        y[idx] = acc;
    } else if (mode == 1) {
        y[idx] = __fadd_rn(resid[idx], acc);
    } else {
        const float* w2r = w2 + (size_t)f * K;
        float up = 0.f;
        for (int k = 0; k < K; ++k) up = __fmaf_rn(xr[k], w2r[k], up);
        y[idx] = __fmul_rn(silu_f(acc), up);
    }
}

// fp32 RoPE on q and k (adjacent pairs), q -> workspace, k and v -> cache rows.
__global__ void k_rope_append_f32(const float* __restrict__ qr, const float* __restrict__ kr,
                                  const float* __restrict__ vr, float* __restrict__ q_out, float* __restrict__ kc,
                                  float* __restrict__ vc, int T, int n_heads, int n_kv_heads, int dh, int kv_seq,
                                  int start_pos, const int* pos_dev, int max_pos, const float* __restrict__ cos_t,
                                  const float* __restrict__ sin_t, int* err) {
    const int n = blockIdx.x;   // token
    const int b = n / T, t = n - b * T;
    const int base = pos_dev ? *pos_dev : start_pos;
    const int pos = base + t;
    if (pos < 0 || pos >= max_pos) {
        if (threadIdx.x == 0) record_error(err, LLAMA_ERR_POS_RANGE);
        return;
    }
    const int qd = n_heads * dh, kd = n_kv_heads * dh;
    for (int i = threadIdx.x; i < qd + 2 * kd; i += blockDim.x) {
        if (i < qd + kd) {
            const bool isq = i < qd;
            const int c = isq ? i : i - qd;
            const float* src = isq ? qr + (size_t)n * qd : kr + (size_t)n * kd;
            const int j = c % dh, pair = j >> 1;
            const float self = src[c], other = src[c ^ 1];
            const float cs = cos_t[(size_t)pos * kRopeMaxPairs + pair];
            const float sn = sin_t[(size_t)pos * kRopeMaxPairs + pair];
            const float v = rope_rotate_elem(self, other, cs, sn, (j & 1) != 0);
            if (isq) {
                q_out[(size_t)n * qd + c] = v;
            } else {
                const int h = c / dh;
                kc[(((size_t)b * n_kv_heads + h) * kv_seq + pos) * dh + j] = v;
            }
        } else {
            const int c = i - qd - kd;
            const int h = c / dh, j = c % dh;
            vc[(((size_t)b * n_kv_heads + h) * kv_seq + pos) * dh + j] = vr[(size_t)n * kd + c];
        }
    }
}

template <typename T>
__global__ void k_embed(const int32_t* __restrict__ ids, const T* __restrict__ w, T* __restrict__ x, int vocab,
                        int d, int32_t* err) {
    const int n = blockIdx.x;
    const int id = ids[n];
    const bool ok = id >= 0 && id < vocab;
    if (!ok && threadIdx.x == 0 && err) atomicCAS(err, 0, LLAMA_ERR_INVALID_ARG);
    const uint4* src = reinterpret_cast<const uint4*>(w + (size_t)(ok ? id : 0) * d);
    uint4* dst = reinterpret_cast<uint4*>(x + (size_t)n * d);
    const int nv = d * (int)sizeof(T) / 16;
    for (int i = threadIdx.x; i < nv; i += blockDim.x) dst[i] = ok ? src[i] : make_uint4(0, 0, 0, 0);
}

// argmax over one row of fp32 logits; ties go to the lowest index.
__global__ void __launch_bounds__(1024) k_argmax_rows(const float* __restrict__ logits, int vocab,
                                                      int32_t* __restrict__ ids) {
    __shared__ float sv[32];
    __shared__ int si[32];
    const int row = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float* lr = logits + (size_t)row * vocab;
    float best = -INFINITY;
    int bi = INT32_MAX;
    for (int i = tid; i < vocab; i += blockDim.x) {
        const float v = lr[i];
        if (v > best) { best = v; bi = i; }   // ascending i: the first maximum stays
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, best, off);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
        if (ov > best || (ov == best && oi < bi)) { best = ov; bi = oi; }
    }
    if (lane == 0) { sv[warp] = best; si[warp] = bi; }
    __syncthreads();
    if (tid == 0) {
        for (int w = 1; w < (int)(blockDim.x / 32); ++w)
            if (sv[w] > best || (sv[w] == best && si[w] < bi)) { best = sv[w]; bi = si[w]; }
        ids[row] = (bi == INT32_MAX) ? 0 : bi;
    }
}

}  // namespace

cudaError_t launch_rmsnorm(const void* x, const void* g, void* y, int rows, int d, float eps, int dtype,
                           unsigned* zero_words, int n_zero, cudaStream_t s) {
    if (rows <= 0) return cudaSuccess;
    if (dtype == LLAMA_BF16)
        return launch_pdl(k_rmsnorm<bf16>, dim3(rows), dim3(kNormThreads), 0, s, (const bf16*)x, (const bf16*)g,
                          (bf16*)y, d, eps, zero_words, n_zero);
    return launch_pdl(k_rmsnorm<float>, dim3(rows), dim3(kNormThreads), 0, s, (const float*)x, (const float*)g,
                      (float*)y, d, eps, zero_words, n_zero);
}

cudaError_t launch_linear_f32(const float* x, const float* w, const float* w2, const float* resid, float* y, int M,
                              int F, int K, int mode, cudaStream_t s) {
    if (M <= 0) return cudaSuccess;
    dim3 grid((F + 127) / 128, M);
    k_linear_f32<<<grid, 128, 0, s>>>(x, w, w2, resid, y, M, F, K, mode);
    return cudaGetLastError();
}

cudaError_t launch_rope_append_f32(const float* qkv_q, const float* qkv_k, const float* qkv_v, float* q_out,
                                   float* kc, float* vc, int M, int T, int n_heads, int n_kv_heads, int head_dim,
                                   int kv_seq, int start_pos, const int* pos_dev, int max_pos,
                                   const float* cos_tab, const float* sin_tab, int* err, cudaStream_t s) {
    if (M <= 0) return cudaSuccess;
    k_rope_append_f32<<<M, 256, 0, s>>>(qkv_q, qkv_k, qkv_v, q_out, kc, vc, T, n_heads, n_kv_heads, head_dim, kv_seq,
                                        start_pos, pos_dev, max_pos, cos_tab, sin_tab, err);
    return cudaGetLastError();
}

cudaError_t launch_embed(const int32_t* ids, int n, const void* w, int vocab, int d, void* x, int32_t* err,
                         cudaStream_t s) {
    if (n <= 0) return cudaSuccess;
    k_embed<bf16><<<n, 256, 0, s>>>(ids, (const bf16*)w, (bf16*)x, vocab, d, err);
    return cudaGetLastError();
}

cudaError_t launch_argmax_rows(const float* logits, int rows, int vocab, int32_t* ids, cudaStream_t s) {
    if (rows <= 0) return cudaSuccess;
    k_argmax_rows<<<rows, 1024, 0, s>>>(logits, vocab, ids);
    return cudaGetLastError();
}

}  // namespace llama
