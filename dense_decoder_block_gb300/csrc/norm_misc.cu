// RMSNorm, the fp32 (CUDA-core) projection path, embedding gather and row argmax.
#include <cfloat>

#include "internal.h"
#include "ptx.cuh"

namespace llama {

namespace {

constexpr int kNormThreads = 256;

__device__ __forceinline__ float to_f(bf16 v) { return __bfloat162float(v); }
__device__ __forceinline__ float to_f(float v) { return v; }

// "Llama 3.1 70B", RMSNorm reference implementation: fp32 mean of squares,
// eps inside the square root, the scaled row cast to the trunk dtype before the
// gain multiplies it.  One 256-thread CTA per row; thread t owns elements
// t, t+256, ... (kept in registers when d/256 is a small power of two).  The sum
// of squares follows the library's one definition for the width (common.cuh:
// 512-element slices when d is a multiple of 512, else one chain per thread and
// rms_tree_256), which the decode reduction fused with RMSNorm reproduces, so
// prefill and decode rows agree bit for bit.
template <typename T, int EPT>
__global__ void __launch_bounds__(kNormThreads) k_rmsnorm(const T* __restrict__ x, const T* __restrict__ g,
                                                          T* __restrict__ y, int d, float eps) {
    __shared__ float red[16 * 8];
    TRACE(const unsigned long long tr0 = trace_stamp();)
    // the projection after RMSNorm reads only its weights before its own wait
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    TRACE(const unsigned long long tr1 = trace_stamp();)
    const int row = blockIdx.x, tid = threadIdx.x;
    const T* xr = x + (size_t)row * d;
    T* yr = y + (size_t)row * d;
    if constexpr (EPT > 0) {
        float v[EPT];
#pragma unroll
        for (int e = 0; e < EPT; ++e) v[e] = to_f(xr[tid + kNormThreads * e]);
        float sumsq;
        if constexpr (EPT >= 4 && EPT % 2 == 0 && EPT / 2 <= 16) {
            sumsq = rms_sumsq_slices<EPT / 2>(v, red);   // width a multiple of 512
        } else {
            float ss = 0.f;
#pragma unroll
            for (int e = 0; e < EPT; ++e) ss = __fmaf_rn(v[e], v[e], ss);
            sumsq = rms_tree_256(ss, red);
        }
        const float r = rms_scale(sumsq, d, eps);
#pragma unroll
        for (int e = 0; e < EPT; ++e) {
            const int i = tid + kNormThreads * e;
            if constexpr (sizeof(T) == 2)
                yr[i] = __float2bfloat16_rn(__fmul_rn(bf16_round(__fmul_rn(v[e], r)), to_f(g[i])));
            else
                yr[i] = __fmul_rn(__fmul_rn(v[e], r), to_f(g[i]));
        }
    } else {
        float ss = 0.f;
        for (int i = tid; i < d; i += kNormThreads) {
            const float v = to_f(xr[i]);
            ss = __fmaf_rn(v, v, ss);
        }
        const float r = rms_scale(rms_tree_256(ss, red), d, eps);
        for (int i = tid; i < d; i += kNormThreads) {
            const float v = to_f(xr[i]);
            if constexpr (sizeof(T) == 2)
                yr[i] = __float2bfloat16_rn(__fmul_rn(bf16_round(__fmul_rn(v, r)), to_f(g[i])));
            else
                yr[i] = __fmul_rn(__fmul_rn(v, r), to_f(g[i]));
        }
    }
    TRACE(trace_cta(TR_RMSNORM, tr0, tr1);)
}

template <typename K, typename... Args>
cudaError_t launch_small(K kern, dim3 grid, dim3 block, cudaStream_t s, Args... args) {
    cudaError_t r = kernel_setup_once((const void*)kern, setup_prefer_shared);
    if (r != cudaSuccess) return r;
    return launch_pdl(kern, grid, block, 0, s, args...);
}

template <typename T>
cudaError_t rmsnorm_dispatch(const T* x, const T* g, T* y, int rows, int d, float eps, cudaStream_t s) {
    const dim3 grid(rows), block(kNormThreads);
    if (d % kNormThreads == 0) {
        switch (d / kNormThreads) {
            case 1: return launch_small(k_rmsnorm<T, 1>, grid, block, s, x, g, y, d, eps);
            case 2: return launch_small(k_rmsnorm<T, 2>, grid, block, s, x, g, y, d, eps);
            case 4: return launch_small(k_rmsnorm<T, 4>, grid, block, s, x, g, y, d, eps);
            case 8: return launch_small(k_rmsnorm<T, 8>, grid, block, s, x, g, y, d, eps);
            case 16: return launch_small(k_rmsnorm<T, 16>, grid, block, s, x, g, y, d, eps);
            case 32: return launch_small(k_rmsnorm<T, 32>, grid, block, s, x, g, y, d, eps);
            default: break;
        }
    }
    return launch_small(k_rmsnorm<T, 0>, grid, block, s, x, g, y, d, eps);
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

// RoPE in place on bf16 rows of 128 (q rows, then the cache rows of k): one
// thread per 8 elements (4 pairs) of kRopeRows rows of the same token -- the
// rotation of those pairs read once from the tables, the rows' 16-byte loads
// issued together, rope_rotate_elem on the bf16 values (the inputs the fused
// epilogue rotates), 16-byte stores.
constexpr int kRopeRows = 4;
__global__ void __launch_bounds__(256) k_rope_inplace(bf16* __restrict__ q, bf16* __restrict__ kc, int M, int T,
                                                      int n_heads, int n_kv_heads, int kv_seq, int start_pos,
                                                      const int* pos_dev, int max_pos,
                                                      const float* __restrict__ cos_tab,
                                                      const float* __restrict__ sin_tab, int* err) {
    TRACE(const unsigned long long tr0 = trace_stamp();)
    // the prefill attention after RoPE reads nothing before its own wait
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    TRACE(const unsigned long long tr1 = trace_stamp();)
    const int n_rows = n_heads + n_kv_heads;                     // 128-wide rows per token
    const int n_grp = (n_rows + kRopeRows - 1) / kRopeRows;      // row groups per token
    const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (long long)M * n_grp * 16) return;
    const int g8 = (int)(idx & 15);                              // 8-element group of the row
    const long long rest = idx >> 4;
    const int n = (int)(rest / n_grp), grp = (int)(rest - (long long)n * n_grp);
    const int b = n / T, t = n - b * T;
    const int pos = (pos_dev ? *pos_dev : start_pos) + t;
    if (pos < 0 || pos >= max_pos) {
        record_error(err, LLAMA_ERR_POS_RANGE);
        return;
    }
    const float4 c = *reinterpret_cast<const float4*>(cos_tab + (size_t)pos * kRopeMaxPairs + g8 * 4);
    const float4 sn = *reinterpret_cast<const float4*>(sin_tab + (size_t)pos * kRopeMaxPairs + g8 * 4);
    const float cv[4] = {c.x, c.y, c.z, c.w}, sv[4] = {sn.x, sn.y, sn.z, sn.w};
    uint4* p[kRopeRows];
    uint4 u[kRopeRows];
#pragma unroll
    for (int r = 0; r < kRopeRows; ++r) {
        const int head = grp * kRopeRows + r;
        p[r] = nullptr;
        if (head < n_rows) {
            bf16* row = head < n_heads ? q + (size_t)n * n_heads * 128 + (size_t)head * 128
                                       : kc + (((size_t)b * n_kv_heads + (head - n_heads)) * kv_seq + pos) * 128;
            p[r] = reinterpret_cast<uint4*>(row + g8 * 8);
            u[r] = *p[r];
        }
    }
#pragma unroll
    for (int r = 0; r < kRopeRows; ++r) {
        if (p[r] == nullptr) continue;
        uint32_t* w = reinterpret_cast<uint32_t*>(&u[r]);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const __nv_bfloat162 pr = *reinterpret_cast<const __nv_bfloat162*>(&w[k]);
            const float a0 = __low2float(pr), a1 = __high2float(pr);
            const __nv_bfloat162 o = __floats2bfloat162_rn(rope_rotate_elem(a0, a1, cv[k], sv[k], false),
                                                           rope_rotate_elem(a1, a0, cv[k], sv[k], true));
            w[k] = *reinterpret_cast<const uint32_t*>(&o);
        }
        *p[r] = u[r];
    }
    TRACE(trace_cta(TR_ROPE, tr0, tr1);)
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

// argmax over one row of fp32 logits; ties go to the lowest index.  If the
// projection that wrote the logits recorded an error in *err (a bounded wait
// expired), the row's id is that (negative) code instead.
//
// One cluster of kArgmaxSplit CTAs per row: CTA c scans the c-th contiguous slice
// of the row with 16-byte loads, eight in flight per thread, and sends its
// (maximum, first index) to CTA 0 of the cluster through distributed shared
// memory.  (One CTA per row left 32 rows of 128,256 logits on 32 SMs, bound by
// load latency at 63 us.)
constexpr int kArgmaxSplit = 8;
constexpr int kArgmaxThreads = 512;

__device__ __forceinline__ void better(float& best, int& bi, float ov, int oi) {
    if (ov > best || (ov == best && oi < bi)) { best = ov; bi = oi; }
}

__global__ void __launch_bounds__(kArgmaxThreads) k_argmax_rows(const float* __restrict__ logits, int vocab,
                                                                int32_t* __restrict__ ids,
                                                                const int* __restrict__ err) {
    __shared__ float sv[kArgmaxThreads / 32];
    __shared__ int si[kArgmaxThreads / 32];
    __shared__ float cv[kArgmaxSplit];
    __shared__ int ci[kArgmaxSplit];
    uint32_t c;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(c));
    const int row = blockIdx.x / kArgmaxSplit, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float* lr = logits + (size_t)row * vocab;
    const int per = (vocab + 4 * kArgmaxSplit - 1) / (4 * kArgmaxSplit) * 4;   // slice length, 4-aligned
    const int lo = min(vocab, (int)c * per), hi = min(vocab, lo + per);
    asm volatile("griddepcontrol.wait;" ::: "memory");
    float best = -INFINITY;
    int bi = INT32_MAX;
    auto take = [&](int i, float v) {
        if (v > best) { best = v; bi = i; }   // ascending i per thread: the first maximum stays
    };
    if ((vocab & 3) == 0 && ((uintptr_t)lr & 15) == 0) {
        const float4* l4 = reinterpret_cast<const float4*>(lr);
        const int e4 = hi >> 2, step = kArgmaxThreads;
        int i = (lo >> 2) + tid;
        for (; i + 7 * step < e4; i += 8 * step) {
            float4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) v[u] = __ldg(l4 + i + u * step);
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int e = 4 * (i + u * step);
                take(e, v[u].x);
                take(e + 1, v[u].y);
                take(e + 2, v[u].z);
                take(e + 3, v[u].w);
            }
        }
        for (; i < e4; i += step) {
            const float4 v = __ldg(l4 + i);
            take(4 * i, v.x);
            take(4 * i + 1, v.y);
            take(4 * i + 2, v.z);
            take(4 * i + 3, v.w);
        }
    } else {
        for (int i = lo + tid; i < hi; i += kArgmaxThreads) take(i, __ldg(lr + i));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        better(best, bi, __shfl_xor_sync(0xffffffffu, best, off), __shfl_xor_sync(0xffffffffu, bi, off));
    if (lane == 0) { sv[warp] = best; si[warp] = bi; }
    __syncthreads();
    if (tid == 0) {
        for (int w = 1; w < kArgmaxThreads / 32; ++w) better(best, bi, sv[w], si[w]);
        // this slice's result into slot c of CTA 0
        uint32_t av = (uint32_t)__cvta_generic_to_shared(&cv[c]), ai = (uint32_t)__cvta_generic_to_shared(&ci[c]);
        uint32_t rv, ri;
        asm volatile("mapa.shared::cluster.u32 %0, %1, 0;" : "=r"(rv) : "r"(av));
        asm volatile("mapa.shared::cluster.u32 %0, %1, 0;" : "=r"(ri) : "r"(ai));
        asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(rv), "f"(best) : "memory");
        asm volatile("st.shared::cluster.s32 [%0], %1;" ::"r"(ri), "r"(bi) : "memory");
    }
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
    if (c == 0 && tid == 0) {
        best = cv[0];
        bi = ci[0];
        for (int k = 1; k < kArgmaxSplit; ++k) better(best, bi, cv[k], ci[k]);
        const int code = err ? *err : 0;
        ids[row] = code != 0 ? code : (bi == INT32_MAX) ? 0 : bi;
    }
}

// Failure-path self-test: one warp waits, through the same bounded wait every
// tcgen05 kernel uses, on an mbarrier that nothing arrives on.  The wait gives up
// after budget_ns, records LLAMA_ERR_DEVICE_TIMEOUT in *err, and the kernel
// returns -- no trap, no fault; the context stays usable.
__global__ void k_expire_wait(int* err, unsigned long long budget_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        ptx::mbar_init(&bar, 1);
        ptx::fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) (void)ptx::mbar_wait_for(&bar, 0, err, budget_ns);
}

}  // namespace

LLAMA_TRACE_UNIT(norm)

cudaError_t launch_rmsnorm(const void* x, const void* g, void* y, int rows, int d, float eps, int dtype,
                           cudaStream_t s) {
    if (rows <= 0) return cudaSuccess;
    if (dtype == LLAMA_BF16) return rmsnorm_dispatch((const bf16*)x, (const bf16*)g, (bf16*)y, rows, d, eps, s);
    return rmsnorm_dispatch((const float*)x, (const float*)g, (float*)y, rows, d, eps, s);
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

cudaError_t launch_rope_inplace(void* q, void* kc, int M, int T, int n_heads, int n_kv_heads, int kv_seq,
                                int start_pos, const int* pos_dev, int max_pos, const float* cos_tab,
                                const float* sin_tab, int* err, cudaStream_t s) {
    if (M <= 0) return cudaSuccess;
    const long long threads = (long long)M * ((n_heads + n_kv_heads + kRopeRows - 1) / kRopeRows) * 16;
    const dim3 grid((unsigned)((threads + 255) / 256));
    return launch_small(k_rope_inplace, grid, dim3(256), s, (bf16*)q, (bf16*)kc, M, T, n_heads, n_kv_heads,
                      kv_seq, start_pos, pos_dev, max_pos, cos_tab, sin_tab, err);
}

cudaError_t launch_embed(const int32_t* ids, int n, const void* w, int vocab, int d, void* x, int32_t* err,
                         cudaStream_t s) {
    if (n <= 0) return cudaSuccess;
    k_embed<bf16><<<n, 256, 0, s>>>(ids, (const bf16*)w, (bf16*)x, vocab, d, err);
    return cudaGetLastError();
}

cudaError_t launch_expire_wait(int* err, unsigned long long budget_ns, cudaStream_t s) {
    k_expire_wait<<<1, 32, 0, s>>>(err, budget_ns);
    return cudaGetLastError();
}

cudaError_t launch_argmax_rows(const float* logits, int rows, int vocab, int32_t* ids, const int* err,
                               cudaStream_t s) {
    if (rows <= 0) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)rows * kArgmaxSplit);
    cfg.blockDim = dim3(kArgmaxThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = kArgmaxSplit;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, k_argmax_rows, logits, vocab, ids, err);
}

}  // namespace llama
