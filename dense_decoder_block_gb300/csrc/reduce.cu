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
#include <algorithm>

#include "internal.h"
#include "reduce_epi.cuh"

namespace llama {

namespace {

constexpr int kThreads = 256;

// Lets the next kernel launch, then waits for the projection.  The trigger comes
// before the wait: what follows a reduction (attention, a projection, RMSNorm)
// reads nothing before its own wait that a kernel still running may write, and its
// CTAs take the SMs as the projection's CTAs leave them instead of after this
// kernel's release.  Returns the time the wait returned (for the optional timeline).
__device__ __forceinline__ unsigned long long griddep() {
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    return trace_stamp();
}

// What a reduction reads before griddepcontrol.wait -- the position, the RoPE
// tables, gains and the residual input -- is never written by the kernel it
// overlaps: a reduction starts only after its projection passed its own wait, so
// everything two or more launches back is complete and visible.
// The residual of each reduction is produced at least two launches earlier (the
// block input, or h four launches before the last reduction).

// 320 threads of at most 48 registers (15,360 per CTA), one item per thread and a
// grid of at most one CTA per SM (threads loop over the items beyond 320 per SM):
// every CTA fits beside a CTA of the QKV projection, so all of them start while the
// projection runs and the attention kernel behind them launches before the
// projection ends, and an attention CTA (192 threads x 256 registers, 49,152) fits
// beside the one reduction CTA of an SM, so the attention streams its older K/V
// chunks while the reduction runs.
constexpr int kQkvThreads = 320;

__global__ void __launch_bounds__(kQkvThreads, 4) k_reduce_qkv(const ReduceArgs r) {
    TRACE(const unsigned long long tr0 = trace_stamp();)
    const int F4 = r.F / 4;
    const int n_items = r.M * F4;
    int idx = blockIdx.x * kQkvThreads + threadIdx.x;
    bool live = idx < n_items;
    int n = live ? idx / F4 : 0, f0 = live ? (idx - n * F4) * 4 : 0;
    Qkv4 p{};
    if (live) p = epi4_qkv_prepare(r.e, n, f0);
    TRACE(const unsigned long long tr1 =) griddep();
    while (live) {
        float4 s, unused;
        seg_sum4<false, 4>(r.partial, (size_t)r.M * r.F, r.n_segs, (size_t)n * r.F + f0, 0, s, unused);
        epi4_qkv_apply(p, s);
        idx += gridDim.x * kQkvThreads;
        live = idx < n_items;
        if (live) {
            n = idx / F4;
            f0 = (idx - n * F4) * 4;
            p = epi4_qkv_prepare(r.e, n, f0);
        }
    }
    TRACE(trace_cta(TR_REDUCE_QKV, tr0, tr1);)
}

__global__ void __launch_bounds__(kThreads, 4) k_reduce_resid(const ReduceArgs r) {
    TRACE(const unsigned long long tr0 = trace_stamp();)
    const int F4 = r.F / 4;
    const int idx = blockIdx.x * kThreads + threadIdx.x;
    const bool live = idx < r.M * F4;
    const int n = live ? idx / F4 : 0, f0 = live ? (idx - n * F4) * 4 : 0;
    const size_t off = (size_t)n * r.F + f0;
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
    if (live) x = load4_bf16(r.e.resid + off);
    TRACE(const unsigned long long tr1 =) griddep();
    if (!live) return;
    float4 s, unused;
    seg_sum4<false, 8>(r.partial, (size_t)r.M * r.F, r.n_segs, off, 0, s, unused);
    epi4_resid(r.e, r.F, n, f0, x, s);
    TRACE(trace_cta(TR_REDUCE_RESID, tr0, tr1);)
}

__global__ void __launch_bounds__(kThreads, 3) k_reduce_swiglu(const ReduceArgs r) {
    TRACE(const unsigned long long tr0 = trace_stamp();)
    TRACE(const unsigned long long tr1 =) griddep();
    const int F4 = r.F / 4;
    const int idx = blockIdx.x * kThreads + threadIdx.x;
    if (idx >= r.M * F4) return;
    const int n = idx / F4, f0 = (idx - n * F4) * 4;
    const size_t off = (size_t)n * r.F + f0;
    const size_t plane = (size_t)r.M * r.F;                  // [seg][gate|up][M][F]
    float4 g, u;
    seg_sum4<true, 4>(r.partial, 2 * plane, r.n_segs, off, plane + off, g, u);
    epi4_swiglu(r.e, r.F, n, f0, g, u);
    TRACE(trace_cta(TR_REDUCE_SWIGLU, tr0, tr1);)
}

// h = resid epilogue, then RMSNorm(h), one cluster of S CTAs per token row: CTA c
// holds the row's slice c (elements c*512 + t and c*512 + t + 256 of thread t),
// computes its slice's sum of squares with rms_tree_256, sends it to every CTA of
// the cluster through distributed shared memory, and after one cluster barrier
// each CTA adds the S slice sums in slice order -- the definition k_rmsnorm uses
// for widths that are multiples of 512.
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void st_cluster_f32(const float* local_addr, uint32_t rank, float v) {
    uint32_t a = (uint32_t)__cvta_generic_to_shared(local_addr), ra;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(rank));
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(ra), "f"(v) : "memory");
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

template <int S>
__global__ void __launch_bounds__(kThreads) k_reduce_resid_norm(const ReduceArgs r, const bf16* __restrict__ gain,
                                                                bf16* __restrict__ hn, float eps) {
    __shared__ float red[8];
    __shared__ float slice_sum[S];
    TRACE(const unsigned long long tr0 = trace_stamp();)
    const int c = (int)cluster_ctarank(), n = blockIdx.y, tid = threadIdx.x;
    const int d = r.F;
    const size_t plane = (size_t)r.M * r.F;
    const size_t row = (size_t)n * d;
    const int i0 = c * 512 + tid, i1 = i0 + 256;
    // the block input and the gains are not written by the kernels this one overlaps
    const float x0 = __bfloat162float(__ldcg(r.e.resid + row + i0));
    const float x1 = __bfloat162float(__ldcg(r.e.resid + row + i1));
    const float g0 = __bfloat162float(gain[i0]), g1 = __bfloat162float(gain[i1]);
    TRACE(const unsigned long long tr1 =) griddep();
    float a0 = -0.f, a1 = -0.f;   // -0 + x == x: the sums equal ((s0 + s1) + s2) + ...
    for (int s0 = 0; s0 < r.n_segs; s0 += 8) {
        float w0[8], w1[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (s0 + i < r.n_segs) {
                w0[i] = __ldcg(r.partial + (size_t)(s0 + i) * plane + row + i0);
                w1[i] = __ldcg(r.partial + (size_t)(s0 + i) * plane + row + i1);
            }
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (s0 + i < r.n_segs) {
                a0 = __fadd_rn(a0, w0[i]);
                a1 = __fadd_rn(a1, w1[i]);
            }
    }
    const bf16 hb0 = __float2bfloat16_rn(epi_resid(x0, a0));
    const bf16 hb1 = __float2bfloat16_rn(epi_resid(x1, a1));
    r.e.out[row + i0] = hb0;
    r.e.out[row + i1] = hb1;
    const float h0 = __bfloat162float(hb0), h1 = __bfloat162float(hb1);
    const float part = rms_tree_256(rms_slice_sq(h0, h1), red);
    if (tid < S) st_cluster_f32(&slice_sum[c], (uint32_t)tid, part);   // to every CTA of the cluster
    cluster_sync();
    float total = slice_sum[0];
#pragma unroll
    for (int k = 1; k < S; ++k) total = __fadd_rn(total, slice_sum[k]);
    const float scale = rms_scale(total, d, eps);
    hn[row + i0] = __float2bfloat16_rn(__fmul_rn(bf16_round(__fmul_rn(h0, scale)), g0));
    hn[row + i1] = __float2bfloat16_rn(__fmul_rn(bf16_round(__fmul_rn(h1, scale)), g1));
    TRACE(trace_cta(TR_REDUCE_RESID_NORM, tr0, tr1);)
}

dim3 grid4(const ReduceArgs& r) { return dim3((unsigned)(((size_t)r.M * (r.F / 4) + kThreads - 1) / kThreads)); }

}  // namespace

LLAMA_TRACE_UNIT(reduce)

cudaError_t launch_reduce(const ReduceArgs& r, int kind, cudaStream_t s) {
    if (r.M <= 0) return cudaSuccess;
    if (r.F % 4) return cudaErrorInvalidValue;
    auto kern = kind == EPI_QKV ? k_reduce_qkv : kind == EPI_RESID ? k_reduce_resid : kind == EPI_SWIGLU ? k_reduce_swiglu
                                                                                                     : nullptr;
    if (!kern) return cudaErrorInvalidValue;
    cudaError_t e = kernel_setup_once((const void*)kern, setup_prefer_shared);
    if (e != cudaSuccess) return e;
    if (kind == EPI_QKV) {   // one item per thread, at most one CTA per SM
        const long need = ((long)r.M * (r.F / 4) + kQkvThreads - 1) / kQkvThreads;
        return launch_pdl(kern, dim3((unsigned)std::min(need, (long)device_sm_count())), dim3(kQkvThreads), 0, s, r);
    }
    return launch_pdl(kern, grid4(r), dim3(kThreads), 0, s, r);
}

// The widths whose k_rmsnorm uses the slice definition (d / 256 in {4, 8, 16, 32}).
bool reduce_resid_norm_supported(int d) {
    return d % 512 == 0 && (d / 512 == 2 || d / 512 == 4 || d / 512 == 8 || d / 512 == 16);
}

template <int S>
static cudaError_t launch_resid_norm(const ReduceArgs& r, const void* gain, void* hn, float eps, cudaStream_t s) {
    auto kern = k_reduce_resid_norm<S>;
    cudaError_t e = kernel_setup_once((const void*)kern, [](const void* k) {
        cudaError_t r = setup_prefer_shared(k);
        if (r == cudaSuccess && S > 8) r = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        return r;
    });
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(S, r.M);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = S;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, r, (const bf16*)gain, (bf16*)hn, eps);
}

cudaError_t launch_reduce_resid_norm(const ReduceArgs& r, const void* gain, void* hn, float eps, cudaStream_t s) {
    if (r.M <= 0) return cudaSuccess;
    switch (r.F / 512) {
        case 2: return launch_resid_norm<2>(r, gain, hn, eps, s);
        case 4: return launch_resid_norm<4>(r, gain, hn, eps, s);
        case 8: return launch_resid_norm<8>(r, gain, hn, eps, s);
        case 16: return launch_resid_norm<16>(r, gain, hn, eps, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace llama
