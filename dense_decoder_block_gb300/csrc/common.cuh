// Shared device/host definitions of the block library (not part of the public ABI).
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <utility>

#include "../../include/llama_block.h"

namespace llama {

using bf16 = __nv_bfloat16;

// Keys per attention chunk: the unit of the softmax partial (m, l, o) that both
// the prefill and the decode attention kernels produce and fold in ascending order.
constexpr int kAttnChunk = 128;
// K-segment length (elements) of every bf16 projection: each output is the
// ascending fp32 sum of per-segment tensor-core accumulations of this length,
// in prefill and decode alike.
constexpr int kSegK = 1024;
constexpr int kRopeMaxPairs = 64;   // head_dim <= 128
// Floats per decode attention chunk partial of one query row: o[head_dim], m, l, 2 pad.
__host__ __device__ constexpr int part_stride(int head_dim) { return head_dim + 4; }
constexpr int kPartStride = part_stride(128);

__device__ __forceinline__ float bf16_round(float v) { return __bfloat162float(__float2bfloat16_rn(v)); }
__device__ __forceinline__ float ld_bf16(const bf16* p) { return __bfloat162float(*p); }

__device__ __forceinline__ void record_error(int* err, int code) {
    if (err) atomicCAS(err, 0, code);
}

// RMSNorm row scale 1/sqrt(ss/d + eps), correctly rounded steps.
__device__ __forceinline__ float rms_scale(float sumsq, int d, float eps) {
    float ms = __fdiv_rn(sumsq, (float)d);
    return __frcp_rn(__fsqrt_rn(__fadd_rn(ms, eps)));
}

// Adjacent-pair rotation of one element: this thread holds `self` at an even
// (first) or odd (second) index of the pair, `other` is its partner.
//   first:  a' = a cos - b sin      second: b' = a sin + b cos
__device__ __forceinline__ float rope_rotate_elem(float self, float other, float c, float s, bool second) {
    return second ? __fmaf_rn(other, s, __fmul_rn(self, c)) : __fmaf_rn(self, c, __fmul_rn(-other, s));
}

// SiLU(z) = z / (1 + e^-z)
__device__ __forceinline__ float silu_f(float z) { return __fdiv_rn(z, __fadd_rn(1.0f, expf(-z))); }

// Epilogue arithmetic shared by every schedule (fused GEMM epilogues and the
// decode segment reductions), so both produce the same bits.
// Residual: bf16(x + bf16(branch)).
__device__ __forceinline__ float epi_resid(float x, float acc) { return __fadd_rn(x, bf16_round(acc)); }
// SwiGLU: bf16(silu(bf16(gate))) * bf16(up), to be rounded by the caller.
__device__ __forceinline__ float epi_swiglu(float gate_acc, float up_acc) {
    const float g = bf16_round(gate_acc);
    const float u = bf16_round(up_acc);
    return __fmul_rn(bf16_round(silu_f(g)), u);
}

// RMSNorm sum-of-squares tree for a 256-thread CTA: each thread's partial (its
// elements tid, tid+256, ... in ascending order), a butterfly inside each warp
// read at lane 0, then the 8 warps in ascending order.  `red` is 8 floats of
// shared memory.  Returns the row total in every thread.
__device__ __forceinline__ float rms_tree_256(float ss, float* red) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, off));
    __syncthreads();   // red may still be read from a previous use
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    float t = red[0];
#pragma unroll
    for (int w = 1; w < 8; ++w) t = __fadd_rn(t, red[w]);
    return t;
}

// RMSNorm sum of squares of a row of S * 512 elements, as every kernel computes it
// when the width is a multiple of 512 (at most 16 slices): the row is cut into
// slices of 512; in slice c thread t (of 256) holds elements c*512 + t and
// c*512 + t + 256 -- v[2c] and v[2c+1], the same ownership as i = t + 256 e --
// and squares them as fma(v1, v1, v0 * v0); each slice is reduced by the tree of
// rms_tree_256 and the slice sums are added in slice order.  A kernel spread over
// S CTAs (one slice each) reproduces it with rms_tree_256 per slice.
__device__ __forceinline__ float rms_slice_sq(float v0, float v1) { return __fmaf_rn(v1, v1, __fmul_rn(v0, v0)); }
template <int S>
__device__ __forceinline__ float rms_sumsq_slices(const float* v, float* red /* [S * 8] */) {
    float p[S];
#pragma unroll
    for (int c = 0; c < S; ++c) {
        p[c] = rms_slice_sq(v[2 * c], v[2 * c + 1]);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) p[c] = __fadd_rn(p[c], __shfl_xor_sync(0xffffffffu, p[c], off));
    }
    __syncthreads();   // red may still be read from a previous use
    if ((threadIdx.x & 31) == 0)
#pragma unroll
        for (int c = 0; c < S; ++c) red[c * 8 + (threadIdx.x >> 5)] = p[c];
    __syncthreads();
    float total = 0.f;
#pragma unroll
    for (int c = 0; c < S; ++c) {
        float t = red[c * 8];
#pragma unroll
        for (int w = 1; w < 8; ++w) t = __fadd_rn(t, red[c * 8 + w]);
        total = (c == 0) ? t : __fadd_rn(total, t);
    }
    return total;
}

// Launch with programmatic stream serialization: the kernel may begin while the
// previous kernel on the stream drains.  Every kernel of the library calls
// griddepcontrol.wait before it reads anything an earlier kernel wrote; when the
// wait returns, every earlier kernel has completed (none completes before its own
// wait returns).  The projection and attention kernels let their dependents start
// (griddepcontrol.launch_dependents) only after that wait, so a kernel that
// follows one of them starts only once everything two places back has completed:
// the reductions read positions, gains and residuals before their wait on that
// ground.  The row-wise kernels (RMSNorm, RoPE, the segment reductions, the
// attention combine) trigger before their wait: the kernel after each (a
// projection or attention) reads only weights, positions and older KV-cache rows
// before its own wait, none of which a kernel still running writes.  A kernel
// that allocates tensor memory triggers only after its allocation: a dependent
// CTA that started earlier on the same SM could otherwise hold the columns while
// it waits for this grid.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// ---------------------------------------------------------------- per-CTA timeline (trace builds)
// In a library built with LLAMA_TRACE, while llama_trace_begin is in effect each
// CTA of the block's step kernels writes one record when its thread 0 finishes:
// {kernel | smid << 16 | cta << 32, %globaltimer at the CTA's start, after its
// grid-dependency wait (0 where the recording thread does not wait), at thread
// 0's end}.  In the product build every hook below compiles to nothing.  The
// control word lives in each translation unit's constant bank (no relocatable
// device code), so every unit with traced kernels has a setter (LLAMA_TRACE_UNIT)
// and llama_trace_begin sets them all.
enum TraceKernel : unsigned int {
    TR_RMSNORM = 1, TR_GEMM_WS = 2, TR_GEMM_TT = 3, TR_REDUCE_QKV = 4, TR_REDUCE_RESID = 5, TR_REDUCE_SWIGLU = 6,
    TR_REDUCE_RESID_NORM = 7, TR_ATTN_DEC = 8, TR_ATTN_COMBINE = 9, TR_ATTN_PF = 10, TR_ROPE = 11, TR_ATTN_WIDE = 12,
};
struct TraceCtl {
    unsigned long long* recs;   // [capacity][4]
    unsigned int* count;        // records claimed (may exceed capacity: the extra ones are dropped)
    unsigned int capacity;
};
__device__ __forceinline__ unsigned long long trace_clock() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// TRACE(statement): the statement in trace builds, nothing in the product build
#ifdef LLAMA_TRACE
#define TRACE(...) __VA_ARGS__
#else
#define TRACE(...)
#endif
#ifdef LLAMA_TRACE
static __constant__ TraceCtl g_trace;
#define LLAMA_TRACE_ON (g_trace.recs != nullptr)
#define LLAMA_TRACE_UNIT(name)                                                  \
    cudaError_t trace_set_##name(const TraceCtl& c) {                           \
        return cudaMemcpyToSymbol(g_trace, &c, sizeof(c));                      \
    }
#else
#define LLAMA_TRACE_ON false
#define LLAMA_TRACE_UNIT(name)                                                  \
    cudaError_t trace_set_##name(const TraceCtl&) { return cudaErrorNotSupported; }
#endif
// %globaltimer for thread 0 while tracing is on, else 0 (no timer read)
__device__ __forceinline__ unsigned long long trace_stamp() {
    return (LLAMA_TRACE_ON && threadIdx.x == 0) ? trace_clock() : 0ull;
}
// thread 0 of the CTA, at its end: `kernel` is a TraceKernel, optionally with the
// epilogue kind in bits 8..11 and bit 12 for a split token-tiled projection
__device__ __forceinline__ void trace_cta(unsigned int kernel, unsigned long long t_start,
                                          unsigned long long t_release) {
#ifdef LLAMA_TRACE
    if (threadIdx.x != 0 || !LLAMA_TRACE_ON) return;
    const TraceCtl c = g_trace;
    const unsigned int i = atomicAdd(c.count, 1u);
    if (i >= c.capacity) return;
    unsigned int smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    const unsigned long long cta =
        blockIdx.x + (unsigned long long)gridDim.x * (blockIdx.y + (unsigned long long)gridDim.y * blockIdx.z);
    unsigned long long* r = c.recs + 4ull * i;
    r[0] = (unsigned long long)(kernel & 0xffffu) | ((unsigned long long)(smid & 0xffffu) << 16) | (cta << 32);
    r[1] = t_start;
    r[2] = t_release;
    r[3] = trace_clock();
#else
    (void)kernel;
    (void)t_start;
    (void)t_release;
#endif
}

}  // namespace llama
