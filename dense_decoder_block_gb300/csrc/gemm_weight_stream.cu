// Weight-streaming (decode, M <= 32) instantiations of the persistent tcgen05 projection kernel.
#include "gemm_ws.cuh"

namespace llama {

LLAMA_TRACE_UNIT(gemm_ws)

template <int BN, bool DUAL, int EPI>
static cudaError_t run_ws(const GemmProblem& p, const GemmKArgs& ka, const CUtensorMap& a0, const CUtensorMap& a1,
                          const CUtensorMap& a2, const bf16* x, cudaStream_t s) {
    using C = WsCfg<BN, DUAL>;
    auto kern = k_gemm_ws<BN, DUAL, EPI>;
    cudaError_t r = kernel_setup_once((const void*)kern, [](const void* k) {
        return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    });
    if (r != cudaSuccess) return r;
    CUtensorMap mb;
    if (!make_tmap_bf16(&mb, x, (uint64_t)p.M, (uint64_t)p.K, BN, nullptr)) return cudaErrorInvalidValue;
    const int n_sm = device_sm_count();
    const int units = (p.F / kTileF) * ka.n_segs;
    dim3 grid(units < n_sm ? units : n_sm);
    return launch_pdl(kern, grid, dim3(kGemmThreads), C::SMEM_BYTES, s, a0, a1, a2, mb, ka);
}

template <int BN>
static cudaError_t dispatch_ws(const GemmProblem& p, const GemmKArgs& ka, const CUtensorMap& a0,
                               const CUtensorMap& a1, const CUtensorMap& a2, const bf16* x, cudaStream_t s) {
    if (p.dual) {
        if (ka.e.kind != EPI_SWIGLU) return cudaErrorInvalidValue;
        return run_ws<BN, true, EPI_SWIGLU>(p, ka, a0, a1, a2, x, s);
    }
    switch (ka.e.kind) {
        case EPI_QKV: return run_ws<BN, false, EPI_QKV>(p, ka, a0, a1, a2, x, s);
        case EPI_RESID: return run_ws<BN, false, EPI_RESID>(p, ka, a0, a1, a2, x, s);
        case EPI_PLAIN: return run_ws<BN, false, EPI_PLAIN>(p, ka, a0, a1, a2, x, s);
        case EPI_LOGITS: return run_ws<BN, false, EPI_LOGITS>(p, ka, a0, a1, a2, x, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_weight_stream(const GemmProblem& p, const GemmKArgs& ka, const CUtensorMap& a0,
                                 const CUtensorMap& a1, const CUtensorMap& a2, const bf16* x, cudaStream_t s) {
    if (p.M <= 16) return dispatch_ws<16>(p, ka, a0, a1, a2, x, s);
    return dispatch_ws<32>(p, ka, a0, a1, a2, x, s);
}

}  // namespace llama
