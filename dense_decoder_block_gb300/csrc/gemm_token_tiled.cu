// Token-tiled (prefill) instantiations of the persistent tcgen05 projection kernel.
#include <algorithm>

#include "gemm_tt.cuh"

namespace llama {

LLAMA_TRACE_UNIT(gemm_tt)

template <int BN, bool DUAL, int EPI>
static cudaError_t run_tt(const GemmProblem& p, const GemmKArgs& ka, const CUtensorMap& a0, const CUtensorMap& a1,
                          const CUtensorMap& a2, const bf16* x, cudaStream_t s) {
    using C = TtCfg<BN, DUAL>;
    auto kern = k_gemm_tt<BN, DUAL, EPI>;
    cudaError_t r = kernel_setup_once((const void*)kern, [](const void* k) {
        // The register split inside the kernel must fit the block's launch allocation.
        cudaFuncAttributes fa;
        cudaError_t e = cudaFuncGetAttributes(&fa, k);
        if (e != cudaSuccess) return e;
        if (fa.numRegs * C::THREADS < C::REGS_NEEDED) return cudaErrorInvalidConfiguration;
        return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    });
    if (r != cudaSuccess) return r;
    CUtensorMap mb;
    if (!make_tmap_bf16(&mb, x, (uint64_t)p.M, (uint64_t)p.K, BN, nullptr)) return cudaErrorInvalidValue;
    const int n_blocks = (p.M + BN - 1) / BN;
    const int tiles = (p.F / kTileF) * n_blocks * (ka.split ? ka.n_segs : 1);
    const int grid = tiles < device_sm_count() ? tiles : device_sm_count();
    // token blocks per group: about 32 MB of activations (a quarter of L2), at least one;
    // a projection with K >= 2F (the down projection) whose whole token range fits in
    // 64 MB takes it as one group, so its weights stream from HBM once (8B down at 2048
    // tokens: nine 6.9 MB blocks, three groups and 338 MB of DRAM reads otherwise)
    GemmKArgs k = ka;
    const long block_bytes = (long)BN * p.K * 2;
    k.group = (int)std::max(1L, std::min((long)n_blocks, (32L << 20) / block_bytes));
    if (p.K >= 2 * p.F && n_blocks * block_bytes <= (64L << 20)) k.group = n_blocks;
    return launch_pdl(kern, dim3(grid), dim3(C::THREADS), C::SMEM_BYTES, s, a0, a1, a2, mb, k);
}

template <int BN>
static cudaError_t dispatch_tt(const GemmProblem& p, const GemmKArgs& ka, const CUtensorMap& a0,
                               const CUtensorMap& a1, const CUtensorMap& a2, const bf16* x, cudaStream_t s) {
    switch (ka.e.kind) {
        case EPI_QKV: return run_tt<BN, false, EPI_QKV>(p, ka, a0, a1, a2, x, s);
        case EPI_RESID: return run_tt<BN, false, EPI_RESID>(p, ka, a0, a1, a2, x, s);
        case EPI_PLAIN: return run_tt<BN, false, EPI_PLAIN>(p, ka, a0, a1, a2, x, s);
        case EPI_LOGITS: return run_tt<BN, false, EPI_LOGITS>(p, ka, a0, a1, a2, x, s);
        default: return cudaErrorInvalidValue;
    }
}

// Token-block width of a single-accumulator projection: 256 (the higher
// arithmetic intensity per loaded byte) unless 192- or 128-token tiles give a
// clearly shorter schedule -- waves of tiles over the SMs times the tile's MMA
// length, at least 20% shorter -- as when 256-token tiles would leave SMs idle
// (few tokens: QKV at 512 tokens has 96 tiles of 256 for 152 SMs, 144 of 192);
// a few percent of span does not pay for the lower intensity (QKV at 8192
// tokens measured 1001 TFLOP/s at 128 against 1226 at 256).  240-token tiles
// load nearly as much per MMA as 256 and are taken whenever their schedule is
// shorter at all: at 2048 tokens the 32 feature tiles of O and down make 288
// tiles of 240 (two waves of 152 SMs, span 480) against 256 of 256 (span 512),
// and QKV's 48 make three waves either way (720 against 768).  The per-element
// result does not depend on the width.
static int tt_width(const GemmProblem& p) {
    const long n_sm = device_sm_count();
    const long ft = p.F / kTileF;
    auto span = [&](long bn) {
        const long tiles = ft * ((p.M + bn - 1) / bn);
        return ((tiles + n_sm - 1) / n_sm) * bn;
    };
    const long s256 = span(256), s240 = span(240), s192 = span(192), s128 = span(128);
    if (5 * s128 <= 4 * s256 && s128 <= s192 && s128 < s240) return 128;
    if (5 * s192 <= 4 * s256 && s192 < s240) return 192;
    if (s240 < s256) return 240;
    return 256;
}

cudaError_t launch_token_tiled(const GemmProblem& p, const GemmKArgs& ka, const CUtensorMap& a0,
                               const CUtensorMap& a1, const CUtensorMap& a2, const bf16* x, cudaStream_t s) {
    if (p.dual) {
        if (ka.e.kind != EPI_SWIGLU) return cudaErrorInvalidValue;
        return run_tt<128, true, EPI_SWIGLU>(p, ka, a0, a1, a2, x, s);
    }
    if (ka.split) return dispatch_tt<256>(p, ka, a0, a1, a2, x, s);
    switch (tt_width(p)) {
        case 128: return dispatch_tt<128>(p, ka, a0, a1, a2, x, s);
        case 192: return dispatch_tt<192>(p, ka, a0, a1, a2, x, s);
        case 240: return dispatch_tt<240>(p, ka, a0, a1, a2, x, s);
        default: return dispatch_tt<256>(p, ka, a0, a1, a2, x, s);
    }
}

}  // namespace llama
