// Persistent weight-streaming projection (decode, M <= 32 tokens).
//
// Same arithmetic as the token-tiled kernel in gemm_tc.cuh (one tcgen05.mma chain
// per K-segment, segments added in ascending fp32 order), scheduled for HBM
// streaming: the work is cut into units (feature tile, K-segment) of
// 128 x seg_kb*64 weights; one CTA per SM walks units blockIdx.x,
// blockIdx.x + gridDim.x, ... with a single TMA ring that never drains between
// units.  The MMA warp accumulates each unit into one of two TMEM buffers; the
// epilogue warps drain a buffer while the next unit streams, store the unit's
// fp32 segment result to the workspace; a small reduction kernel (reduce.cu),
// launched right behind it, adds each output's segments in ascending order and
// runs the fused epilogue.  With a single segment the epilogue runs here.
#pragma once
#include "gemm_tc.cuh"

namespace llama {

template <int BN, bool DUAL>
struct WsCfg {
    static constexpr int NACC = DUAL ? 2 : 1;
    static constexpr int B_BYTES = BN * kBlockK * 2;
    static constexpr int STAGE_BYTES = NACC * kABytes + B_BYTES;
    static constexpr int STAGES_RAW = (208 * 1024) / STAGE_BYTES;
    static constexpr int STAGES = STAGES_RAW > 12 ? 12 : STAGES_RAW;
    static constexpr int ACC_COLS = NACC * BN;
    static constexpr int TMEM_NEED = 2 * ACC_COLS;
    static constexpr int TMEM_COLS = TMEM_NEED <= 32 ? 32 : TMEM_NEED <= 64 ? 64 : TMEM_NEED <= 128 ? 128 : 256;
    static constexpr int CPT = BN / 2;
    static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 512;
    static_assert(BN == 16 || BN == 32, "weight-streaming tile widths");
};

template <int BN, bool DUAL, int EPI>
__global__ void __launch_bounds__(kGemmThreads, 1)
    k_gemm_ws(const __grid_constant__ CUtensorMap mA0, const __grid_constant__ CUtensorMap mA1,
              const __grid_constant__ CUtensorMap mA2, const __grid_constant__ CUtensorMap mB, const GemmKArgs a) {
    using C = WsCfg<BN, DUAL>;
    constexpr int NACC = C::NACC;
    constexpr int CPT = C::CPT;
    constexpr uint32_t IDESC = ptx::idesc_bf16_f32(128, BN);

    TRACE(const unsigned long long tr0 = trace_stamp();)
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t* full = (uint64_t*)(smem + C::STAGES * C::STAGE_BYTES);
    uint64_t* empty = full + C::STAGES;
    uint64_t* tfull = empty + C::STAGES;
    uint64_t* tempty = tfull + 2;
    uint32_t* tmem_holder = (uint32_t*)(tempty + 2);
    // trace builds: when the MMA thread's wait returned
    TRACE(unsigned long long* tr_release = (unsigned long long*)(tempty + 3);)

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int total_kb = a.K / kBlockK;
    const int n_tiles = a.F / kTileF;
    const int n_units = n_tiles * a.n_segs;
    int* err = a.e.err;

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::STAGES; ++i) { ptx::mbar_init(&full[i], 1); ptx::mbar_init(&empty[i], 1); }
        for (int i = 0; i < 2; ++i) { ptx::mbar_init(&tfull[i], 1); ptx::mbar_init(&tempty[i], 8); }
        ptx::fence_mbar_init();
        TRACE(*tr_release = 0;)
    }
    if (warp == 1) {
        ptx::tmem_alloc(tmem_holder, C::TMEM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;

    // unit u -> (tile, segment), segments of one tile on neighbouring CTAs
    auto unit_tile = [&](int u) { return u / a.n_segs; };
    auto unit_kb0 = [&](int u) { return (u % a.n_segs) * a.seg_kb; };
    auto unit_kb1 = [&](int u) { return min(unit_kb0(u) + a.seg_kb, total_kb); };

    if (warp == 0) {
        // ---------------------------------------------------------- TMA producer
        if (lane == 0) {
            ptx::prefetch_tmap(&mA0);
            if (EPI == EPI_QKV || DUAL) ptx::prefetch_tmap(&mA1);
            if (EPI == EPI_QKV) ptx::prefetch_tmap(&mA2);
            ptx::prefetch_tmap(&mB);
            const uint64_t pol_w = ptx::policy_evict_first();
            int n_iter = 0;
            for (int u = blockIdx.x; u < n_units; u += gridDim.x) n_iter += unit_kb1(u) - unit_kb0(u);
            const int n_pre = min(C::STAGES, n_iter);
            int stage = 0, it = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
                const int tile = unit_tile(u);
                const CUtensorMap* mapA = &mA0;
                int arow = tile * kTileF;
                if constexpr (EPI == EPI_QKV) {
                    if (tile >= a.q_tiles + a.k_tiles) { mapA = &mA2; arow = (tile - a.q_tiles - a.k_tiles) * kTileF; }
                    else if (tile >= a.q_tiles) { mapA = &mA1; arow = (tile - a.q_tiles) * kTileF; }
                }
                for (int kb = unit_kb0(u); kb < unit_kb1(u); ++kb, ++it) {
                    uint8_t* dst = smem + stage * C::STAGE_BYTES;
                    if (it >= n_pre) {
                        if (!ptx::mbar_wait(&empty[stage], phase ^ 1, err)) { ok = false; break; }
                    }
                    ptx::mbar_arrive_expect_tx(&full[stage], C::STAGE_BYTES);
                    ptx::tma_load_2d_hint(dst, mapA, &full[stage], kb * kBlockK, arow, pol_w);
                    if (DUAL) ptx::tma_load_2d_hint(dst + kABytes, &mA1, &full[stage], kb * kBlockK, arow, pol_w);
                    // The weights do not depend on earlier kernels: the first n_pre stages
                    // stream before the wait.  Their activations are loaded by the MMA thread
                    // as soon as the wait returns (issuing the weight copies takes this thread
                    // about 2 us); the stage completes only with this thread's arrival and
                    // both copies, in whatever order they land.
                    if (it >= n_pre) {
                        if (it == n_pre) ptx::griddep_wait();
                        ptx::tma_load_2d(dst + NACC * kABytes, &mB, &full[stage], kb * kBlockK, 0);
                    }
                    if (++stage == C::STAGES) { stage = 0; phase ^= 1; }
                }
            }
            if (!ok) {
                for (int i = 0; i < C::STAGES; ++i) ptx::mbar_wait_drain(&full[i], phase ^ (i < stage ? 0u : 1u));
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            // first the activations of the prefetched stages (see the producer)
            ptx::prefetch_tmap(&mB);
            ptx::griddep_wait();
            TRACE(if (LLAMA_TRACE_ON) *tr_release = trace_clock();)
            ptx::griddep_launch_dependents();
            {
                int n_iter = 0;
                for (int u = blockIdx.x; u < n_units; u += gridDim.x) n_iter += unit_kb1(u) - unit_kb0(u);
                const int n_pre = min(C::STAGES, n_iter);
                int j = 0;
                for (int u = blockIdx.x; u < n_units && j < n_pre; u += gridDim.x)
                    for (int kb = unit_kb0(u); kb < unit_kb1(u) && j < n_pre; ++kb, ++j)
                        ptx::tma_load_2d(smem + j * C::STAGE_BYTES + NACC * kABytes, &mB, &full[j], kb * kBlockK, 0);
            }
            int stage = 0, use = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++use) {
                const int buf = use & 1;
                if (!ptx::mbar_wait(&tempty[buf], ((use >> 1) & 1) ^ 1, err)) { ok = false; break; }
                ptx::tc_fence_after();
                const uint32_t d = tmem_base + buf * C::ACC_COLS;
                const int kb0 = unit_kb0(u);
                for (int kb = kb0; kb < unit_kb1(u); ++kb) {
                    if (!ptx::mbar_wait(&full[stage], phase, err)) { ok = false; break; }
                    ptx::tc_fence_after();
                    const uint32_t sa = ptx::smem_u32(smem + stage * C::STAGE_BYTES);
                    const uint32_t sb = sa + NACC * kABytes;
                    const uint64_t bdesc = ptx::sw128_kmajor_desc(sb);
                    ptx::umma_kblock(d, ptx::sw128_kmajor_desc(sa), bdesc, IDESC, kb > kb0);
                    if (DUAL) ptx::umma_kblock(d + BN, ptx::sw128_kmajor_desc(sa + kABytes), bdesc, IDESC, kb > kb0);
                    ptx::umma_commit(&empty[stage]);
                    if (++stage == C::STAGES) { stage = 0; phase ^= 1; }
                }
                if (ok) ptx::umma_commit(&tfull[buf]);
            }
        }
    } else {
        // ---------------------------------------------------------- epilogue (8 warps)
        ptx::griddep_wait();   // residuals come from earlier kernels
        const int ew = warp - 2;
        const int quarter = warp & 3;
        const int half = ew >> 2;
        const int row = quarter * 32 + lane;
        const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
        const int ncol0 = half * CPT;
        int use = 0;
        for (int u = blockIdx.x; u < n_units; u += gridDim.x, ++use) {
            const int buf = use & 1;
            const int tile = unit_tile(u);
            const int seg = u % a.n_segs;
            const int f = tile * kTileF + row;
            float acc[NACC][CPT];
            bool ok = ptx::mbar_wait(&tfull[buf], (use >> 1) & 1, err);
            if (ok) {
                ptx::tc_fence_after();
#pragma unroll
                for (int ac = 0; ac < NACC; ++ac) {
                    ptx::tmem_ld<CPT>(tmem_base + lane_addr + buf * C::ACC_COLS + ac * BN + half * CPT, acc[ac]);
                    ptx::tmem_wait_ld();
                }
                ptx::tc_fence_before();
            }
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&tempty[buf]);
            if (a.n_segs > 1) {
                // fp32 segment result, [seg][acc][token][feature]; the reduction kernel of
                // this projection adds the segments in ascending order and runs the epilogue
                if (ok) {
#pragma unroll
                    for (int ac = 0; ac < NACC; ++ac)
#pragma unroll
                        for (int j = 0; j < CPT; ++j) {
                            const int n = ncol0 + j;
                            if (n < a.M) a.partial[(((size_t)seg * NACC + ac) * a.M + n) * a.F + f] = acc[ac][j];
                        }
                }
                continue;
            }
            if (ok) epi_store_cols<EPI, CPT>(a, tile, row, ncol0, acc[0], acc[NACC - 1]);
        }
    }

    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
    TRACE(trace_cta(TR_GEMM_WS | (EPI << 8), tr0, *tr_release);)
}

}  // namespace llama
