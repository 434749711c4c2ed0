// Persistent token-tiled projection (prefill, M > 32 tokens).
//
// Same arithmetic as the weight-streaming kernel (gemm_ws.cuh): per output, one
// tcgen05.mma chain per K-segment of seg_kb k-blocks, segment results added in
// ascending fp32 order.  Here one CTA per SM walks output tiles of 128 features
// x BN tokens (BN = 256, 240, 192 or 128 as the host picks; 128 with the gate/up
// pair); for every tile it runs the
// segments' chains into two alternating TMEM buffers while sixteen epilogue
// warps (four per TMEM lane quarter, each owning a quarter of the columns) keep
// the running sums in registers; after a tile's last segment they apply the
// fused epilogue and store, while the MMAs of the next tile already run.
// Tiles are taken in groups of `group` token blocks per feature tile (chosen on
// the host so that a group's activations stay well inside L2), so a weight
// tile is streamed from HBM once per group and reused from L2 by the CTAs
// working on it.
//
// Warp roles (640 threads): warp 0 = TMA producer, warp 1 = TMEM owner + MMA
// issuer, warps 2-3 idle; warps 4..19 = epilogue, warp w reading TMEM lane
// quarter w % 4 and column quarter (w - 4) / 4.  Warpgroup 0 gives registers
// to the epilogue warpgroups, whose running sums take 64 per thread.
//
// Split mode (few tokens, a.split): the work units are (feature tile, K-segment,
// token block) instead of whole tiles, so that more SMs share a projection whose
// tiles would not fill them; each unit's segment result goes out in fp32, laid
// out [segment][token][feature] as the weight-streaming kernel lays it, and the
// same reduction kernels add the segments in ascending order and apply the
// epilogue.  Per output the operations are the same (one MMA chain per segment,
// ascending fp32 sum, the same epilogue functions).  Units of one feature tile
// and segment are consecutive, so the CTAs that share a weight tile read it in
// step.
#pragma once
#include "gemm_tc.cuh"

namespace llama {

template <int BN, bool DUAL>
struct TtCfg {
    static constexpr int NACC = DUAL ? 2 : 1;
    static constexpr int B_BYTES = BN * kBlockK * 2;
    static constexpr int STAGE_BYTES = NACC * kABytes + B_BYTES;
    static constexpr int STAGES_RAW = (200 * 1024) / STAGE_BYTES;
    static constexpr int STAGES = STAGES_RAW > 6 ? 6 : STAGES_RAW;
    // TMEM columns per accumulator and the epilogue's column split: a 240-token tile
    // keeps the 256-column layout (its MMA writes columns 0..239; the last column
    // group's threads store 48 of their 64)
    static constexpr int NCOLS = BN == 240 ? 256 : BN;
    static constexpr int ACC_COLS = NACC * NCOLS;              // one TMEM buffer
    static constexpr int TMEM_COLS = 512;                      // two buffers
    static constexpr int EPI_WARPS = 16;
    static constexpr int CPT = NCOLS / 4;                      // columns per thread per accumulator
    static constexpr int THREADS = 128 + 32 * EPI_WARPS;       // warpgroup 0 + four epilogue warpgroups
    static constexpr int REGS_CTRL = 56;                       // warpgroup 0 after the split
    static constexpr int REGS_EPI = 104;                       // epilogue warpgroups after the split
    static constexpr int REGS_NEEDED = 128 * REGS_CTRL + 32 * EPI_WARPS * REGS_EPI;
    static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 256;
    static_assert(2 * ACC_COLS <= 512, "two TMEM buffers");
    static_assert(BN % 16 == 0 && BN <= NCOLS && NCOLS % 64 == 0, "MMA N and the epilogue's 16-column loads");
};

template <int BN, bool DUAL, int EPI>
__global__ void __launch_bounds__(TtCfg<BN, DUAL>::THREADS, 1)
    k_gemm_tt(const __grid_constant__ CUtensorMap mA0, const __grid_constant__ CUtensorMap mA1,
              const __grid_constant__ CUtensorMap mA2, const __grid_constant__ CUtensorMap mB, const GemmKArgs a) {
    using C = TtCfg<BN, DUAL>;
    constexpr int NACC = C::NACC;
    constexpr int CPT = C::CPT;
    // The gate/up pair runs with the roles swapped: the 128 tokens are the A
    // operand and the gate and up tiles of the same 128 features, stored one after
    // the other, one B operand of 256 rows -- one N = 256 MMA per K step instead of
    // two N = 128 MMAs that each re-read the token tile from shared memory.
    // Accumulator lane = token, columns 0..127 gate, 128..255 up.
    constexpr uint32_t IDESC = DUAL ? ptx::idesc_bf16_f32(128, 2 * BN) : ptx::idesc_bf16_f32(128, BN);

    TRACE(const unsigned long long tr0 = trace_stamp();)
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t* full = (uint64_t*)(smem + C::STAGES * C::STAGE_BYTES);
    uint64_t* empty = full + C::STAGES;
    uint64_t* tfull = empty + C::STAGES;
    uint64_t* tempty = tfull + 2;
    uint32_t* tmem_holder = (uint32_t*)(tempty + 2);
    // trace builds: when the producer's wait returned
    TRACE(unsigned long long* tr_release = (unsigned long long*)(tempty + 3);)

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int total_kb = a.K / kBlockK;
    const int m_tiles = a.F / kTileF;
    const int n_blocks = (a.M + BN - 1) / BN;
    const int n_tiles = m_tiles * n_blocks;
    const bool split = a.split != 0;
    const int n_work = split ? n_tiles * a.n_segs : n_tiles;   // units per pass of the CTAs
    int* err = a.e.err;

    // tile t -> (feature tile m, token block n), groups of a.group token blocks
    const int G = a.group;
    auto tile_mn = [&](int t, int& m, int& n) {
        const int grp = t / (G * m_tiles);
        const int rem = t - grp * G * m_tiles;
        const int gn = min(G, n_blocks - grp * G);
        m = rem / gn;
        n = grp * G + (rem - m * gn);
    };
    // work item w -> (feature tile m, token block n, k-blocks [kb0, kb1), segment)
    auto work_of = [&](int w, int& m, int& n, int& kb0, int& kb1, int& seg) {
        if (split) {
            m = w / (a.n_segs * n_blocks);
            const int rem = w - m * a.n_segs * n_blocks;
            seg = rem / n_blocks;
            n = rem - seg * n_blocks;
            kb0 = seg * a.seg_kb;
            kb1 = min(kb0 + a.seg_kb, total_kb);
        } else {
            tile_mn(w, m, n);
            seg = 0;
            kb0 = 0;
            kb1 = total_kb;
        }
    };

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::STAGES; ++i) { ptx::mbar_init(&full[i], 1); ptx::mbar_init(&empty[i], 1); }
        for (int i = 0; i < 2; ++i) { ptx::mbar_init(&tfull[i], 1); ptx::mbar_init(&tempty[i], C::EPI_WARPS); }
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
    if (warp < 4) {
        ptx::setmaxnreg_dec<C::REGS_CTRL>();
        if (warp == 0) {
            // ---------------------------------------------------------- TMA producer
            if (lane == 0) {
                ptx::prefetch_tmap(&mA0);
                if (EPI == EPI_QKV || DUAL) ptx::prefetch_tmap(&mA1);
                if (EPI == EPI_QKV) ptx::prefetch_tmap(&mA2);
                ptx::prefetch_tmap(&mB);
                int stage = 0;
                uint32_t phase = 0;
                int it = 0;
                bool waited = false, ok = true;
                // (k-block, token block) of the first STAGES loads: their activations are
                // issued once the grid dependency resolves
                int pre_kb[C::STAGES] = {}, pre_n[C::STAGES] = {};
                auto load_b_of = [&](int j) {
                    ptx::tma_load_2d(smem + j * C::STAGE_BYTES + NACC * kABytes, &mB, &full[j], pre_kb[j] * kBlockK,
                                     pre_n[j] * BN);
                };
                for (int t = blockIdx.x; t < n_work && ok; t += gridDim.x) {
                    int m, n, kb0, kb1, seg;
                    work_of(t, m, n, kb0, kb1, seg);
                    const CUtensorMap* mapA = &mA0;
                    int arow = m * kTileF;
                    if constexpr (EPI == EPI_QKV) {
                        if (m >= a.q_tiles + a.k_tiles) { mapA = &mA2; arow = (m - a.q_tiles - a.k_tiles) * kTileF; }
                        else if (m >= a.q_tiles) { mapA = &mA1; arow = (m - a.q_tiles) * kTileF; }
                    }
                    for (int kb = kb0; kb < kb1; ++kb, ++it) {
                        uint8_t* dst = smem + stage * C::STAGE_BYTES;
                        if (it >= C::STAGES && !ptx::mbar_wait(&empty[stage], phase ^ 1, err)) { ok = false; break; }
                        ptx::mbar_arrive_expect_tx(&full[stage], C::STAGE_BYTES);
                        ptx::tma_load_2d(dst, mapA, &full[stage], kb * kBlockK, arow);
                        if (DUAL) ptx::tma_load_2d(dst + kABytes, &mA1, &full[stage], kb * kBlockK, arow);
                        if (waited) {
                            ptx::tma_load_2d(dst + NACC * kABytes, &mB, &full[stage], kb * kBlockK, n * BN);
                        } else {
                            pre_kb[it] = kb;
                            pre_n[it] = n;
                            if (it == C::STAGES - 1) {
                                // The weights do not depend on the previous kernel: the first stages
                                // of them are in flight before waiting for it; then the activations.
                                ptx::griddep_wait();
                                TRACE(if (LLAMA_TRACE_ON) *tr_release = trace_clock();)
                                ptx::griddep_launch_dependents();
                                for (int j = 0; j <= it; ++j) load_b_of(j);
                                waited = true;
                            }
                        }
                        if (++stage == C::STAGES) { stage = 0; phase ^= 1; }
                    }
                }
                if (!waited && ok) {   // fewer k-blocks than stages in total
                    ptx::griddep_wait();
                    TRACE(if (LLAMA_TRACE_ON) *tr_release = trace_clock();)
                    ptx::griddep_launch_dependents();
                    for (int j = 0; j < it; ++j) load_b_of(j);
                }
                if (!ok) {
                    for (int i = 0; i < C::STAGES; ++i) ptx::mbar_wait_drain(&full[i], phase ^ (i < stage ? 0u : 1u));
                }
            }
        } else if (warp == 1) {
            // ---------------------------------------------------------- MMA issuer
            if (lane == 0) {
                int stage = 0, use = 0;
                uint32_t phase = 0;
                bool ok = true;
                for (int t = blockIdx.x; t < n_work && ok; t += gridDim.x) {
                    int wm, wn, wkb0, wkb1, wseg;
                    work_of(t, wm, wn, wkb0, wkb1, wseg);
                    const int seg_first = split ? wseg : 0, seg_end = split ? wseg + 1 : a.n_segs;
                    for (int seg = seg_first; seg < seg_end && ok; ++seg, ++use) {
                        const int buf = use & 1;
                        if (!ptx::mbar_wait(&tempty[buf], ((use >> 1) & 1) ^ 1, err)) { ok = false; break; }
                        ptx::tc_fence_after();
                        const uint32_t d = tmem_base + buf * C::ACC_COLS;
                        const int kb0 = seg * a.seg_kb;
                        const int kb1 = min(kb0 + a.seg_kb, total_kb);
                        for (int kb = kb0; kb < kb1; ++kb) {
                            if (!ptx::mbar_wait(&full[stage], phase, err)) { ok = false; break; }
                            ptx::tc_fence_after();
                            const uint32_t sa = ptx::smem_u32(smem + stage * C::STAGE_BYTES);
                            const uint32_t sb = sa + NACC * kABytes;
                            if (DUAL)   // A = tokens, B = gate rows then up rows
                                ptx::umma_kblock(d, ptx::sw128_kmajor_desc(sb), ptx::sw128_kmajor_desc(sa), IDESC, kb > kb0);
                            else        // A = weights, B = tokens
                                ptx::umma_kblock(d, ptx::sw128_kmajor_desc(sa), ptx::sw128_kmajor_desc(sb), IDESC, kb > kb0);
                            ptx::umma_commit(&empty[stage]);
                            if (++stage == C::STAGES) { stage = 0; phase ^= 1; }
                        }
                        if (ok) ptx::umma_commit(&tfull[buf]);
                    }
                }
            }
        }
    } else {
        // ---------------------------------------------------------- epilogue (16 warps)
        ptx::setmaxnreg_inc<C::REGS_EPI>();
        ptx::griddep_wait();   // residuals come from earlier kernels
        const int ew = warp - 4;
        const int quarter = warp & 3;
        const int cg = ew >> 2;                   // column group 0..3
        const int row = quarter * 32 + lane;
        const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
        int use = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < n_work; t += gridDim.x) {
            int m, n, wkb0, wkb1, wseg;
            work_of(t, m, n, wkb0, wkb1, wseg);
            // -0 + s == s for every fp32 s, so the sum starts exactly at segment 0
            float acc[NACC][CPT];
#pragma unroll
            for (int ac = 0; ac < NACC; ++ac)
#pragma unroll
                for (int j = 0; j < CPT; ++j) acc[ac][j] = -0.0f;
            const int seg_first = split ? wseg : 0, seg_end = split ? wseg + 1 : a.n_segs;
            for (int seg = seg_first; seg < seg_end; ++seg, ++use) {
                const int buf = use & 1;
                if (ok) ok = ptx::mbar_wait(&tfull[buf], (use >> 1) & 1, err);
                ptx::tc_fence_after();
#pragma unroll
                for (int ac = 0; ac < NACC; ++ac) {
                    constexpr int CH = 16;
#pragma unroll
                    for (int c = 0; c < CPT / CH; ++c) {
                        float tmp[CH];
                        ptx::tmem_ld<CH>(tmem_base + lane_addr + buf * C::ACC_COLS + ac * C::NCOLS + cg * CPT + c * CH,
                                         tmp);
                        ptx::tmem_wait_ld();
#pragma unroll
                        for (int j = 0; j < CH; ++j) acc[ac][c * CH + j] = __fadd_rn(acc[ac][c * CH + j], tmp[j]);
                    }
                }
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&tempty[buf]);
            }
            if (ok && split) {
                // the unit's fp32 segment result, [seg][token][feature] (the reduction adds them)
                if constexpr (!DUAL) {
                    const int f = m * kTileF + row;
                    const int n0 = n * BN + cg * CPT;
                    float* dst = a.partial + ((size_t)wseg * a.M + n0) * a.F + f;
#pragma unroll
                    for (int j = 0; j < CPT; ++j)
                        if (n0 + j < a.M && cg * CPT + j < BN) dst[(size_t)j * a.F] = acc[0][j];
                }
            } else if (ok) {
                if constexpr (DUAL) {
                    // lane = token n * BN + row, columns = features m * 128 + cg * CPT + j
                    const int tok = n * BN + row;
                    if (tok < a.M) epi_swiglu_row<CPT>(a.e.out + (size_t)tok * a.F + m * kTileF + cg * CPT, acc[0], acc[1]);
                } else {
                    epi_store_cols<EPI, CPT>(a, m, row, n * BN + cg * CPT, acc[0], acc[NACC - 1], BN - cg * CPT);
                }
            }
        }
    }

    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
    TRACE(trace_cta(TR_GEMM_TT | (EPI << 8) | (a.split ? 1u << 12 : 0u), tr0, *tr_release);)
}

}  // namespace llama
