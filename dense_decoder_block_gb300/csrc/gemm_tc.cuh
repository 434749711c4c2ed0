// tcgen05 projection kernel: Y[M, F] = X[M, K] . W[F, K]^T, bf16 in, fp32 accumulate in TMEM.
//
// Operand roles.  The weight is the MMA's A operand (M side, 128 output
// features per tile, one head when head_dim = 128) and the tokens are the B
// operand (N side).  Both are K-major, loaded by TMA with 128-byte swizzle.
// The accumulator tile is [128 features (TMEM lanes)] x [N tokens (columns)].
//
// Reduction schedule (the same in every mode, which is what makes decode
// results bit-identical to prefill rows): K is cut into segments of seg_kb
// 64-element k-blocks (fixed per projection when the handle is created); each segment is one tcgen05.mma chain (64-element k-blocks, four
// K=16 instructions each, ascending) started from zero; the segment results
// are added in fp32 in ascending segment order.
//
// Two schedules share that arithmetic:
//   token-tiled  (prefill, this file): grid = (feature tiles, token tiles); one
//                CTA runs every segment of its tile into alternating TMEM buffers
//                and the epilogue warps keep the running sum in registers.
//   weight-stream (decode, M <= 32, gemm_ws.cuh): persistent CTAs stream
//                (tile, segment) units, store fp32 segment results, and the last
//                CTA of a feature tile (atomic ticket) adds them in order.
//
// Warp roles (320 threads): warp 0 = TMA producer, warp 1 = TMEM owner + MMA
// issuer, warps 2..9 = epilogue.  Epilogue warp w reads TMEM lane quarter
// (w % 4) and half (w - 2) / 4 of the accumulator columns.
#pragma once
#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace llama {

constexpr int kGemmThreads = 320;
constexpr int kTileF = 128;           // features per tile (MMA M)
constexpr int kBlockK = 64;           // elements per k-block (128 bytes)
constexpr int kABytes = kTileF * kBlockK * 2;

template <int BN, bool DUAL>
struct GemmCfg {
    static constexpr int NACC = DUAL ? 2 : 1;
    static constexpr int B_BYTES = BN * kBlockK * 2;
    static constexpr int STAGE_BYTES = NACC * kABytes + B_BYTES;
    static constexpr int STAGES_RAW = (200 * 1024) / STAGE_BYTES;
    static constexpr int STAGES = STAGES_RAW > 8 ? 8 : STAGES_RAW;
    static constexpr int ACC_COLS = NACC * BN;
    static constexpr int TMEM_NEED = 2 * ACC_COLS;
    static constexpr int TMEM_COLS = TMEM_NEED <= 32 ? 32 : TMEM_NEED <= 64 ? 64 : TMEM_NEED <= 128 ? 128
                                     : TMEM_NEED <= 256 ? 256 : 512;
    static constexpr int CPT = BN / 2;   // accumulator columns per epilogue thread (per accumulator)
    static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 /*align*/ + 256 /*barriers*/;
    static_assert(TMEM_NEED <= 512, "TMEM budget");
    static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "UMMA N for M=128");
};

struct GemmKArgs {
    int M, F, K;
    int n_segs, seg_kb;
    int q_tiles, k_tiles;     // QKV: feature tiles per map (wq, wk); the rest are wv
    GemmEpi e;
    float* partial;   // weight-streaming: fp32 segment results [seg][acc][M][F]
};

__device__ __forceinline__ void named_bar_sync(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// ------------------------------------------------------------------ epilogue store of one column
template <int EPI>
__device__ __forceinline__ void epi_store(const GemmKArgs& a, int tile, int row, int n, float acc, float acc_up,
                                          bool valid) {
    const GemmEpi& e = a.e;
    const int f = tile * kTileF + row;
    if constexpr (EPI == EPI_QKV) {
        // tile kind: q heads, then k heads, then v heads (one head per tile)
        int kind, head;
        if (tile < a.q_tiles) { kind = 0; head = tile; }
        else if (tile < a.q_tiles + a.k_tiles) { kind = 1; head = tile - a.q_tiles; }
        else { kind = 2; head = tile - a.q_tiles - a.k_tiles; }
        const int T = e.tokens_per_seq;
        const int b = n / T, t = n - b * T;
        const int base = e.pos_dev ? *e.pos_dev : e.start_pos;
        const int pos = base + t;
        const bool pos_ok = (pos >= 0) && (pos < e.max_pos);
        float v = bf16_round(acc);
        if (kind < 2) {
            const float other = __shfl_xor_sync(0xffffffffu, v, 1);
            const int i = row >> 1;
            const int pc = pos_ok ? pos : 0;
            const float c = __ldg(e.cos_tab + (size_t)pc * kRopeMaxPairs + i);
            const float s = __ldg(e.sin_tab + (size_t)pc * kRopeMaxPairs + i);
            v = rope_rotate_elem(v, other, c, s, (row & 1) != 0);
        }
        if (!valid) return;
        if (!pos_ok) { record_error(e.err, LLAMA_ERR_POS_RANGE); return; }
        const bf16 r = __float2bfloat16_rn(v);
        if (kind == 0) {
            e.out[(size_t)n * (e.n_heads * 128) + head * 128 + row] = r;
        } else {
            bf16* dst = (kind == 1) ? e.kc : e.vc;
            dst[(((size_t)b * e.n_kv_heads + head) * e.kv_seq + pos) * 128 + row] = r;
        }
    } else {
        if (!valid) return;
        const size_t idx = (size_t)n * a.F + f;
        if constexpr (EPI == EPI_RESID) {
            e.out[idx] = __float2bfloat16_rn(epi_resid(__bfloat162float(e.resid[idx]), acc));
        } else if constexpr (EPI == EPI_SWIGLU) {
            e.out[idx] = __float2bfloat16_rn(epi_swiglu(acc, acc_up));
        } else if constexpr (EPI == EPI_PLAIN) {
            e.out[idx] = __float2bfloat16_rn(acc);
        } else {  // EPI_LOGITS
            e.out_f32[idx] = acc;
        }
    }
}

// ------------------------------------------------------------------ the kernel
template <int BN, bool DUAL, int EPI>
__global__ void __launch_bounds__(kGemmThreads, 1)
    k_gemm_tc(const __grid_constant__ CUtensorMap mA0, const __grid_constant__ CUtensorMap mA1,
              const __grid_constant__ CUtensorMap mA2, const __grid_constant__ CUtensorMap mB,
              const GemmKArgs a) {
    using C = GemmCfg<BN, DUAL>;
    constexpr int NACC = C::NACC;
    constexpr int CPT = C::CPT;
    constexpr uint32_t IDESC = ptx::idesc_bf16_f32(128, BN);

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t* full = (uint64_t*)(smem + C::STAGES * C::STAGE_BYTES);
    uint64_t* empty = full + C::STAGES;
    uint64_t* tfull = empty + C::STAGES;
    uint64_t* tempty = tfull + 2;
    uint32_t* tmem_holder = (uint32_t*)(tempty + 2);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tile = blockIdx.x;
    const int n0 = blockIdx.y * BN;
    const int seg_begin = 0;
    const int seg_end = a.n_segs;
    const int total_kb = a.K / kBlockK;
    int* err = a.e.err;

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::STAGES; ++i) { ptx::mbar_init(&full[i], 1); ptx::mbar_init(&empty[i], 1); }
        for (int i = 0; i < 2; ++i) { ptx::mbar_init(&tfull[i], 1); ptx::mbar_init(&tempty[i], 8); }
        ptx::fence_mbar_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc(tmem_holder, C::TMEM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;

    // A operand source for this feature tile
    const CUtensorMap* mapA = &mA0;
    int arow = tile * kTileF;
    if constexpr (EPI == EPI_QKV) {
        if (tile >= a.q_tiles + a.k_tiles) { mapA = &mA2; arow = (tile - a.q_tiles - a.k_tiles) * kTileF; }
        else if (tile >= a.q_tiles) { mapA = &mA1; arow = (tile - a.q_tiles) * kTileF; }
    }


    if (warp == 0) {
        // ---------------------------------------------------------- TMA producer
        if (lane == 0) {
            ptx::prefetch_tmap(mapA);
            if (DUAL) ptx::prefetch_tmap(&mA1);
            ptx::prefetch_tmap(&mB);
            const uint64_t pol_w = ptx::policy_evict_first();
            // k-blocks this CTA walks, segment after segment (only the last segment may be short)
            const int kb_first = seg_begin * a.seg_kb;
            const int n_iter = min(seg_end * a.seg_kb, total_kb) - kb_first;
            auto load_a = [&](int st, int kb) {
                uint8_t* dst = smem + st * C::STAGE_BYTES;
                ptx::tma_load_2d_hint(dst, mapA, &full[st], kb * kBlockK, arow, pol_w);
                if (DUAL) ptx::tma_load_2d_hint(dst + kABytes, &mA1, &full[st], kb * kBlockK, arow, pol_w);
            };
            auto load_b = [&](int st, int kb) {
                ptx::tma_load_2d(smem + st * C::STAGE_BYTES + NACC * kABytes, &mB, &full[st], kb * kBlockK, n0);
            };
            // The weights do not depend on the previous kernel: stream the first stages
            // of them before waiting for it, then fetch the activations.
            const int n_pre = min(C::STAGES, n_iter);
            for (int it = 0; it < n_pre; ++it) {
                ptx::mbar_arrive_expect_tx(&full[it], C::STAGE_BYTES);
                load_a(it, kb_first + it);
            }
            ptx::griddep_wait();
            ptx::griddep_launch_dependents();
            for (int it = 0; it < n_pre; ++it) load_b(it, kb_first + it);
            int stage = n_pre % C::STAGES;
            uint32_t phase = (n_pre == C::STAGES) ? 1u : 0u;
            bool ok = true;
            for (int it = n_pre; it < n_iter; ++it) {
                if (!ptx::mbar_wait(&empty[stage], phase ^ 1, err)) { ok = false; break; }
                ptx::mbar_arrive_expect_tx(&full[stage], C::STAGE_BYTES);
                load_a(stage, kb_first + it);
                load_b(stage, kb_first + it);
                if (++stage == C::STAGES) { stage = 0; phase ^= 1; }
            }
            if (!ok) {
                // drain: wait (bounded) for loads this thread issued that nobody consumed
                for (int i = 0; i < C::STAGES; ++i) ptx::mbar_wait_drain(&full[i], phase ^ (i < stage ? 0u : 1u));
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int use = 0;
            bool ok = true;
            for (int seg = seg_begin; seg < seg_end && ok; ++seg, ++use) {
                const int buf = use & 1;
                const uint32_t tph = (use >> 1) & 1;
                if (!ptx::mbar_wait(&tempty[buf], tph ^ 1, err)) { ok = false; break; }
                ptx::tc_fence_after();
                const uint32_t d = tmem_base + buf * C::ACC_COLS;
                const int kb0 = seg * a.seg_kb;
                const int kb1 = min(kb0 + a.seg_kb, total_kb);
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!ptx::mbar_wait(&full[stage], phase, err)) { ok = false; break; }
                    ptx::tc_fence_after();
                    const uint32_t sa = ptx::smem_u32(smem + stage * C::STAGE_BYTES);
                    const uint32_t sb = sa + NACC * kABytes;
#pragma unroll
                    for (int k = 0; k < kBlockK / 16; ++k) {
                        const uint32_t accum = (kb > kb0 || k > 0) ? 1u : 0u;
                        const uint64_t bdesc = ptx::sw128_kmajor_desc(sb + 32 * k);
                        ptx::umma_bf16(d, ptx::sw128_kmajor_desc(sa + 32 * k), bdesc, IDESC, accum);
                        if (DUAL) ptx::umma_bf16(d + BN, ptx::sw128_kmajor_desc(sa + kABytes + 32 * k), bdesc, IDESC, accum);
                    }
                    ptx::umma_commit(&empty[stage]);
                    if (++stage == C::STAGES) { stage = 0; phase ^= 1; }
                }
                if (ok) ptx::umma_commit(&tfull[buf]);
            }
        }
    } else {
        // ---------------------------------------------------------- epilogue (8 warps)
        ptx::griddep_wait();   // residuals, partials and tickets come from earlier kernels
        const int ew = warp - 2;
        const int quarter = warp & 3;
        const int half = ew >> 2;
        const int row = quarter * 32 + lane;
        const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
        float acc[NACC][CPT];
        int use = 0;
        bool ok = true;
        for (int seg = seg_begin; seg < seg_end; ++seg, ++use) {
            const int buf = use & 1;
            const uint32_t tph = (use >> 1) & 1;
            if (!ptx::mbar_wait(&tfull[buf], tph, err)) { ok = false; break; }
            ptx::tc_fence_after();
#pragma unroll
            for (int ac = 0; ac < NACC; ++ac) {
                constexpr int CH = CPT >= 16 ? 16 : CPT;
#pragma unroll
                for (int c = 0; c < CPT / CH; ++c) {
                    float tmp[CH];
                    ptx::tmem_ld<CH>(tmem_base + lane_addr + buf * C::ACC_COLS + ac * BN + half * CPT + c * CH, tmp);
                    ptx::tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < CH; ++j)
                        acc[ac][c * CH + j] = (seg == seg_begin) ? tmp[j] : __fadd_rn(acc[ac][c * CH + j], tmp[j]);
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&tempty[buf]);
        }

        const int ncol0 = n0 + half * CPT;
        if (ok) {
#pragma unroll
            for (int j = 0; j < CPT; ++j) {
                const int n = ncol0 + j;
                epi_store<EPI>(a, tile, row, n, acc[0][j], acc[NACC - 1][j], n < a.M);
            }
        }
    }

    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

}  // namespace llama
