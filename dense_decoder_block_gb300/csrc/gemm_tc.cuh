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
//   token-tiled  (prefill, gemm_tt.cuh): persistent CTAs walk (feature tile,
//                token block) tiles; each runs every segment of its tile into
//                alternating TMEM buffers and the epilogue warps keep the
//                running sum in registers.
//   weight-stream (decode, M <= 32, gemm_ws.cuh): persistent CTAs stream
//                (tile, segment) units and store fp32 segment results; the
//                reduction kernels add them in order and apply the epilogue.
//
// This header holds what both share: tile constants, kernel arguments and the
// per-column epilogue store.
#pragma once
#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace llama {

constexpr int kGemmThreads = 320;     // weight-streaming kernel: producer, MMA, 8 epilogue warps
constexpr int kTileF = 128;           // features per tile (MMA M)
constexpr int kBlockK = 64;           // elements per k-block (128 bytes)
constexpr int kABytes = kTileF * kBlockK * 2;

struct GemmKArgs {
    int M, F, K;
    int n_segs, seg_kb;
    int q_tiles, k_tiles;     // QKV: feature tiles per map (wq, wk); the rest are wv
    int group;                // token-tiled: token blocks taken per feature tile in a row
    int split;                // token-tiled: one (tile, K-segment) unit per CTA pass, fp32 results out
    GemmEpi e;
    float* partial;   // weight-streaming and split token-tiled: fp32 segment results [seg][acc][M][F]
};

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

// SwiGLU of CPT consecutive features of one token, u = bf16(bf16(silu(bf16(g))) *
// bf16(up)) (epi_swiglu), stored as 16-byte runs.
template <int CPT>
__device__ __forceinline__ void epi_swiglu_row(bf16* dst, const float (&g)[CPT], const float (&u)[CPT]) {
    static_assert(CPT % 8 == 0, "16-byte runs");
#pragma unroll
    for (int j0 = 0; j0 < CPT; j0 += 8) {
        uint32_t w[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const __nv_bfloat162 v = __floats2bfloat162_rn(epi_swiglu(g[j0 + 2 * t], u[j0 + 2 * t]),
                                                           epi_swiglu(g[j0 + 2 * t + 1], u[j0 + 2 * t + 1]));
            w[t] = *reinterpret_cast<const uint32_t*>(&v);
        }
        *reinterpret_cast<uint4*>(dst + j0) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// The fused epilogue of CPT consecutive columns (tokens n0 .. n0 + CPT - 1) of one
// accumulator row (feature row `row` of tile `tile`); columns >= M are skipped.
// What the epilogue reads -- the position, the RoPE factors, the residual -- is
// loaded for a chunk of columns before that chunk's stores: the outputs may
// alias the inputs as far as the compiler knows, so a load per column after the
// previous column's store costs one memory round trip per column.  Per element
// the arithmetic is epi_store's.
template <int EPI, int CPT>
__device__ __forceinline__ void epi_store_cols(const GemmKArgs& a, int tile, int row, int n0, const float (&acc)[CPT],
                                               const float (&acc_up)[CPT], int n_cols = CPT) {
    const GemmEpi& e = a.e;
    const int f = tile * kTileF + row;
    // columns j < n_valid are tokens of the call (and of this thread's n_cols)
    const int n_valid = min(a.M - n0, n_cols);
    if constexpr (EPI == EPI_QKV) {
        constexpr int CH = CPT < 4 ? CPT : 4;
        int kind, head;
        if (tile < a.q_tiles) { kind = 0; head = tile; }
        else if (tile < a.q_tiles + a.k_tiles) { kind = 1; head = tile - a.q_tiles; }
        else { kind = 2; head = tile - a.q_tiles - a.k_tiles; }
        const int T = e.tokens_per_seq;
        const int base = e.pos_dev ? *e.pos_dev : e.start_pos;
        // sequence bb at index tt; with per-sequence positions (T = 1) sequence bb
        // is token bb, read only for tokens of the call
        const int* ps = e.pos_seq;
        auto pos_at = [&](int bb, int tt) { return ps ? (bb < a.M ? ps[bb] : 0) : base + tt; };
        const int i = row >> 1;
        const bool rope = kind < 2 && !e.rope_later;   // warp-uniform
        // token n0 + j = (sequence b, index t), advanced column by column
        int b = n0 / T, t = n0 - b * T;
        const size_t q_stride = (size_t)e.n_heads * 128;
        bf16* qp = e.out + (size_t)n0 * q_stride + head * 128 + row;   // kind 0
        bf16* cp = ((kind == 1) ? e.kc : e.vc) + (size_t)head * e.kv_seq * 128 + row;   // kinds 1, 2
        const size_t seq_stride = (size_t)e.n_kv_heads * e.kv_seq * 128;
        if (!rope && !ps && base >= 0 && base + T <= e.max_pos) {
            // Every position of the call is valid and nothing is rotated here: short
            // straight-line stores (bf16(bf16_round(x)) == bf16(x)).  The general
            // loop below would keep a large unrolled body in the instruction cache.
            if (kind == 0) {
#pragma unroll
                for (int j = 0; j < CPT; ++j)
                    if (j < n_valid) qp[(size_t)j * q_stride] = __float2bfloat16_rn(acc[j]);
            } else {
                bf16* dst = cp + (size_t)b * seq_stride + (size_t)(base + t) * 128;
#pragma unroll
                for (int j = 0; j < CPT; ++j) {
                    if (j < n_valid) *dst = __float2bfloat16_rn(acc[j]);
                    dst += 128;
                    if (++t == T) { t = 0; ++b; dst = cp + (size_t)b * seq_stride + (size_t)base * 128; }
                }
            }
            return;
        }
#pragma unroll
        for (int c0 = 0; c0 < CPT; c0 += CH) {
            float cs[CH], sn[CH];
            if (rope) {
                int bb = b, tt = t;
#pragma unroll
                for (int j = 0; j < CH; ++j) {
                    const int pos = pos_at(bb, tt);
                    const int pc = (pos >= 0 && pos < e.max_pos) ? pos : 0;
                    cs[j] = __ldg(e.cos_tab + (size_t)pc * kRopeMaxPairs + i);
                    sn[j] = __ldg(e.sin_tab + (size_t)pc * kRopeMaxPairs + i);
                    if (++tt == T) { tt = 0; ++bb; }
                }
            }
#pragma unroll
            for (int j = 0; j < CH; ++j) {
                const int pos = pos_at(b, t);
                const bool pos_ok = (pos >= 0) && (pos < e.max_pos);
                float v = bf16_round(acc[c0 + j]);
                if (rope) {
                    const float other = __shfl_xor_sync(0xffffffffu, v, 1);
                    v = rope_rotate_elem(v, other, cs[j], sn[j], (row & 1) != 0);
                }
                if (c0 + j < n_valid) {
                    if (!pos_ok) {
                        record_error(e.err, LLAMA_ERR_POS_RANGE);
                    } else {
                        const bf16 r = __float2bfloat16_rn(v);
                        if (kind == 0) qp[(size_t)(c0 + j) * q_stride] = r;
                        else cp[(size_t)b * seq_stride + (size_t)pos * 128] = r;
                    }
                }
                if (++t == T) { t = 0; ++b; }
            }
        }
    } else if constexpr (EPI == EPI_RESID) {
        constexpr int CH = CPT < 8 ? CPT : 8;
        const size_t F = a.F;
        const bf16* rp = e.resid + (size_t)n0 * F + f;
        bf16* op = e.out + (size_t)n0 * F + f;
#pragma unroll
        for (int c0 = 0; c0 < CPT; c0 += CH) {
            float x[CH];
#pragma unroll
            for (int j = 0; j < CH; ++j) x[j] = c0 + j < n_valid ? __bfloat162float(rp[(c0 + j) * F]) : 0.f;
#pragma unroll
            for (int j = 0; j < CH; ++j)
                if (c0 + j < n_valid) op[(c0 + j) * F] = __float2bfloat16_rn(epi_resid(x[j], acc[c0 + j]));
        }
    } else {
#pragma unroll
        for (int j = 0; j < CPT; ++j) epi_store<EPI>(a, tile, row, n0 + j, acc[j], acc_up[j], j < n_valid);
    }
}

}  // namespace llama
