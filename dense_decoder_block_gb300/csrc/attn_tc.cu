// Causal GQA attention on the tensor cores (tcgen05), prefill and decode, with
// one reduction schedule shared by both.
//
// "Llama 3.1 70B", Grouped-Query Attention: scores q.k / sqrt(d_h), causal,
// softmax over keys, weights average V; query head h reads KV head
// h / (n_heads / n_kv_heads).  "Llama 3 8B · Prepare Q, K, V": K and V are
// cached at KV-head size; one pass over a KV head serves its whole group.
//
// Unit of work: a 128-row query tile of one KV group against one 128-key chunk.
// Prefill tiles hold 128 / n_rep consecutive tokens x the n_rep heads of the
// group (row = token * n_rep + head); decode tiles hold the group's n_rep heads
// of one token (the other rows are zero).
//   S   = Q K^T        tcgen05.mma M=128 N=128 K=128, both operands K-major
//   softmax, one thread per row (sequential over the chunk's keys):
//         t_j = S_j * log2(e)/sqrt(d_h); m = max_{j<=jmax} t_j;
//         p_j = bf16(2^(t_j - m)) (0 past jmax); l = sum_j p_j in key order
//   O_c = P V          tcgen05.mma M=128 N=128 K=128, V MN-major (as cached)
// Chunks are folded in ascending order from chunk 0 with one fold formula:
// prefill folds in TMEM as it walks the chunks, decode stores each chunk's
// (O_c, m, l) and the combine kernel (attn_simt.cu) folds them in the same order,
// so a decode row equals the prefill row at the same position bit for bit.
//
// Warps: 0 = TMA producer, 1 = TMEM owner + MMA issuer, 2..5 = softmax / fold
// (thread = row; warp w reads TMEM lane quarter w % 4).
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>

#include "internal.h"
#include "ptx.cuh"

namespace llama {

namespace {

constexpr int kThreads = 192;
constexpr int kSub = 128 * 128;                 // one [128 rows][64 bf16] swizzled sub-tile, bytes
constexpr int OFF_Q = 0;                        // Q: 2 sub-tiles (d 0-63, 64-127)
constexpr int OFF_KV = 2 * kSub;                // 2 stages x (K: 2 sub-tiles, V: 2 sub-tiles)
constexpr int KV_STAGE = 4 * kSub;
constexpr int OFF_P = OFF_KV + 2 * KV_STAGE;    // P: 2 sub-tiles (keys 0-63, 64-127)
constexpr int OFF_BAR = OFF_P + 2 * kSub;
constexpr int SMEM_BYTES = OFF_BAR + 256 + 1024;
constexpr int TM_S = 0, TM_OC = 128, TM_O = 256;   // TMEM columns
constexpr uint32_t IDESC_S = ptx::idesc_bf16_f32(128, 128);
constexpr uint32_t IDESC_PV = ptx::idesc_bf16_f32_bmn(128, 128);

struct TcArgs {
    int batch, tokens, n_heads, n_kv_heads, kv_seq, start_pos, max_pos;
    const int* pos_dev;
    float scale_log2;
    const bf16* q;       // decode: [B, Hq * 128]
    bf16* o;             // prefill: [B * T, Hq * 128]
    float* partial;      // decode: [B, Hkv, n_chunks, n_rep, kPartStride]
    int n_chunks;        // decode: chunk slots per (sequence, KV head)
    int chunks_per_cta;  // decode
    int tq;              // prefill: tokens per query tile
    int* err;
};

// Byte offset of the 16-byte chunk `c16` (0..7) of row `r` in a 128-byte-swizzled sub-tile.
__device__ __forceinline__ uint32_t sw_off(int r, int c16) { return (uint32_t)(r * 128 + ((c16 ^ (r & 7)) << 4)); }

// 2^x on the special-function unit (PTX ex2.approx: max relative error 2^-22,
// far below the bf16 rounding of p that follows).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// The softmax of one query row over one 128-key chunk.  Both kernels compute
// exactly this (prefill with one thread per row, decode with four lanes per row):
//   t_j = S_j * scale_log2                      (keys 0..jmax visible; jmax < 0: none)
//   m   = max_{j <= jmax} t_j                   (exact, any order)
//   p_j = bf16(2^(t_j - m)), 0 for hidden keys
//   l   = ((L0 + L1) + L2) + L3,  Lq = sum of p_j over keys 32q..32q+31 in key order
// The P row goes to the two 64-key sub-tiles of the swizzled K-major P operand
// (p_sub_stride bytes apart) at row `prow` when write_p.
__device__ __forceinline__ void softmax_quarter(const float* sv, int j0, int jmax, float scale_log2, float m,
                                                uint32_t (&packed)[16], float& lq) {
    lq = 0.f;
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
        float p0 = 0.f, p1 = 0.f;
        if (j0 + j <= jmax) p0 = ex2(__fsub_rn(__fmul_rn(sv[j], scale_log2), m));
        if (j0 + j + 1 <= jmax) p1 = ex2(__fsub_rn(__fmul_rn(sv[j + 1], scale_log2), m));
        const __nv_bfloat162 pb = __floats2bfloat162_rn(p0, p1);
        lq = __fadd_rn(lq, __low2float(pb));
        lq = __fadd_rn(lq, __high2float(pb));
        packed[j >> 1] = *reinterpret_cast<const uint32_t*>(&pb);
    }
}
__device__ __forceinline__ void store_p_quarter(uint8_t* p_base, uint32_t p_sub_stride, int prow, int q,
                                                const uint32_t (&packed)[16]) {
    uint8_t* psub = p_base + (q >> 1) * p_sub_stride;
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4)
        *reinterpret_cast<uint4*>(psub + sw_off(prow, (q & 1) * 4 + q4)) =
            make_uint4(packed[4 * q4], packed[4 * q4 + 1], packed[4 * q4 + 2], packed[4 * q4 + 3]);
}
__device__ __forceinline__ float quarter_max(const float* sv, int j0, int jmax, float scale_log2) {
    float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
    for (int j = 0; j < 32; ++j)
        if (j0 + j <= jmax) mx[j & 3] = fmaxf(mx[j & 3], __fmul_rn(sv[j], scale_log2));
    return fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
}

// Thread-per-row form (prefill): this thread's S row is at s_taddr in TMEM.
__device__ __forceinline__ void softmax_row(uint32_t s_taddr, int jmax, float scale_log2, uint8_t* p_base,
                                            uint32_t p_sub_stride, int prow, bool write_p, float& m_out,
                                            float& l_out) {
    float m = -INFINITY;
#pragma unroll
    for (int cb = 0; cb < 4; ++cb) {
        float sv[32];
        ptx::tmem_ld<32>(s_taddr + cb * 32, sv);
        ptx::tmem_wait_ld();
        m = fmaxf(m, quarter_max(sv, cb * 32, jmax, scale_log2));
    }
    float lq[4];
#pragma unroll
    for (int cb = 0; cb < 4; ++cb) {
        float sv[32];
        ptx::tmem_ld<32>(s_taddr + cb * 32, sv);
        ptx::tmem_wait_ld();
        uint32_t packed[16];
        softmax_quarter(sv, cb * 32, jmax, scale_log2, m, packed, lq[cb]);
        if (write_p) store_p_quarter(p_base, p_sub_stride, prow, cb, packed);
    }
    m_out = m;
    l_out = __fadd_rn(__fadd_rn(__fadd_rn(lq[0], lq[1]), lq[2]), lq[3]);
}

// Four-lanes-per-row form (decode): rows 0..7 of the chunk, lane L works on row
// L / 4, keys 32 (L % 4) .. +31.  srow: this warp's 8 x 128 fp32 staging area.
// Every lane returns its row's m and l.
__device__ __forceinline__ void softmax_rows8(uint32_t s_taddr, float* srow, int jmax_of_row, float scale_log2,
                                              uint8_t* p_base, uint32_t p_sub_stride, float& m_out, float& l_out) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int cb = 0; cb < 4; ++cb) {
        float sv[32];
        ptx::tmem_ld<32>(s_taddr + cb * 32, sv);
        ptx::tmem_wait_ld();
        if (lane < 8)
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4)
                *reinterpret_cast<float4*>(srow + lane * 128 + cb * 32 + 4 * q4) =
                    make_float4(sv[4 * q4], sv[4 * q4 + 1], sv[4 * q4 + 2], sv[4 * q4 + 3]);
    }
    __syncwarp();
    const int r = lane >> 2, q = lane & 3;
    float sv[32];
#pragma unroll
    for (int q4 = 0; q4 < 8; ++q4) {
        const float4 v = *reinterpret_cast<const float4*>(srow + r * 128 + q * 32 + 4 * q4);
        sv[4 * q4] = v.x; sv[4 * q4 + 1] = v.y; sv[4 * q4 + 2] = v.z; sv[4 * q4 + 3] = v.w;
    }
    const int jmax = __shfl_sync(0xffffffffu, jmax_of_row, r);
    float m = quarter_max(sv, q * 32, jmax, scale_log2);
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
    uint32_t packed[16];
    float lq;
    softmax_quarter(sv, q * 32, jmax, scale_log2, m, packed, lq);
    store_p_quarter(p_base, p_sub_stride, r, q, packed);
    const float l0 = __shfl_sync(0xffffffffu, lq, r * 4), l1 = __shfl_sync(0xffffffffu, lq, r * 4 + 1);
    const float l2 = __shfl_sync(0xffffffffu, lq, r * 4 + 2), l3 = __shfl_sync(0xffffffffu, lq, r * 4 + 3);
    const float l = __fadd_rn(__fadd_rn(__fadd_rn(l0, l1), l2), l3);
    // hand row r's (m, l) back to lane r
    m_out = __shfl_sync(0xffffffffu, m, (lane & 7) * 4);
    l_out = __shfl_sync(0xffffffffu, l, (lane & 7) * 4);
    __syncwarp();
}

template <bool DECODE>
__global__ void __launch_bounds__(kThreads, 1)
    k_attn_tc(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
              const __grid_constant__ CUtensorMap mV, const TcArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t* bars = (uint64_t*)(sm + OFF_BAR);
    uint64_t* q_full = bars + 0;
    uint64_t* kv_full = bars + 1;    // [2]
    uint64_t* kv_empty = bars + 3;   // [2]
    uint64_t* s_full = bars + 5;
    uint64_t* s_empty = bars + 6;
    uint64_t* p_full = bars + 7;
    uint64_t* o_full = bars + 8;
    uint64_t* oc_empty = bars + 9;
    uint32_t* tmem_holder = (uint32_t*)(bars + 10);
    constexpr uint32_t TMEM_COLS = DECODE ? 256 : 512;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    ptx::griddep_wait();   // q and the cache rows come from the projection kernels
    if (threadIdx.x == 0) ptx::griddep_launch_dependents();

    const int g = blockIdx.y, b = blockIdx.z;
    const int n_rep = a.n_heads / a.n_kv_heads;
    const int base = a.pos_dev ? *a.pos_dev : a.start_pos;
    int t0 = 0, c_begin = 0, c_end = 0, kv_last = 0;
    if constexpr (DECODE) {
        if (base < 0 || base >= a.max_pos) {
            if (threadIdx.x == 0 && blockIdx.x == 0 && g == 0 && b == 0) record_error(a.err, LLAMA_ERR_POS_RANGE);
            return;
        }
        kv_last = base;
        const int n_total = base / kAttnChunk + 1;
        c_begin = blockIdx.x * a.chunks_per_cta;
        c_end = min(c_begin + a.chunks_per_cta, n_total);
        if (c_begin >= c_end) return;
    } else {
        t0 = (gridDim.x - 1 - blockIdx.x) * a.tq;   // longest tiles first
        const int t_last = min(t0 + a.tq, a.tokens) - 1;
        if (base < 0 || base + t_last >= a.max_pos) {
            if (threadIdx.x == 0) record_error(a.err, LLAMA_ERR_POS_RANGE);
            return;
        }
        kv_last = base + t_last;
        c_end = kv_last / kAttnChunk + 1;
    }
    const int n_iter = c_end - c_begin;
    int* err = a.err;

    if (threadIdx.x == 0) {
        ptx::mbar_init(q_full, 1);
        for (int i = 0; i < 2; ++i) { ptx::mbar_init(&kv_full[i], 1); ptx::mbar_init(&kv_empty[i], 1); }
        ptx::mbar_init(s_full, 1);
        ptx::mbar_init(s_empty, 4);
        ptx::mbar_init(p_full, 4);
        ptx::mbar_init(o_full, 1);
        ptx::mbar_init(oc_empty, 4);
        ptx::fence_mbar_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc(tmem_holder, TMEM_COLS);
        ptx::tmem_relinquish();
    }
    if constexpr (DECODE) {
        // decode query tile: rows 0..n_rep-1 = the group's heads, the rest zero
        if (warp >= 2) {
            const int r = threadIdx.x - 64;
            for (int half = 0; half < 2; ++half) {
                uint8_t* sub = sm + OFF_Q + half * kSub;
                for (int c = 0; c < 8; ++c) {
                    uint4 v = make_uint4(0, 0, 0, 0);
                    if (r < n_rep)
                        v = *reinterpret_cast<const uint4*>(a.q + (size_t)b * a.n_heads * 128 +
                                                            (size_t)(g * n_rep + r) * 128 + half * 64 + c * 8);
                    *reinterpret_cast<uint4*>(sub + sw_off(r, c)) = v;
                }
            }
            ptx::fence_proxy_async_smem();
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp == 0) {
        // ------------------------------------------------------------------ TMA producer
        if (lane == 0) {
            ptx::prefetch_tmap(&mK);
            ptx::prefetch_tmap(&mV);
            if constexpr (!DECODE) {
                ptx::prefetch_tmap(&mQ);
                ptx::mbar_arrive_expect_tx(q_full, 2 * kSub);
                asm volatile(
                    "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                    " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(ptx::smem_u32(sm + OFF_Q)),
                    "l"(reinterpret_cast<uint64_t>(&mQ)), "r"(ptx::smem_u32(q_full)), "r"(0), "r"(g * n_rep),
                    "r"(b * a.tokens + t0)
                    : "memory");
                asm volatile(
                    "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                    " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(ptx::smem_u32(sm + OFF_Q + kSub)),
                    "l"(reinterpret_cast<uint64_t>(&mQ)), "r"(ptx::smem_u32(q_full)), "r"(64), "r"(g * n_rep),
                    "r"(b * a.tokens + t0)
                    : "memory");
            }
            const int head_row0 = (b * a.n_kv_heads + g) * a.kv_seq;
            for (int i = 0; i < n_iter; ++i) {
                const int st = i & 1;
                if (i >= 2 && !ptx::mbar_wait(&kv_empty[st], ((i >> 1) & 1) ^ 1, err)) break;
                uint8_t* kv = sm + OFF_KV + st * KV_STAGE;
                const int row = head_row0 + (c_begin + i) * kAttnChunk;
                ptx::mbar_arrive_expect_tx(&kv_full[st], 4 * kSub);
                ptx::tma_load_2d(kv, &mK, &kv_full[st], 0, row);
                ptx::tma_load_2d(kv + kSub, &mK, &kv_full[st], 64, row);
                ptx::tma_load_2d(kv + 2 * kSub, &mV, &kv_full[st], 0, row);
                ptx::tma_load_2d(kv + 3 * kSub, &mV, &kv_full[st], 64, row);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            bool ok = DECODE ? true : ptx::mbar_wait(q_full, 0, err);
            const uint32_t q_addr = ptx::smem_u32(sm + OFF_Q);
            const uint32_t p_addr = ptx::smem_u32(sm + OFF_P);
            for (int i = 0; i < n_iter && ok; ++i) {
                const int st = i & 1;
                const uint32_t k_addr = ptx::smem_u32(sm + OFF_KV + st * KV_STAGE);
                const uint32_t v_addr = k_addr + 2 * kSub;
                if (!ptx::mbar_wait(&kv_full[st], (i >> 1) & 1, err)) break;
                if (i > 0 && !ptx::mbar_wait(s_empty, (i - 1) & 1, err)) break;
                ptx::tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t off = (ks >> 2) * kSub + (ks & 3) * 32;
                    ptx::umma_bf16(tmem + TM_S, ptx::sw128_kmajor_desc(q_addr + off),
                                   ptx::sw128_kmajor_desc(k_addr + off), IDESC_S, ks > 0 ? 1u : 0u);
                }
                ptx::umma_commit(s_full);
                if (!ptx::mbar_wait(p_full, i & 1, err)) break;
                if (i > 0 && !ptx::mbar_wait(oc_empty, (i - 1) & 1, err)) break;
                ptx::tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t aoff = (ks >> 2) * kSub + (ks & 3) * 32;
                    ptx::umma_bf16(tmem + TM_OC, ptx::sw128_kmajor_desc(p_addr + aoff),
                                   ptx::sw128_mnmajor_desc(v_addr + ks * 2048, kSub), IDESC_PV, ks > 0 ? 1u : 0u);
                }
                ptx::umma_commit(o_full);
                ptx::umma_commit(&kv_empty[st]);
            }
        }
    } else {
        // ------------------------------------------------------------------ softmax + fold, thread = row
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
        const int t_local = row / n_rep, h_local = row - t_local * n_rep;
        bool valid;
        int pos_r;
        if constexpr (DECODE) {
            valid = row < n_rep;
            pos_r = base;
        } else {
            valid = (t_local < a.tq) && (t0 + t_local < a.tokens);
            pos_r = base + t0 + t_local;
        }
        float M = -INFINITY, L = 0.f;
        bool ok = true;
        for (int i = 0; i < n_iter; ++i) {
            const int c = c_begin + i;
            const int st = i & 1;
            if (ok) ok = ptx::mbar_wait(s_full, i & 1, err);
            ptx::tc_fence_after();
            const int jmax = valid ? min(kAttnChunk - 1, pos_r - c * kAttnChunk) : -1;
            float m, l;
            softmax_row(tmem + lane_addr + TM_S, jmax, a.scale_log2, sm + OFF_P, kSub, row, true, m, l);
            ptx::tc_fence_before();
            // value rows past the last visible key of this tile are zeroed (they may hold
            // anything, including NaN; P is 0 there and 0 * NaN would poison O)
            if (c * kAttnChunk + row > kv_last) {
                uint8_t* vrow = sm + OFF_KV + st * KV_STAGE + 2 * kSub + row * 128;
#pragma unroll
                for (int c16 = 0; c16 < 8; ++c16) {
                    *reinterpret_cast<uint4*>(vrow + c16 * 16) = make_uint4(0, 0, 0, 0);
                    *reinterpret_cast<uint4*>(vrow + kSub + c16 * 16) = make_uint4(0, 0, 0, 0);
                }
            }
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                ptx::mbar_arrive(s_empty);
                ptx::mbar_arrive(p_full);
            }
            if (ok) ok = ptx::mbar_wait(o_full, i & 1, err);
            ptx::tc_fence_after();
            if constexpr (DECODE) {
                float* dst = a.partial + ((((size_t)b * a.n_kv_heads + g) * a.n_chunks + c) * n_rep + row) * kPartStride;
#pragma unroll
                for (int cb = 0; cb < 4; ++cb) {
                    float ov[32];
                    ptx::tmem_ld<32>(tmem + lane_addr + TM_OC + cb * 32, ov);
                    ptx::tmem_wait_ld();
                    if (valid)
#pragma unroll
                        for (int q4 = 0; q4 < 8; ++q4)
                            *reinterpret_cast<float4*>(dst + cb * 32 + 4 * q4) =
                                make_float4(ov[4 * q4], ov[4 * q4 + 1], ov[4 * q4 + 2], ov[4 * q4 + 3]);
                }
                if (valid) {
                    dst[128] = m;
                    dst[129] = l;
                }
            } else {
                // fold the chunk into the running state (the combine kernel's formula)
                float alpha = 1.f, beta = 0.f;
                const bool first = (i == 0);
                if (!first) {
                    const float Mn = fmaxf(M, m);
                    alpha = exp2f(__fsub_rn(M, Mn));
                    beta = exp2f(__fsub_rn(m, Mn));
                    L = __fmaf_rn(L, alpha, __fmul_rn(l, beta));
                    M = Mn;
                } else {
                    M = m;
                    L = l;
                }
#pragma unroll
                for (int cb = 0; cb < 4; ++cb) {
                    float oc[32], orun[32];
                    ptx::tmem_ld<32>(tmem + lane_addr + TM_OC + cb * 32, oc);
                    if (!first) ptx::tmem_ld<32>(tmem + lane_addr + TM_O + cb * 32, orun);
                    ptx::tmem_wait_ld();
                    if (first) {
#pragma unroll
                        for (int j = 0; j < 32; ++j) orun[j] = oc[j];
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j) orun[j] = __fmaf_rn(orun[j], alpha, __fmul_rn(oc[j], beta));
                    }
                    ptx::tmem_st32(tmem + lane_addr + TM_O + cb * 32, orun);
                }
                ptx::tmem_wait_st();
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(oc_empty);
        }
        if constexpr (!DECODE) {
            // o = O / L, rounded to bf16
            ptx::tc_fence_after();
            bf16* dst = a.o + ((size_t)b * a.tokens + t0 + t_local) * a.n_heads * 128 + (size_t)(g * n_rep + h_local) * 128;
#pragma unroll
            for (int cb = 0; cb < 4; ++cb) {
                float ov[32];
                ptx::tmem_ld<32>(tmem + lane_addr + TM_O + cb * 32, ov);
                ptx::tmem_wait_ld();
                if (valid && ok) {
                    uint32_t packed[16];
#pragma unroll
                    for (int j = 0; j < 32; j += 2) {
                        const __nv_bfloat162 v2 = __floats2bfloat162_rn(__fdiv_rn(ov[j], L), __fdiv_rn(ov[j + 1], L));
                        packed[j >> 1] = *reinterpret_cast<const uint32_t*>(&v2);
                    }
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4)
                        *reinterpret_cast<uint4*>(dst + cb * 32 + 8 * q4) =
                            make_uint4(packed[4 * q4], packed[4 * q4 + 1], packed[4 * q4 + 2], packed[4 * q4 + 3]);
                }
            }
        }
    }

    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, TMEM_COLS);
    }
}

// ----------------------------------------------------------------------------- decode
// Persistent decode attention for groups of n_rep <= 8 query heads.  The work
// units are (sequence, KV head, chunk); CTA i walks a contiguous range of them.
// Query and P tiles hold 8 rows; their descriptors use an 8-row-group stride of
// 0, so the MMA's 128 rows alias those 8 (rows 8..127 repeat rows 0..7 and are
// ignored).  Two TMEM slots (S and O_c of one unit share a slot's 128 columns)
// and two softmax warps take alternate units; the MMA thread issues S of unit
// i+1 before PV of unit i, so the tensor core works while a softmax runs; K/V
// stream through a three-stage TMA ring.  Warps: 0 and 4 = softmax + partial
// store for slots 0 and 1 (rows 0..7 are TMEM lanes 0..7, which warps 0 and 4
// may read), 1 = TMA producer, 2 = TMEM owner + MMA issuer, 3 idle.
constexpr int kDecThreads = 160;
constexpr int kDecStages = 3;
constexpr int D_OFF_Q = 0;                              // [slot][half] 1 KB each
constexpr int D_OFF_P = 4096;                           // [slot][half] 1 KB each
constexpr int D_OFF_S = 8192;                           // [slot] 8 x 128 fp32 score staging
constexpr int D_OFF_KV = 16384;                         // [stage] K: 2 sub-tiles, V: 2 sub-tiles
constexpr int D_OFF_BAR = D_OFF_KV + kDecStages * 4 * kSub;
constexpr int D_SMEM_BYTES = D_OFF_BAR + 256 + 1024;

__device__ __forceinline__ uint64_t sw128_kmajor_desc_rows8(uint32_t smem_addr) {
    return ptx::sw128_kmajor_desc(smem_addr) & ~(0x3FFFull << 32);   // stride byte offset 0
}

struct DecUnit {
    int b, g, c;
};
__device__ __forceinline__ DecUnit dec_unit(int u, int n_total, int n_kv) {
    DecUnit d;
    d.c = u % n_total;
    const int bg = u / n_total;
    d.g = bg % n_kv;
    d.b = bg / n_kv;
    return d;
}

__global__ void __launch_bounds__(kDecThreads, 1) k_attn_tc_dec(const __grid_constant__ CUtensorMap mK,
                                                                const __grid_constant__ CUtensorMap mV,
                                                                const TcArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t* bars = (uint64_t*)(sm + D_OFF_BAR);
    uint64_t* kv_full = bars + 0;             // [3]
    uint64_t* kv_empty = bars + 3;            // [3]
    uint64_t* slot_ready = bars + 6;          // [2] query tile filled, previous unit of the slot drained
    uint64_t* s_full = bars + 8;              // [2]
    uint64_t* p_full = bars + 10;             // [2]
    uint64_t* o_full = bars + 12;             // [2]
    uint32_t* tmem_holder = (uint32_t*)(bars + 14);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // The position comes from the host side (set before the step is launched), not
    // from the kernels this one overlaps; cache rows below it were written by
    // earlier steps.  Only q and the newest cache row need griddepcontrol.wait.
    const int n_rep = a.n_heads / a.n_kv_heads;
    const int pos = a.pos_dev ? *a.pos_dev : a.start_pos;
    if (pos < 0 || pos >= a.max_pos) {
        if (threadIdx.x == 0 && blockIdx.x == 0) record_error(a.err, LLAMA_ERR_POS_RANGE);
        return;
    }
    const int n_total = pos / kAttnChunk + 1;
    const int n_units = a.batch * a.n_kv_heads * n_total;
    const int u_begin = (int)(((long)n_units * blockIdx.x) / gridDim.x);
    const int u_end = (int)(((long)n_units * (blockIdx.x + 1)) / gridDim.x);
    const int n_iter = u_end - u_begin;
    if (n_iter <= 0) return;
    int* err = a.err;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kDecStages; ++i) { ptx::mbar_init(&kv_full[i], 1); ptx::mbar_init(&kv_empty[i], 1); }
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(&slot_ready[i], 1);
            ptx::mbar_init(&s_full[i], 1);
            ptx::mbar_init(&p_full[i], 1);
            ptx::mbar_init(&o_full[i], 1);
        }
        ptx::fence_mbar_init();
    }
    if (warp == 2) {
        ptx::tmem_alloc(tmem_holder, 256);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp == 1) {
        // ------------------------------------------------------------------ TMA producer
        if (lane == 0) {
            ptx::prefetch_tmap(&mK);
            ptx::prefetch_tmap(&mV);
            bool waited = false;
            for (int i = 0; i < n_iter; ++i) {
                const int st = i % kDecStages;
                if (i >= kDecStages && !ptx::mbar_wait(&kv_empty[st], ((i / kDecStages) - 1) & 1, err)) break;
                const DecUnit d = dec_unit(u_begin + i, n_total, a.n_kv_heads);
                if (!waited && d.c == n_total - 1) {   // this chunk holds the row the QKV step writes
                    ptx::griddep_wait();
                    waited = true;
                }
                const int row = (d.b * a.n_kv_heads + d.g) * a.kv_seq + d.c * kAttnChunk;
                uint8_t* kv = sm + D_OFF_KV + st * 4 * kSub;
                ptx::mbar_arrive_expect_tx(&kv_full[st], 4 * kSub);
                ptx::tma_load_2d(kv, &mK, &kv_full[st], 0, row);
                ptx::tma_load_2d(kv + kSub, &mK, &kv_full[st], 64, row);
                ptx::tma_load_2d(kv + 2 * kSub, &mV, &kv_full[st], 0, row);
                ptx::tma_load_2d(kv + 3 * kSub, &mV, &kv_full[st], 64, row);
            }
        }
    } else if (warp == 2) {
        // ------------------------------------------------------------------ MMA issuer: S(i), then PV(i-1)
        if (lane == 0) {
            auto issue_pv = [&](int j) -> bool {
                const int slot = j & 1, st = j % kDecStages;
                if (!ptx::mbar_wait(&p_full[slot], (j >> 1) & 1, err)) return false;
                ptx::tc_fence_after();
                const uint32_t p_addr = ptx::smem_u32(sm + D_OFF_P + slot * 2048);
                const uint32_t v_addr = ptx::smem_u32(sm + D_OFF_KV + st * 4 * kSub + 2 * kSub);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    ptx::umma_bf16(tmem + slot * 128, sw128_kmajor_desc_rows8(p_addr + (ks >> 2) * 1024 + (ks & 3) * 32),
                                   ptx::sw128_mnmajor_desc(v_addr + ks * 2048, kSub), IDESC_PV, ks > 0 ? 1u : 0u);
                ptx::umma_commit(&o_full[slot]);
                ptx::umma_commit(&kv_empty[st]);
                return true;
            };
            bool ok = true;
            for (int i = 0; i < n_iter && ok; ++i) {
                const int slot = i & 1, st = i % kDecStages;
                if (!ptx::mbar_wait(&kv_full[st], (i / kDecStages) & 1, err)) { ok = false; break; }
                if (!ptx::mbar_wait(&slot_ready[slot], (i >> 1) & 1, err)) { ok = false; break; }
                ptx::tc_fence_after();
                const uint32_t q_addr = ptx::smem_u32(sm + D_OFF_Q + slot * 2048);
                const uint32_t k_addr = ptx::smem_u32(sm + D_OFF_KV + st * 4 * kSub);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    ptx::umma_bf16(tmem + slot * 128, sw128_kmajor_desc_rows8(q_addr + (ks >> 2) * 1024 + (ks & 3) * 32),
                                   ptx::sw128_kmajor_desc(k_addr + (ks >> 2) * kSub + (ks & 3) * 32), IDESC_S,
                                   ks > 0 ? 1u : 0u);
                ptx::umma_commit(&s_full[slot]);
                if (i > 0) ok = issue_pv(i - 1);
            }
            if (ok) issue_pv(n_iter - 1);
        }
    } else if (warp == 0 || warp == 4) {
        // ------------------------------------------------------------------ softmax + partial store
        const int slot = warp >> 2;
        const bool valid = lane < n_rep;
        const uint32_t taddr = tmem + slot * 128;   // TMEM lanes 0..31 (warp 0 and warp 4)
        uint8_t* qs = sm + D_OFF_Q + slot * 2048;
        uint8_t* ps = sm + D_OFF_P + slot * 2048;
        float* srow = reinterpret_cast<float*>(sm + D_OFF_S + slot * 4096);
        ptx::griddep_wait();   // q comes from the QKV step
        if (threadIdx.x == 0) ptx::griddep_launch_dependents();
        int q_bg = -1;         // (sequence, KV head) whose query rows the slot's tile holds
        bool ok = true;
        for (int i = slot, k = 0; i < n_iter; i += 2, ++k) {
            const DecUnit d = dec_unit(u_begin + i, n_total, a.n_kv_heads);
            const int st = i % kDecStages;
            const int bg = d.b * a.n_kv_heads + d.g;
            if (bg != q_bg) {
                // query rows 0..n_rep-1 of (b, g), zero rows up to 8
                if (lane < 8) {
#pragma unroll
                    for (int half = 0; half < 2; ++half)
#pragma unroll
                        for (int c = 0; c < 8; ++c) {
                            uint4 v = make_uint4(0, 0, 0, 0);
                            if (valid)
                                v = *reinterpret_cast<const uint4*>(a.q + (size_t)d.b * a.n_heads * 128 +
                                                                    (size_t)(d.g * n_rep + lane) * 128 + half * 64 + c * 8);
                            *reinterpret_cast<uint4*>(qs + half * 1024 + sw_off(lane, c)) = v;
                        }
                }
                q_bg = bg;
                ptx::fence_proxy_async_smem();
            }
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&slot_ready[slot]);
            if (ok) ok = ptx::mbar_wait(&s_full[slot], k & 1, err);
            ptx::tc_fence_after();
            const int jmax = valid ? min(kAttnChunk - 1, pos - d.c * kAttnChunk) : -1;
            float m, l;
            softmax_rows8(taddr, srow, jmax, a.scale_log2, ps, 1024, m, l);
            ptx::tc_fence_before();
            // value rows past the position hold anything (NaN included): zero them
            if (d.c == n_total - 1) {
#pragma unroll
                for (int r4 = 0; r4 < 4; ++r4) {
                    const int vr = lane + 32 * r4;
                    if (d.c * kAttnChunk + vr > pos) {
                        uint8_t* vrow = sm + D_OFF_KV + st * 4 * kSub + 2 * kSub + vr * 128;
#pragma unroll
                        for (int c16 = 0; c16 < 8; ++c16) {
                            *reinterpret_cast<uint4*>(vrow + c16 * 16) = make_uint4(0, 0, 0, 0);
                            *reinterpret_cast<uint4*>(vrow + kSub + c16 * 16) = make_uint4(0, 0, 0, 0);
                        }
                    }
                }
            }
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&p_full[slot]);
            if (ok) ok = ptx::mbar_wait(&o_full[slot], k & 1, err);
            ptx::tc_fence_after();
            float* dst = a.partial + ((((size_t)d.b * a.n_kv_heads + d.g) * a.n_chunks + d.c) * n_rep + lane) * kPartStride;
#pragma unroll
            for (int cb = 0; cb < 4; ++cb) {
                float ov[32];
                ptx::tmem_ld<32>(taddr + cb * 32, ov);
                ptx::tmem_wait_ld();
                if (valid)
#pragma unroll
                    for (int q4 = 0; q4 < 8; ++q4)
                        *reinterpret_cast<float4*>(dst + cb * 32 + 4 * q4) =
                            make_float4(ov[4 * q4], ov[4 * q4 + 1], ov[4 * q4 + 2], ov[4 * q4 + 3]);
            }
            if (valid) {
                dst[128] = m;
                dst[129] = l;
            }
            ptx::tc_fence_before();
        }
    }
    __syncthreads();
    if (warp == 2) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 256);
    }
}

bool make_tmap_q3d(CUtensorMap* map, const void* q, int n_heads, int tokens, int n_rep, int tq) {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult qr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &qr) !=
                cudaSuccess ||
            qr != cudaDriverEntryPointSuccess)
            return false;
        fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    cuuint64_t dims[3] = {128, (cuuint64_t)n_heads, (cuuint64_t)tokens};
    cuuint64_t strides[2] = {128 * 2, (cuuint64_t)n_heads * 128 * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)n_rep, (cuuint32_t)tq};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

TcArgs make_args(const AttnArgs& a) {
    TcArgs k{};
    k.batch = a.batch;
    k.tokens = a.tokens;
    k.n_heads = a.n_heads;
    k.n_kv_heads = a.n_kv_heads;
    k.kv_seq = a.kv_seq;
    k.start_pos = a.start_pos;
    k.max_pos = a.max_pos;
    k.pos_dev = a.pos_dev;
    k.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)a.head_dim));
    k.q = (const bf16*)a.q;
    k.o = (bf16*)a.o;
    k.partial = a.partial;
    k.n_chunks = a.n_chunks;
    k.err = a.err;
    return k;
}

}  // namespace

bool attention_tc_supported(int n_heads, int n_kv_heads, int head_dim) {
    const int n_rep = n_heads / n_kv_heads;
    return head_dim == 128 && n_rep >= 1 && n_rep <= 128 && (128 % n_rep) == 0;
}

cudaError_t launch_attention_tc_prefill(const AttnArgs& a, cudaStream_t s) {
    if (a.batch <= 0 || a.tokens <= 0) return cudaSuccess;
    if (!attention_tc_supported(a.n_heads, a.n_kv_heads, a.head_dim)) return cudaErrorInvalidValue;
    TcArgs k = make_args(a);
    const int n_rep = a.n_heads / a.n_kv_heads;
    k.tq = 128 / n_rep;
    CUtensorMap mq, mk, mv;
    if (!make_tmap_q3d(&mq, a.q, a.n_heads, a.batch * a.tokens, n_rep, k.tq)) return cudaErrorInvalidValue;
    const uint64_t cache_rows = (uint64_t)a.batch * a.n_kv_heads * a.kv_seq;
    if (!make_tmap_bf16(&mk, a.kc, cache_rows, 128, 128, nullptr) ||
        !make_tmap_bf16(&mv, a.vc, cache_rows, 128, 128, nullptr))
        return cudaErrorInvalidValue;
    auto kern = k_attn_tc<false>;
    static bool attr = false;
    if (!attr) {
        cudaError_t r = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
        if (r != cudaSuccess) return r;
        attr = true;
    }
    dim3 grid((a.tokens + k.tq - 1) / k.tq, a.n_kv_heads, a.batch);
    return launch_pdl(kern, grid, dim3(kThreads), SMEM_BYTES, s, mq, mk, mv, k);
}

cudaError_t launch_attention_tc_decode(const AttnArgs& a, int chunks_per_cta, cudaStream_t s) {
    if (a.batch <= 0) return cudaSuccess;
    if (!attention_tc_supported(a.n_heads, a.n_kv_heads, a.head_dim)) return cudaErrorInvalidValue;
    TcArgs k = make_args(a);
    CUtensorMap mk, mv;
    const uint64_t cache_rows = (uint64_t)a.batch * a.n_kv_heads * a.kv_seq;
    if (!make_tmap_bf16(&mk, a.kc, cache_rows, 128, 128, nullptr) ||
        !make_tmap_bf16(&mv, a.vc, cache_rows, 128, 128, nullptr))
        return cudaErrorInvalidValue;
    const int n_rep = a.n_heads / a.n_kv_heads;
    if (n_rep <= 8) {
        // persistent: one CTA per SM (units assigned on the device from the position)
        static const int n_sm = device_sm_count();
        const long max_units = (long)a.batch * a.n_kv_heads * a.n_chunks;
        static bool attr_dec = false;
        if (!attr_dec) {
            cudaError_t r = cudaFuncSetAttribute(k_attn_tc_dec, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 D_SMEM_BYTES);
            if (r != cudaSuccess) return r;
            attr_dec = true;
        }
        dim3 grid((unsigned)std::min<long>(max_units, n_sm));
        cudaError_t r = launch_pdl(k_attn_tc_dec, grid, dim3(kDecThreads), D_SMEM_BYTES, s, mk, mv, k);
        if (r != cudaSuccess) return r;
        return launch_attention_combine(a, s);
    }
    if (chunks_per_cta <= 0) chunks_per_cta = 2;
    k.chunks_per_cta = chunks_per_cta;
    auto kern = k_attn_tc<true>;
    static bool attr = false;
    if (!attr) {
        cudaError_t r = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
        if (r != cudaSuccess) return r;
        attr = true;
    }
    dim3 grid((a.n_chunks + chunks_per_cta - 1) / chunks_per_cta, a.n_kv_heads, a.batch);
    cudaError_t r = launch_pdl(kern, grid, dim3(kThreads), SMEM_BYTES, s, mk, mk, mv, k);
    if (r != cudaSuccess) return r;
    return launch_attention_combine(a, s);
}

}  // namespace llama
