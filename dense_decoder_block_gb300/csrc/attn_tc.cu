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
// of one token.
//   S   = Q K^T        tcgen05.mma M=128 N=128 K=128, both operands K-major
//   softmax of each row over the chunk (softmax_keys below gives the exact
//         definition every kernel follows), P rounded to bf16
//   O_c = P V          tcgen05.mma M=128 N=128 K=128, V MN-major (as cached)
// Chunks are folded in ascending order from chunk 0 with one fold formula:
// prefill folds as it walks the chunks, decode stores each chunk's (O_c, m, l)
// and the combine kernel (attn_simt.cu) folds them in the same order, so a
// decode row equals the prefill row at the same position bit for bit.
// Kernels: k_attn_pf (prefill), k_attn_tc_dec (decode, up to 8 query heads per
// KV head), k_attn_tc_wide (decode, larger groups).
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
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
constexpr int TM_S = 0, TM_OC = 128;   // TMEM columns
constexpr uint32_t IDESC_S = ptx::idesc_bf16_f32(128, 128);
constexpr uint32_t IDESC_PV = ptx::idesc_bf16_f32_bmn(128, 128);

struct TcArgs {
    int batch, tokens, n_heads, n_kv_heads, kv_seq, start_pos, max_pos;
    const int* pos_dev;
    const int* pos_seq;  // decode: sequence b at position pos_seq[b] (the k_attn_tc_dec kernel only)
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

// 2^x on the special-function unit (PTX ex2.approx.ftz: max relative error
// 2^-22, far below the bf16 rounding of p that follows; results below the
// smallest normal float are flushed to zero).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Two fp32 lanes in one 64-bit register pair, for the packed f32x2 arithmetic of
// sm_100 and later: each lane is the IEEE round-to-nearest operation of its scalar
// form (no flush to zero), so a packed result equals the two scalar results bit for
// bit -- it halves the instructions, not the precision.
__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void unpack2(uint64_t v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {   // a * b + c, one rounding
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

// acc + (the bf16 in the low / high half of p), exactly fadd(acc, float(half)):
// the mixed-precision add widens its bf16 operand exactly and rounds once.
__device__ __forceinline__ float add_bf16_lo(uint32_t p, float acc) {
    float r;
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tadd.rn.f32.bf16 %0, lo, %2;\n\t}"
        : "=f"(r) : "r"(p), "f"(acc));
    return r;
}
__device__ __forceinline__ float add_bf16_hi(uint32_t p, float acc) {
    float r;
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tadd.rn.f32.bf16 %0, hi, %2;\n\t}"
        : "=f"(r) : "r"(p), "f"(acc));
    return r;
}
// max(a, b, c), exact like every max
__device__ __forceinline__ float max3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// The softmax of one query row over one 128-key chunk.  Every kernel computes
// exactly this (prefill with one thread per row, decode with four lanes per row):
//   m   = c * max_{j <= jmax} S_j,  c = log2(e) / sqrt(d_h)   (keys 0..jmax visible;
//         jmax < 0: none, m = -inf); rounding is monotonic, so this equals the
//         max of the rounded products c * S_j whatever the order
//   p_j = bf16(2^fma(S_j, c, -m)), 0 for hidden keys
//   l   = ((L0 + L1) + L2) + L3,  Lq = sum of p_j over keys 32q..32q+31 in key order
// The P row goes to the two 64-key sub-tiles of the swizzled K-major P operand
// (p_sub_stride bytes apart) at row `prow`.
template <int N>
__device__ __forceinline__ void softmax_keys(const float* sv, int j0, int jmax, float scale_log2, float m,
                                             uint32_t* packed, float& lq) {
    const uint64_t c2 = pack2(scale_log2, scale_log2), nm2 = pack2(-m, -m);
#pragma unroll
    for (int j = 0; j < N; j += 2) {
        float x0, x1;   // fma(S_j, c, -m) for the pair
        unpack2(fma2(pack2(sv[j], sv[j + 1]), c2, nm2), x0, x1);
        const float p0 = (j0 + j <= jmax) ? ex2(x0) : 0.f;
        const float p1 = (j0 + j + 1 <= jmax) ? ex2(x1) : 0.f;
        const __nv_bfloat162 pb = __floats2bfloat162_rn(p0, p1);
        packed[j >> 1] = *reinterpret_cast<const uint32_t*>(&pb);
        lq = add_bf16_hi(packed[j >> 1], add_bf16_lo(packed[j >> 1], lq));
    }
}
__device__ __forceinline__ void softmax_quarter(const float* sv, int j0, int jmax, float scale_log2, float m,
                                                uint32_t (&packed)[16], float& lq) {
    lq = 0.f;
    softmax_keys<32>(sv, j0, jmax, scale_log2, m, packed, lq);
}
__device__ __forceinline__ void store_p_quarter(uint8_t* p_base, uint32_t p_sub_stride, int prow, int q,
                                                const uint32_t (&packed)[16]) {
    uint8_t* psub = p_base + (q >> 1) * p_sub_stride;
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4)
        *reinterpret_cast<uint4*>(psub + sw_off(prow, (q & 1) * 4 + q4)) =
            make_uint4(packed[4 * q4], packed[4 * q4 + 1], packed[4 * q4 + 2], packed[4 * q4 + 3]);
}
// max of the visible raw scores among sv[0..31] (keys j0..j0+31); -inf if none
__device__ __forceinline__ float quarter_max_raw(const float* sv, int j0, int jmax) {
    float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
    for (int j = 0; j < 32; ++j)
        if (j0 + j <= jmax) mx[j & 3] = fmaxf(mx[j & 3], sv[j]);
    return fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
}


// Eight 32-bit TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&v)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(v[0]),
                 "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
                 : "memory");
}

// Eight K = 16 steps of one accumulator chain from a single asm block.  Step ks's
// descriptors are step 0's plus the step's byte offset / 16 in the start-address
// field (shared-memory addresses stay below 256 KB, so the 14-bit field never
// carries: the same descriptors the per-step helpers build), the accumulate
// predicate off for step 0 and on after.  The issuing thread shares its scheduler
// with softmax and fold warps; this keeps its instructions per MMA few.
//
// Both operands from shared memory.  A is K-major in two 64-column sub-tiles
// A_SUB16 x 16 bytes apart (step ks at (ks / 4) sub-tiles + (ks % 4) * 32 bytes);
// B likewise with B_SUB16, or MN-major (B_MN: step ks 16 rows = 2048 bytes on).
template <int A_SUB16, int B_SUB16, bool B_MN>
__device__ __forceinline__ void umma8_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc) {
#define LLAMA_AOFF(ks) ((ks) / 4 * A_SUB16 + (ks) % 4 * 2)
#define LLAMA_BOFF(ks) (B_MN ? (ks) * 128 : (ks) / 4 * B_SUB16 + (ks) % 4 * 2)
    asm volatile(
        "{\n\t.reg .pred pf, pt;\n\t.reg .b64 a<8>, b<8>;\n\t"
        "setp.ne.b32 pf, %3, %3;\n\tsetp.eq.b32 pt, %3, %3;\n\t"
        "add.s64 a1, %1, %4;\n\tadd.s64 b1, %2, %11;\n\t"
        "add.s64 a2, %1, %5;\n\tadd.s64 b2, %2, %12;\n\t"
        "add.s64 a3, %1, %6;\n\tadd.s64 b3, %2, %13;\n\t"
        "add.s64 a4, %1, %7;\n\tadd.s64 b4, %2, %14;\n\t"
        "add.s64 a5, %1, %8;\n\tadd.s64 b5, %2, %15;\n\t"
        "add.s64 a6, %1, %9;\n\tadd.s64 b6, %2, %16;\n\t"
        "add.s64 a7, %1, %10;\n\tadd.s64 b7, %2, %17;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, pf;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %3, pt;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], a2, b2, %3, pt;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], a3, b3, %3, pt;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], a4, b4, %3, pt;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], a5, b5, %3, pt;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], a6, b6, %3, pt;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], a7, b7, %3, pt;\n\t"
        "}" ::"r"(d), "l"(a), "l"(b), "r"(idesc),
        "n"(LLAMA_AOFF(1)), "n"(LLAMA_AOFF(2)), "n"(LLAMA_AOFF(3)), "n"(LLAMA_AOFF(4)), "n"(LLAMA_AOFF(5)),
        "n"(LLAMA_AOFF(6)), "n"(LLAMA_AOFF(7)), "n"(LLAMA_BOFF(1)), "n"(LLAMA_BOFF(2)), "n"(LLAMA_BOFF(3)),
        "n"(LLAMA_BOFF(4)), "n"(LLAMA_BOFF(5)), "n"(LLAMA_BOFF(6)), "n"(LLAMA_BOFF(7))
        : "memory");
#undef LLAMA_AOFF
#undef LLAMA_BOFF
}
// A from tensor memory (step ks 8 columns on: 16 bf16 per row), B MN-major from
// shared memory (step ks 16 rows = 2048 bytes on).
__device__ __forceinline__ void umma8_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc) {
    asm volatile(
        "{\n\t.reg .pred pf, pt;\n\t.reg .b32 t<8>;\n\t.reg .b64 b<8>;\n\t"
        "setp.ne.b32 pf, %3, %3;\n\tsetp.eq.b32 pt, %3, %3;\n\t"
        "add.u32 t1, %1, 8;\n\tadd.s64 b1, %2, 128;\n\t"
        "add.u32 t2, %1, 16;\n\tadd.s64 b2, %2, 256;\n\t"
        "add.u32 t3, %1, 24;\n\tadd.s64 b3, %2, 384;\n\t"
        "add.u32 t4, %1, 32;\n\tadd.s64 b4, %2, 512;\n\t"
        "add.u32 t5, %1, 40;\n\tadd.s64 b5, %2, 640;\n\t"
        "add.u32 t6, %1, 48;\n\tadd.s64 b6, %2, 768;\n\t"
        "add.u32 t7, %1, 56;\n\tadd.s64 b7, %2, 896;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, pf;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [t1], b1, %3, pt;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [t2], b2, %3, pt;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [t3], b3, %3, pt;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [t4], b4, %3, pt;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [t5], b5, %3, pt;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [t6], b6, %3, pt;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [t7], b7, %3, pt;\n\t"
        "}"
        ::"r"(d), "r"(a_tmem), "l"(b), "r"(idesc)
        : "memory");
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
        m = fmaxf(m, quarter_max_raw(sv, cb * 32, jmax));
    }
    m = __fmul_rn(m, scale_log2);
    float lq[4];
#pragma unroll
    for (int cb = 0; cb < 4; ++cb) {
        // 16 keys at a time (fewer live registers); the sum runs on in key order
        lq[cb] = 0.f;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            float sv[16];
            ptx::tmem_ld<16>(s_taddr + cb * 32 + hh * 16, sv);
            ptx::tmem_wait_ld();
            uint32_t packed[8];
            softmax_keys<16>(sv, cb * 32 + hh * 16, jmax, scale_log2, m, packed, lq[cb]);
            if (write_p) {
                uint8_t* psub = p_base + (cb >> 1) * p_sub_stride;
#pragma unroll
                for (int q4 = 0; q4 < 2; ++q4)
                    *reinterpret_cast<uint4*>(psub + sw_off(prow, (cb & 1) * 4 + hh * 2 + q4)) =
                        make_uint4(packed[4 * q4], packed[4 * q4 + 1], packed[4 * q4 + 2], packed[4 * q4 + 3]);
            }
        }
    }
    m_out = m;
    l_out = __fadd_rn(__fadd_rn(__fadd_rn(lq[0], lq[1]), lq[2]), lq[3]);
}


// Decode attention for groups of more than 8 query heads per KV head (a query
// tile holds the group's heads, the other rows are zero).  The chunks of one
// (sequence, KV head) are split over CTAs; each CTA stores every chunk's
// (O_c, m, l) for the combine kernel.  Warps: 0 = TMA producer, 1 = TMEM owner +
// MMA issuer, 2..5 = softmax + partial store (thread = row; warp w reads TMEM
// lane quarter w % 4).
__global__ void __launch_bounds__(kThreads, 1)
    k_attn_tc_wide(const __grid_constant__ CUtensorMap mK, const __grid_constant__ CUtensorMap mV, const TcArgs a) {
    TRACE(const unsigned long long tr0 = trace_stamp();)
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t* bars = (uint64_t*)(sm + OFF_BAR);
    uint64_t* kv_full = bars + 1;    // [2]
    uint64_t* kv_empty = bars + 3;   // [2]
    uint64_t* s_full = bars + 5;
    uint64_t* s_empty = bars + 6;
    uint64_t* p_full = bars + 7;
    uint64_t* o_full = bars + 8;
    uint64_t* oc_empty = bars + 9;
    uint32_t* tmem_holder = (uint32_t*)(bars + 10);
    constexpr uint32_t TMEM_COLS = 256;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    ptx::griddep_wait();   // q and the cache rows come from the projection kernels
    TRACE(const unsigned long long tr1 = trace_stamp();)

    const int g = blockIdx.y, b = blockIdx.z;
    const int n_rep = a.n_heads / a.n_kv_heads;
    const int base = a.pos_dev ? *a.pos_dev : a.start_pos;
    if (base < 0 || base >= a.max_pos) {
        if (threadIdx.x == 0 && blockIdx.x == 0 && g == 0 && b == 0) record_error(a.err, LLAMA_ERR_POS_RANGE);
        return;
    }
    const int kv_last = base;
    const int n_total = base / kAttnChunk + 1;
    const int c_begin = blockIdx.x * a.chunks_per_cta;
    const int c_end = min(c_begin + a.chunks_per_cta, n_total);
    if (c_begin >= c_end) return;
    const int n_iter = c_end - c_begin;
    int* err = a.err;

    if (threadIdx.x == 0) {
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
    // query tile: rows 0..n_rep-1 = the group's heads, the rest zero
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
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    // dependents start only once this CTA holds its tensor memory (one that started
    // earlier on this SM could take the columns and then wait for this grid)
    if (threadIdx.x == 0) ptx::griddep_launch_dependents();

    if (warp == 0) {
        // ------------------------------------------------------------------ TMA producer
        if (lane == 0) {
            ptx::prefetch_tmap(&mK);
            ptx::prefetch_tmap(&mV);
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
            bool ok = true;
            const uint32_t q_addr = ptx::smem_u32(sm + OFF_Q);
            const uint32_t p_addr = ptx::smem_u32(sm + OFF_P);
            for (int i = 0; i < n_iter && ok; ++i) {
                const int st = i & 1;
                const uint32_t k_addr = ptx::smem_u32(sm + OFF_KV + st * KV_STAGE);
                const uint32_t v_addr = k_addr + 2 * kSub;
                if (!ptx::mbar_wait(&kv_full[st], (i >> 1) & 1, err)) break;
                if (i > 0 && !ptx::mbar_wait(s_empty, (i - 1) & 1, err)) break;
                ptx::tc_fence_after();
                umma8_ss<kSub / 16, kSub / 16, false>(tmem + TM_S, ptx::sw128_kmajor_desc(q_addr),
                                                      ptx::sw128_kmajor_desc(k_addr), IDESC_S);
                ptx::umma_commit(s_full);
                if (!ptx::mbar_wait(p_full, i & 1, err)) break;
                if (i > 0 && !ptx::mbar_wait(oc_empty, (i - 1) & 1, err)) break;
                ptx::tc_fence_after();
                umma8_ss<kSub / 16, 0, true>(tmem + TM_OC, ptx::sw128_kmajor_desc(p_addr),
                                             ptx::sw128_mnmajor_desc(v_addr, kSub), IDESC_PV);
                ptx::umma_commit(o_full);
                ptx::umma_commit(&kv_empty[st]);
            }
        }
    } else {
        // ------------------------------------------------------------------ softmax + partial store, thread = row
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
        const bool valid = row < n_rep;
        const int pos_r = base;
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
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(oc_empty);
        }
    }

    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, TMEM_COLS);
    }
    TRACE(trace_cta(TR_ATTN_WIDE, tr0, tr1);)
}

// ----------------------------------------------------------------------------- prefill
// Pipelined prefill attention.  Same unit (one 128-row query tile of a KV group,
// its chunks in ascending order) and the same arithmetic as above, split over
// roles that overlap.  The kernel is persistent (at most one CTA per SM, each
// walking its tiles in turn) and every role counts the chunks of all its CTA's
// tiles in one sequence, so one tile's first copies and S MMAs overlap the
// previous tile's last softmax, fold and output store:
//   warp 0       TMA: each tile's Q (two buffers, the next tile's loading while
//                this one's S MMAs run), then its K chunks through a two-stage ring
//   warp 2       TMA: V chunks through a two-stage ring (K(i+2) loads once S(i)
//                has read K(i); V(i+2) once PV(i) has read V(i))
//   warp 1       TMEM owner + MMA: PV(i) into O_c with P read from TMEM, then
//                S(i+3) = Q K^T into the S buffer that chunk i used (three S
//                buffers, one O_c)
//   warps 4-11   softmax of every chunk, two threads per row: warps 4-7 take
//                keys 0..63 and warps 8-11 keys 64..127 of the rows of their
//                TMEM lane quarter, exchanging the row max and two quarter sums
//                through shared memory; P (bf16 pairs) overwrites the first 64
//                columns of the S row once both halves hold their scores, the
//                row's (m, l) goes to columns 64, 65.
//   warps 12-15  fold of every chunk into the running (O, M, L), thread = row,
//                with the row's O in registers; then o = O * (1 / L)
// Warp 3 only keeps the roles aligned to warpgroups.  A chunk that is wholly
// in a row's future (all its keys hidden) is skipped by that row's fold, so the
// row folds exactly chunks 0 .. pos / 128 -- the chunks a decode step at the
// same position folds.
constexpr int kPfThreads = 512;
// register split (launch: 128 per thread): warpgroup 0 and the softmax give up
// registers so that each fold thread can hold its row of O (128 floats)
constexpr int kPfRegsCtrl = 56;
constexpr int kPfRegsSoftmax = 112;
constexpr int kPfRegsFold = 232;
constexpr int kPfRegsNeeded = 128 * kPfRegsCtrl + 256 * kPfRegsSoftmax + 128 * kPfRegsFold;
static_assert(kPfRegsNeeded <= 128 * kPfThreads, "register split exceeds the launch allocation");
constexpr int PF_OFF_Q = 0;                          // [buffer] Q: 2 sub-tiles
constexpr int PF_OFF_K = 4 * kSub;                   // [stage] K: 2 sub-tiles
constexpr int PF_OFF_V = PF_OFF_K + 4 * kSub;        // [stage] V: 2 sub-tiles
constexpr int PF_OFF_BAR = PF_OFF_V + 4 * kSub;
constexpr int PF_OFF_XCH = PF_OFF_BAR + 256;         // softmax halves' exchange: 4 x 128 floats
constexpr int PF_SMEM_BYTES = PF_OFF_XCH + 2048 + 1024;
// S[i % 3] at columns 0 / 128 / 256, O_c at 384: three S buffers let S(i + 3) be
// issued behind PV(i), so the softmax works up to two chunks ahead of the MMAs
// that feed it; O_c needs one buffer, since the fold reads it before the softmax
// of the next chunk has finished.
constexpr int kPfSBufs = 3;
constexpr int PF_TM_S = 0, PF_TM_OC = 384;
// In S[parity], the softmax leaves P (bf16 pairs) in columns 0..63 and the row's
// (m, l) in columns 64, 65.
constexpr int PF_TM_ML = 64;
static_assert(PF_SMEM_BYTES <= 232448, "shared memory per CTA");

// Prefill softmax of one query row over one 128-key chunk, the keys split over
// two threads (two warps of the same TMEM lane quarter): half h holds keys
// 64h .. 64h+63 of the row's S in registers.  It computes exactly the canonical
// softmax: the row max over the visible keys is the max of the two halves' maxima
// (exchanged through shared memory; max is exact), p = bf16(2^(s c - m)) with
// hidden keys at -inf, and l = ((L0 + L1) + L2) + L3 with each quarter sum in
// ascending key order -- half 0 holds L0, L1, half 1 passes L2, L3 over.  Block c
// (keys 16c .. 16c+15) of P, packed as bf16 pairs, goes to columns 8c .. 8c+7 of
// the S row once both halves hold their scores in registers; half 0 writes the
// row's (m, l) to the ML columns.  `xch` is 4 x 128 floats of shared memory; `bar`
// the barrier id of this lane quarter.
__device__ __forceinline__ void softmax_half_tmem(uint32_t s_taddr, int h, int row, int jmax, float scale_log2,
                                                  float* xch, int bar, float& m_out) {
    float v[64];
    ptx::tmem_ld<32>(s_taddr + h * 64, v);
    ptx::tmem_ld<32>(s_taddr + h * 64 + 32, v + 32);
    ptx::tmem_wait_ld();
    const int jl = jmax - h * 64;   // last visible key of this half, local index
    const bool full = __all_sync(0xffffffffu, jl >= 63);
    float mx;
    if (full) {
        float a0 = v[0], a1 = v[1];
#pragma unroll
        for (int j = 2; j < 64; j += 4) {
            a0 = max3(a0, v[j], v[j + 1]);
            a1 = max3(a1, v[j + 2], v[j + 3]);
        }
        mx = fmaxf(a0, a1);
    } else {
        float a[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int j = 0; j < 64; ++j)
            if (j <= jl) a[j & 3] = fmaxf(a[j & 3], v[j]);
        mx = fmaxf(fmaxf(a[0], a[1]), fmaxf(a[2], a[3]));
    }
    xch[h * 128 + row] = mx;
    ptx::named_bar_sync(bar, 64);   // both halves' maxima written, both S halves read
    const float m = __fmul_rn(fmaxf(xch[row], xch[128 + row]), scale_log2);
    const float m_use = (jmax >= 0) ? m : 0.f;   // a row with no visible key: every p is 0
    if (!full) {
#pragma unroll
        for (int j = 0; j < 64; ++j)
            if (j > jl) v[j] = -INFINITY;
    }
    // The two quarter sums of this half (blocks 0, 1: quarter 2h; blocks 2, 3:
    // quarter 2h + 1) advance side by side, each in ascending key order, each
    // rounded p added straight from its bf16 half.
    const uint64_t c2 = pack2(scale_log2, scale_log2), nm2 = pack2(-m_use, -m_use);
    float lq[2] = {0.f, 0.f};
#pragma unroll
    for (int cp = 0; cp < 2; ++cp) {   // blocks cp (keys 64h + 16cp ..) and cp + 2
        const float* va = v + cp * 16;
        const float* vb = v + (cp + 2) * 16;
        uint32_t pa[8], pb[8];
#pragma unroll
        for (int t = 0; t < 16; t += 2) {
            float xa0, xa1, xb0, xb1;
            unpack2(fma2(pack2(va[t], va[t + 1]), c2, nm2), xa0, xa1);
            unpack2(fma2(pack2(vb[t], vb[t + 1]), c2, nm2), xb0, xb1);
            const __nv_bfloat162 ba = __floats2bfloat162_rn(ex2(xa0), ex2(xa1));
            const __nv_bfloat162 bb = __floats2bfloat162_rn(ex2(xb0), ex2(xb1));
            pa[t >> 1] = *reinterpret_cast<const uint32_t*>(&ba);
            pb[t >> 1] = *reinterpret_cast<const uint32_t*>(&bb);
            lq[0] = add_bf16_hi(pa[t >> 1], add_bf16_lo(pa[t >> 1], lq[0]));
            lq[1] = add_bf16_hi(pb[t >> 1], add_bf16_lo(pb[t >> 1], lq[1]));
        }
        tmem_st8(s_taddr + (h * 4 + cp) * 8, pa);
        tmem_st8(s_taddr + (h * 4 + cp + 2) * 8, pb);
    }
    if (h == 1) {
        xch[256 + row] = lq[0];
        xch[384 + row] = lq[1];
    }
    ptx::named_bar_sync(bar, 64);   // L2, L3 written; the maxima read
    if (h == 0) {
        const float l = __fadd_rn(__fadd_rn(__fadd_rn(lq[0], lq[1]), xch[256 + row]), xch[384 + row]);
        ptx::tmem_st2(s_taddr + PF_TM_ML, m, l);
    }
    ptx::tmem_wait_st();
    m_out = m;
}

// The tiles of a launch: tile L is KV group bg = L % n_bg (sequence bg / n_kv_heads,
// KV head bg % n_kv_heads) and query tile y = L / n_bg counted from the last, so
// lower L are longer (causal: later tokens see more chunks).  CTA c takes its
// tiles in rounds, c in round 0, then from the other end of the next round
// (G - 1 - c), and so on (snake order): every pair of rounds gives each CTA a long
// tile and a short one.
struct PfTile {
    int b, g, t0, t_last, kv_last, n_iter;
};
__device__ __forceinline__ int pf_tile_index(int j, int n_ctas) {
    const int c = (j & 1) ? (n_ctas - 1 - (int)blockIdx.x) : (int)blockIdx.x;
    return j * n_ctas + c;
}
__device__ __forceinline__ PfTile pf_tile(const TcArgs& a, int L, int base) {
    const int n_bg = a.batch * a.n_kv_heads;
    const int n_qt = (a.tokens + a.tq - 1) / a.tq;
    const int bg = L % n_bg, y = L / n_bg;
    PfTile t;
    t.g = bg % a.n_kv_heads;
    t.b = bg / a.n_kv_heads;
    t.t0 = (n_qt - 1 - y) * a.tq;
    t.t_last = min(t.t0 + a.tq, a.tokens) - 1;
    t.kv_last = base + t.t_last;
    t.n_iter = t.kv_last / kAttnChunk + 1;
    return t;
}

__global__ void __launch_bounds__(kPfThreads, 1)
    k_attn_pf(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
              const __grid_constant__ CUtensorMap mV, const TcArgs a) {
    TRACE(const unsigned long long tr0 = trace_stamp();)
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t* bars = (uint64_t*)(sm + PF_OFF_BAR);
    uint64_t* q_full = bars + 0;     // [2] TMA -> MMA (the Q tile of this CTA's tile j in buffer j % 2)
    uint64_t* q_empty = bars + 2;    // [2] MMA (after the tile's last S) -> TMA
    uint64_t* k_full = bars + 4;     // [2] TMA -> MMA
    uint64_t* k_empty = bars + 6;    // [2] MMA (after S) -> TMA
    uint64_t* v_full = bars + 8;     // [2] TMA -> MMA (and the softmax, before it zeroes rows)
    uint64_t* v_empty = bars + 10;   // [2] MMA (after PV) -> TMA
    uint64_t* s_full = bars + 12;    // [3] MMA (after S) -> softmax
    uint64_t* p_full = bars + 15;    // [3] softmax (P, m, l written) -> MMA, fold
    uint64_t* s_free = bars + 18;    // [3] fold (m, l read) -> MMA
    uint64_t* oc_full = bars + 21;   // MMA (after PV) -> fold
    uint64_t* oc_free = bars + 22;   // fold (O_c read) -> MMA
    uint32_t* tmem_holder = (uint32_t*)(bars + 23);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    ptx::griddep_wait();   // q and the cache rows come from the projection kernels
    TRACE(const unsigned long long tr1 = trace_stamp();)

    // Persistent: this CTA walks tiles j = 0, 1, ... (pf_tile_index) while in range.
    // Every ring and buffer below counts the chunks of all its tiles in one sequence
    // (gi), so a tile's first loads and S MMAs go out while the previous tile's last
    // chunks are still in the softmax and the fold.
    const int n_rep = a.n_heads / a.n_kv_heads;
    const int base = a.pos_dev ? *a.pos_dev : a.start_pos;
    if (base < 0 || base + a.tokens - 1 >= a.max_pos) {
        if (threadIdx.x == 0 && blockIdx.x == 0) record_error(a.err, LLAMA_ERR_POS_RANGE);
        return;
    }
    const int n_tiles = a.batch * a.n_kv_heads * ((a.tokens + a.tq - 1) / a.tq);
    const int G = gridDim.x;
    int* err = a.err;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(&q_full[i], 1);
            ptx::mbar_init(&q_empty[i], 1);
            ptx::mbar_init(&k_full[i], 1);
            ptx::mbar_init(&k_empty[i], 1);
            ptx::mbar_init(&v_full[i], 1);
            ptx::mbar_init(&v_empty[i], 1);
        }
        for (int i = 0; i < kPfSBufs; ++i) {
            ptx::mbar_init(&s_full[i], 1);
            ptx::mbar_init(&p_full[i], 8);
            ptx::mbar_init(&s_free[i], 4);
        }
        ptx::mbar_init(oc_full, 1);
        ptx::mbar_init(oc_free, 4);
        ptx::fence_mbar_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc(tmem_holder, 512);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    // dependents start only once this CTA holds its tensor memory (one that started
    // earlier on this SM could take the columns and then wait for this grid)
    if (threadIdx.x == 0) ptx::griddep_launch_dependents();

    if (warp < 4) {
        ptx::setmaxnreg_dec<kPfRegsCtrl>();
        if (warp == 0 || warp == 2) {
            // ------------------------------------------------------------------ TMA producers
            if (lane == 0) {
                const bool is_k = (warp == 0);
                const CUtensorMap* map = is_k ? &mK : &mV;
                uint64_t* full = is_k ? k_full : v_full;
                uint64_t* empty = is_k ? k_empty : v_empty;
                uint8_t* ring = sm + (is_k ? PF_OFF_K : PF_OFF_V);
                ptx::prefetch_tmap(map);
                if (is_k) ptx::prefetch_tmap(&mQ);
                int gi = 0, n_q = 0;   // chunks and Q tiles issued
                bool ok = true;
                for (int j = 0; ok; ++j) {
                    const int L = pf_tile_index(j, G);
                    if (L >= n_tiles) break;
                    const PfTile t = pf_tile(a, L, base);
                    if (is_k) {
                        // Q of tile j into buffer j % 2 once tile j - 2's S MMAs are done with it
                        const int qb = j & 1;
                        if (j >= 2 && !ptx::mbar_wait(&q_empty[qb], ((j >> 1) - 1) & 1, err)) { ok = false; break; }
                        ptx::mbar_arrive_expect_tx(&q_full[qb], 2 * kSub);
                        for (int half = 0; half < 2; ++half)
                            asm volatile(
                                "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                                " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(
                                    ptx::smem_u32(sm + PF_OFF_Q + qb * 2 * kSub + half * kSub)),
                                "l"(reinterpret_cast<uint64_t>(&mQ)), "r"(ptx::smem_u32(&q_full[qb])), "r"(half * 64),
                                "r"(t.g * n_rep), "r"(t.b * a.tokens + t.t0)
                                : "memory");
                        ++n_q;
                    }
                    const int head_row0 = (t.b * a.n_kv_heads + t.g) * a.kv_seq;
                    for (int i = 0; i < t.n_iter; ++i, ++gi) {
                        const int st = gi & 1;
                        if (gi >= 2 && !ptx::mbar_wait(&empty[st], ((gi >> 1) & 1) ^ 1, err)) { ok = false; break; }
                        uint8_t* dst = ring + st * 2 * kSub;
                        const int row = head_row0 + i * kAttnChunk;
                        ptx::mbar_arrive_expect_tx(&full[st], 2 * kSub);
                        ptx::tma_load_2d(dst, map, &full[st], 0, row);
                        ptx::tma_load_2d(dst + kSub, map, &full[st], 64, row);
                    }
                }
                // no copy may still be landing when the CTA exits (it has landed already
                // unless a wait above gave up)
                for (int j = max(0, n_q - 2); j < n_q; ++j) ptx::mbar_wait_drain(&q_full[j & 1], (j >> 1) & 1);
                for (int i = max(0, gi - 2); i < gi; ++i) ptx::mbar_wait_drain(&full[i & 1], (i >> 1) & 1);
            }
        } else if (warp == 1) {
            // ------------------------------------------------------------------ MMA issuer
            if (lane == 0) {
                int n_total = 0;   // chunks of all this CTA's tiles
                for (int j = 0;; ++j) {
                    const int L = pf_tile_index(j, G);
                    if (L >= n_tiles) break;
                    n_total += pf_tile(a, L, base).n_iter;
                }
                // S(gi) into S[gi % 3]: Q of its tile landed (at the tile's first chunk),
                // K(gi) landed, and the fold has read chunk gi - 3's (m, l) from that buffer
                // (PV(gi - 3), which read its P, was issued before and the MMAs run in issue
                // order).  After a tile's last S its Q buffer is released.
                int s_j = 0, s_i = 0, s_n = 0;   // tile and chunk of the next S
                if (n_total > 0) s_n = pf_tile(a, pf_tile_index(0, G), base).n_iter;
                auto issue_s = [&](int gi) -> bool {
                    const int k = gi & 1, sb = gi % kPfSBufs, qb = s_j & 1;
                    if (s_i == 0 && !ptx::mbar_wait(&q_full[qb], (s_j >> 1) & 1, err)) return false;
                    if (!ptx::mbar_wait(&k_full[k], (gi >> 1) & 1, err)) return false;
                    if (gi >= kPfSBufs && !ptx::mbar_wait(&s_free[sb], ((gi / kPfSBufs) & 1) ^ 1, err)) return false;
                    ptx::tc_fence_after();
                    const uint64_t q_desc = ptx::sw128_kmajor_desc(ptx::smem_u32(sm + PF_OFF_Q + qb * 2 * kSub));
                    const uint32_t k_addr = ptx::smem_u32(sm + PF_OFF_K + k * 2 * kSub);
                    umma8_ss<kSub / 16, kSub / 16, false>(tmem + PF_TM_S + sb * 128, q_desc,
                                                          ptx::sw128_kmajor_desc(k_addr), IDESC_S);
                    ptx::umma_commit(&s_full[sb]);
                    ptx::umma_commit(&k_empty[k]);
                    if (++s_i == s_n) {
                        ptx::umma_commit(&q_empty[qb]);
                        ++s_j;
                        s_i = 0;
                        const int L = pf_tile_index(s_j, G);
                        s_n = L < n_tiles ? pf_tile(a, L, base).n_iter : 0;
                    }
                    return true;
                };
                bool ok = true;
                for (int gi = 0; gi < kPfSBufs && gi < n_total && ok; ++gi) ok = issue_s(gi);
                for (int gi = 0; gi < n_total && ok; ++gi) {
                    const int k = gi & 1, sb = gi % kPfSBufs;
                    if (!ptx::mbar_wait(&p_full[sb], (gi / kPfSBufs) & 1, err)) break;
                    // O_c is overwritten once the fold has read chunk gi - 1's
                    if (gi >= 1 && !ptx::mbar_wait(oc_free, (gi - 1) & 1, err)) break;
                    if (!ptx::mbar_wait(&v_full[k], (gi >> 1) & 1, err)) break;
                    ptx::tc_fence_after();
                    const uint32_t v_addr = ptx::smem_u32(sm + PF_OFF_V + k * 2 * kSub);
                    // P of keys 16ks.. in TMEM columns 8ks.., V rows 16ks..
                    umma8_ts(tmem + PF_TM_OC, tmem + PF_TM_S + sb * 128, ptx::sw128_mnmajor_desc(v_addr, kSub), IDESC_PV);
                    ptx::umma_commit(oc_full);
                    ptx::umma_commit(&v_empty[k]);
                    if (gi + kPfSBufs < n_total) ok = issue_s(gi + kPfSBufs);
                }
            }
        }
    } else if (warp < 12) {
        // ------------------------------------------------------------------ softmax, two threads per row
        ptx::setmaxnreg_dec<kPfRegsSoftmax>();
        const int h = (warp - 4) >> 2;   // key half of this warpgroup
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
        const int t_local = row / n_rep;
        float* xch = reinterpret_cast<float*>(sm + PF_OFF_XCH);
        bool ok = true;
        int gi = 0;
        for (int j = 0;; ++j) {
            const int L = pf_tile_index(j, G);
            if (L >= n_tiles) break;
            const PfTile t = pf_tile(a, L, base);
            const bool valid = (t_local < a.tq) && (t.t0 + t_local < a.tokens);
            const int pos_r = base + t.t0 + t_local;
            for (int i = 0; i < t.n_iter; ++i, ++gi) {
                const int k = gi & 1, sb = gi % kPfSBufs;
                // s_full(gi) also means PV(gi - 3) -- issued before S(gi) -- is done with the P in S[sb]
                if (ok) ok = ptx::mbar_wait(&s_full[sb], (gi / kPfSBufs) & 1, err);
                ptx::tc_fence_after();
                const int jmax = valid ? min(kAttnChunk - 1, pos_r - i * kAttnChunk) : -1;
                float m;
                // both halves reach the two barriers inside on every chunk, whatever `ok` says
                softmax_half_tmem(tmem + lane_addr + PF_TM_S + sb * 128, h, row, jmax, a.scale_log2, xch, 1 + quarter,
                                  m);
                if (h == 0) {
                    // value rows past the last visible key of this tile are zeroed (they may hold
                    // anything, including NaN; P is 0 there and 0 * NaN would poison O), once
                    // the chunk's V has landed
                    if (i * kAttnChunk + kAttnChunk - 1 > t.kv_last && ok)
                        ok = ptx::mbar_wait(&v_full[k], (gi >> 1) & 1, err);
                    if (i * kAttnChunk + row > t.kv_last) {
                        uint8_t* vrow = sm + PF_OFF_V + k * 2 * kSub + row * 128;
#pragma unroll
                        for (int c16 = 0; c16 < 8; ++c16) {
                            *reinterpret_cast<uint4*>(vrow + c16 * 16) = make_uint4(0, 0, 0, 0);
                            *reinterpret_cast<uint4*>(vrow + kSub + c16 * 16) = make_uint4(0, 0, 0, 0);
                        }
                    }
                    ptx::fence_proxy_async_smem();
                }
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&p_full[sb]);
            }
        }
    } else {
        // ------------------------------------------------------------------ fold + output
        ptx::setmaxnreg_inc<kPfRegsFold>();
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
        const int t_local = row / n_rep, h_local = row - t_local * n_rep;
        float O[128];
        bool ok = true;
        int gi = 0;
        for (int j = 0;; ++j) {
            const int L = pf_tile_index(j, G);
            if (L >= n_tiles) break;
            const PfTile t = pf_tile(a, L, base);
            const bool valid = (t_local < a.tq) && (t.t0 + t_local < a.tokens);
            float M = -INFINITY, L_sum = 0.f;
            bool started = false;
#pragma unroll 1
            for (int i = 0; i < t.n_iter; ++i, ++gi) {
                const int sb = gi % kPfSBufs;
                if (ok) ok = ptx::mbar_wait(&p_full[sb], (gi / kPfSBufs) & 1, err);
                ptx::tc_fence_after();
                float ml[2];
                ptx::tmem_ld<2>(tmem + lane_addr + PF_TM_S + sb * 128 + PF_TM_ML, ml);
                ptx::tmem_wait_ld();
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&s_free[sb]);
                const float m = ml[0], l = ml[1];
                if (ok) ok = ptx::mbar_wait(oc_full, gi & 1, err);
                ptx::tc_fence_after();
                // Per row: skip a chunk with no visible key, start from the first one, fold the
                // rest (the combine kernel's formula).  The TMEM loads are issued by the whole
                // warp whatever each row does (they are warp-collective).
                const bool use = (m != -INFINITY);
                const bool fold = use && started;
                float alpha = 1.f, beta = 0.f;
                if (fold) {
                    const float Mn = fmaxf(M, m);
                    alpha = exp2f(__fsub_rn(M, Mn));
                    beta = exp2f(__fsub_rn(m, Mn));
                    L_sum = __fmaf_rn(L_sum, alpha, __fmul_rn(l, beta));
                    M = Mn;
                } else if (use) {
                    M = m;
                    L_sum = l;
                }
                const uint32_t oc_addr = tmem + lane_addr + PF_TM_OC;
#pragma unroll
                for (int cb = 0; cb < 4; ++cb) {
                    float oc[32];
                    ptx::tmem_ld<32>(oc_addr + cb * 32, oc);
                    ptx::tmem_wait_ld();
                    if (cb == 3) {   // O_c fully read: PV(gi + 1) may overwrite it
                        ptx::tc_fence_before();
                        __syncwarp();
                        if (lane == 0) ptx::mbar_arrive(oc_free);
                    }
                    if (fold) {   // o = fma(o, alpha, oc * beta), two columns per instruction
                        const uint64_t a2 = pack2(alpha, alpha), b2 = pack2(beta, beta);
#pragma unroll
                        for (int jj = 0; jj < 32; jj += 2) {
                            float& o0 = O[cb * 32 + jj];
                            float& o1 = O[cb * 32 + jj + 1];
                            unpack2(fma2(pack2(o0, o1), a2, mul2(pack2(oc[jj], oc[jj + 1]), b2)), o0, o1);
                        }
                    } else if (use) {
#pragma unroll
                        for (int jj = 0; jj < 32; ++jj) O[cb * 32 + jj] = oc[jj];
                    }
                }
                started = started || use;
            }
            // o = O * (1 / L), rounded to bf16, while the next tile's chunks run
            if (valid && ok && started) {
                const float inv_l = __frcp_rn(L_sum);
                bf16* dst = a.o + ((size_t)t.b * a.tokens + t.t0 + t_local) * a.n_heads * 128 +
                            (size_t)(t.g * n_rep + h_local) * 128;
#pragma unroll
                for (int c8 = 0; c8 < 16; ++c8) {
                    uint32_t packed[4];
#pragma unroll
                    for (int jj = 0; jj < 8; jj += 2) {
                        const __nv_bfloat162 v2 = __floats2bfloat162_rn(__fmul_rn(O[c8 * 8 + jj], inv_l),
                                                                        __fmul_rn(O[c8 * 8 + jj + 1], inv_l));
                        packed[jj >> 1] = *reinterpret_cast<const uint32_t*>(&v2);
                    }
                    *reinterpret_cast<uint4*>(dst + c8 * 8) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
                }
            }
        }
    }

    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 512);
    }
    TRACE(trace_cta(TR_ATTN_PF, tr0, tr1);)
}

// ----------------------------------------------------------------------------- decode
// One TMA copy of a whole 128-key chunk of K or V: the cache viewed as
// [2 halves of 64 columns][rows][64] (strides 128 B and 256 B), box [2][128][64],
// lands as the two 16 KB sub-tiles [half][row][64] the MMA reads.
// The cache is read once per step: evict-first, so that streaming it does not
// push out of L2 the small buffers the step's kernels hand to one another (the
// chunk partials, activations, segment results).  Measured 2.4 us faster per
// 8B batch-32 decode step than the default policy.
__device__ __forceinline__ void tma_load_chunk(void* dst, const CUtensorMap* map, uint64_t* bar, int row,
                                               uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(ptx::smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(ptx::smem_u32(bar)), "r"(0), "r"(row), "r"(0), "l"(policy)
        : "memory");
}

// Persistent decode attention for groups of n_rep <= 8 query heads.  The work
// units are (sequence, KV head, chunk); CTA i walks a contiguous range of them.
// Query and P tiles hold 8 rows; their descriptors use an 8-row-group stride of
// 0, so the MMA's 128 rows repeat rows 0..7: TMEM lane 8g + r holds row r for
// every g, and all 32 lanes of a warp's lane quarter see the 8 rows.  A softmax
// warp therefore works on (row r = lane % 8, key quarter g = lane / 8) straight
// from TMEM.  Three TMEM slots (S and then O_c of one unit share a slot's 128
// columns) and three softmax warps take units in turn; the MMA thread issues
// S of unit i before PV of unit i-1.  K and V stream through separate
// three-stage TMA rings: K is released as soon as S has read it, V after PV,
// which follows the unit's softmax.  (Four slots with a 2-stage K ring and a
// 4-stage V ring, in the same shared memory, measured no faster.)
// Warps: 0..2 = softmax + partial store of slots 0..2, 3 = K producer,
// 4 = TMEM owner + MMA issuer, 5 = V producer.
constexpr int kDecSlots = 3;
constexpr int kDecThreads = 32 * (kDecSlots + 3);
constexpr int kDecStagesK = 3;   // K is released as soon as S has read it
constexpr int kDecStagesV = 3;   // V is held until PV, after the softmax of its unit
constexpr int D_OFF_Q = 0;                              // [slot][half] 1 KB each
constexpr int D_OFF_P = 8192;                           // [slot][half] 1 KB each
constexpr int D_OFF_K = 16384;                          // [stage] K: 2 sub-tiles
constexpr int D_OFF_V = D_OFF_K + kDecStagesK * 2 * kSub;   // [stage] V: 2 sub-tiles
constexpr int D_OFF_BAR = D_OFF_V + kDecStagesV * 2 * kSub;
static_assert(kDecSlots * 2048 <= D_OFF_P && D_OFF_P + kDecSlots * 2048 <= D_OFF_K, "query / P tiles");
static_assert(kDecSlots * 128 <= 512, "TMEM columns");
constexpr int D_SMEM_BYTES = D_OFF_BAR + 256 + 1024;

__device__ __forceinline__ uint64_t sw128_kmajor_desc_rows8(uint32_t smem_addr) {
    return ptx::sw128_kmajor_desc(smem_addr) & ~(0x3FFFull << 32);   // stride byte offset 0
}

// Decode units: (sequence b, KV head g, chunk c), c fastest, then g, then b.  With
// one position for the whole batch every sequence has n_total chunks; with one
// position per sequence, sequence b has nt(b) = pos_b / 128 + 1 and `pre` (shared
// memory) holds the prefix sums pre[b] = nt(0) + ... + nt(b - 1).
struct DecUnit {
    int b, g, c;
    int nt, pos;   // the sequence's chunk count and position
};
struct DecMap {
    int n_kv, n_total, pos, batch;
    const int* pre;    // null: one position for the batch
    const int* spos;   // per-sequence positions (shared memory)
};
constexpr int kSeqPosMax = 1024;   // sequences per call with per-sequence positions
__device__ __forceinline__ DecUnit dec_unit(const DecMap& m, int u) {
    DecUnit d;
    if (m.pre == nullptr) {
        d.c = u % m.n_total;
        const int bg = u / m.n_total;
        d.g = bg % m.n_kv;
        d.b = bg / m.n_kv;
        d.nt = m.n_total;
        d.pos = m.pos;
        return d;
    }
    int lo = 0, hi = m.batch - 1;   // the last sequence whose units start at or before u
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (m.pre[mid] * m.n_kv <= u) lo = mid;
        else hi = mid - 1;
    }
    d.b = lo;
    d.nt = m.pre[lo + 1] - m.pre[lo];
    const int r = u - m.pre[lo] * m.n_kv;
    d.g = r / d.nt;
    d.c = r - d.g * d.nt;
    d.pos = m.spos[lo];
    return d;
}

// The 128 columns at taddr, each lane keeping the 32 of its key quarter q.
__device__ __forceinline__ void tmem_ld_quarter(uint32_t taddr, int q, float (&out)[32]) {
#pragma unroll
    for (int cb = 0; cb < 4; ++cb) {
        float v[32];
        ptx::tmem_ld<32>(taddr + cb * 32, v);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) out[j] = (cb == q) ? v[j] : out[j];
    }
}

__global__ void __launch_bounds__(kDecThreads, 1) k_attn_tc_dec(const __grid_constant__ CUtensorMap mK,
                                                                const __grid_constant__ CUtensorMap mV,
                                                                const TcArgs a) {
    TRACE(const unsigned long long tr0 = trace_stamp();)
    // trace builds: when the first producer's wait returned
    TRACE(__shared__ unsigned long long s_tr_release;)
    TRACE(if (threadIdx.x == 0) s_tr_release = 0;)
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t* bars = (uint64_t*)(sm + D_OFF_BAR);
    uint64_t* k_full = bars + 0;                         // [stages]
    uint64_t* k_empty = bars + kDecStagesK;              // [K stages] S of the unit done
    uint64_t* v_full = bars + 2 * kDecStagesK;           // [V stages]
    uint64_t* v_empty = v_full + kDecStagesV;            // [V stages] PV of the unit done
    uint64_t* slot_ready = v_empty + kDecStagesV;        // [slots] query tile filled, slot's O_c read
    uint64_t* s_full = slot_ready + kDecSlots;           // [slots]
    uint64_t* p_full = s_full + kDecSlots;               // [slots]
    uint64_t* o_full = p_full + kDecSlots;               // [slots]
    uint32_t* tmem_holder = (uint32_t*)(o_full + kDecSlots);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // The position comes from the host side (set before the step is launched), not
    // from the kernels this one overlaps; cache rows below it were written by
    // earlier steps.  Only q and the newest cache row need griddepcontrol.wait.
    const int n_rep = a.n_heads / a.n_kv_heads;
    __shared__ int s_pre[kSeqPosMax + 1], s_pos[kSeqPosMax];
    __shared__ int s_bad;
    DecMap dm{a.n_kv_heads, 0, 0, a.batch, nullptr, nullptr};
    int n_units;
    if (a.pos_seq) {
        // per-sequence positions: chunk counts and their prefix sums, one warp
        if (warp == 0) {
            int run = 0, bad = 0;
            for (int b0 = 0; b0 < a.batch; b0 += 32) {
                const int b = b0 + lane;
                const int p = b < a.batch ? a.pos_seq[b] : 0;
                const bool in = b < a.batch && p >= 0 && p < a.max_pos;
                if (b < a.batch && !in) bad = 1;
                int nt = in ? p / kAttnChunk + 1 : 0;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const int v = __shfl_up_sync(0xffffffffu, nt, off);
                    if (lane >= off) nt += v;
                }
                if (b < a.batch) {
                    s_pre[b + 1] = run + nt;
                    s_pos[b] = p;
                }
                run += __shfl_sync(0xffffffffu, nt, 31);
            }
            bad = __any_sync(0xffffffffu, bad);
            if (lane == 0) {
                s_pre[0] = 0;
                s_bad = bad;
            }
        }
        __syncthreads();
        if (s_bad) {
            if (threadIdx.x == 0 && blockIdx.x == 0) record_error(a.err, LLAMA_ERR_POS_RANGE);
            return;
        }
        dm.pre = s_pre;
        dm.spos = s_pos;
        n_units = s_pre[a.batch] * a.n_kv_heads;
    } else {
        const int pos = a.pos_dev ? *a.pos_dev : a.start_pos;
        if (pos < 0 || pos >= a.max_pos) {
            if (threadIdx.x == 0 && blockIdx.x == 0) record_error(a.err, LLAMA_ERR_POS_RANGE);
            return;
        }
        dm.pos = pos;
        dm.n_total = pos / kAttnChunk + 1;
        n_units = a.batch * a.n_kv_heads * dm.n_total;
    }
    const int u_begin = (int)(((long)n_units * blockIdx.x) / gridDim.x);
    const int u_end = (int)(((long)n_units * (blockIdx.x + 1)) / gridDim.x);
    const int n_iter = u_end - u_begin;
    if (n_iter <= 0) return;
    int* err = a.err;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kDecStagesK; ++i) {
            ptx::mbar_init(&k_full[i], 1);
            ptx::mbar_init(&k_empty[i], 1);
        }
        for (int i = 0; i < kDecStagesV; ++i) {
            ptx::mbar_init(&v_full[i], 1);
            ptx::mbar_init(&v_empty[i], 1);
        }
        for (int i = 0; i < kDecSlots; ++i) {
            ptx::mbar_init(&slot_ready[i], 1);
            ptx::mbar_init(&s_full[i], 1);
            ptx::mbar_init(&p_full[i], 1);
            ptx::mbar_init(&o_full[i], 1);
        }
        ptx::fence_mbar_init();
    }
    if (warp == kDecSlots + 1) {
        ptx::tmem_alloc(tmem_holder, 512);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp == kDecSlots || warp == kDecSlots + 2) {
        // ------------------------------------------------------------------ TMA producers (K, V)
        if (lane == 0) {
            const bool is_k = (warp == kDecSlots);
            const CUtensorMap* map = is_k ? &mK : &mV;
            uint64_t* full = is_k ? k_full : v_full;
            uint64_t* empty = is_k ? k_empty : v_empty;
            uint8_t* ring = sm + (is_k ? D_OFF_K : D_OFF_V);
            const int n_st = is_k ? kDecStagesK : kDecStagesV;
            ptx::prefetch_tmap(map);
            const uint64_t pol = ptx::policy_evict_first();
            bool waited = false;
            int issued = 0;
            for (int i = 0; i < n_iter; ++i, ++issued) {
                const int st = i % n_st;
                if (i >= n_st && !ptx::mbar_wait(&empty[st], ((i / n_st) - 1) & 1, err)) break;
                const DecUnit d = dec_unit(dm, u_begin + i);
                if (!waited && d.c == d.nt - 1) {   // this chunk holds the row the QKV step writes
                    ptx::griddep_wait();
                    TRACE(if (LLAMA_TRACE_ON && is_k) s_tr_release = trace_clock();)
                    waited = true;
                }
                const int row = (d.b * a.n_kv_heads + d.g) * a.kv_seq + d.c * kAttnChunk;
                uint8_t* dst = ring + st * 2 * kSub;
                ptx::mbar_arrive_expect_tx(&full[st], 2 * kSub);
                tma_load_chunk(dst, map, &full[st], row, pol);
            }
            // no copy may still be landing when the CTA exits (it has landed already
            // unless a wait above gave up)
            for (int i = max(0, issued - n_st); i < issued; ++i)
                ptx::mbar_wait_drain(&full[i % n_st], (i / n_st) & 1);
        }
    } else if (warp == kDecSlots + 1) {
        // ------------------------------------------------------------------ MMA issuer: S(i), then PV(i-1)
        if (lane == 0) {
            auto issue_pv = [&](int j) -> bool {
                const int slot = j % kDecSlots, st = j % kDecStagesV;
                if (!ptx::mbar_wait(&p_full[slot], (j / kDecSlots) & 1, err)) return false;
                ptx::tc_fence_after();
                const uint32_t p_addr = ptx::smem_u32(sm + D_OFF_P + slot * 2048);
                if (!ptx::mbar_wait(&v_full[st], (j / kDecStagesV) & 1, err)) return false;
                const uint32_t v_addr = ptx::smem_u32(sm + D_OFF_V + st * 2 * kSub);
                umma8_ss<1024 / 16, 0, true>(tmem + slot * 128, sw128_kmajor_desc_rows8(p_addr),
                                             ptx::sw128_mnmajor_desc(v_addr, kSub), IDESC_PV);
                ptx::umma_commit(&o_full[slot]);
                ptx::umma_commit(&v_empty[st]);
                return true;
            };
            bool ok = true;
            for (int i = 0; i < n_iter && ok; ++i) {
                const int slot = i % kDecSlots, st = i % kDecStagesK;
                if (!ptx::mbar_wait(&k_full[st], (i / kDecStagesK) & 1, err)) { ok = false; break; }
                if (!ptx::mbar_wait(&slot_ready[slot], (i / kDecSlots) & 1, err)) { ok = false; break; }
                ptx::tc_fence_after();
                const uint32_t q_addr = ptx::smem_u32(sm + D_OFF_Q + slot * 2048);
                const uint32_t k_addr = ptx::smem_u32(sm + D_OFF_K + st * 2 * kSub);
                umma8_ss<1024 / 16, kSub / 16, false>(tmem + slot * 128, sw128_kmajor_desc_rows8(q_addr),
                                                      ptx::sw128_kmajor_desc(k_addr), IDESC_S);
                ptx::umma_commit(&s_full[slot]);
                ptx::umma_commit(&k_empty[st]);
                if (i > 0) ok = issue_pv(i - 1);
            }
            if (ok) issue_pv(n_iter - 1);
        }
    } else {
        // ------------------------------------------------------------------ softmax + partial store
        const int slot = warp;
        const int r = lane & 7, q = lane >> 3;   // row, key quarter (output column quarter for O_c)
        const bool valid = r < n_rep;
        // this warp's lane quarter (every quarter holds the 8 rows), the slot's columns
        const uint32_t taddr = tmem + ((uint32_t)((warp & 3) * 32) << 16) + slot * 128;
        uint8_t* qs = sm + D_OFF_Q + slot * 2048;
        uint8_t* ps = sm + D_OFF_P + slot * 2048;
        ptx::griddep_wait();   // q comes from the QKV step
        if (threadIdx.x == 0) ptx::griddep_launch_dependents();
        int q_bg = -1;         // (sequence, KV head) whose query rows the slot's tile holds
        bool ok = true;
        // The slot's query tile for unit i: rows 0..n_rep-1 of (b, g), zero rows up to 8;
        // lane = row r x 16-byte column blocks 2q, 2q+1 of both halves.  fetch_q loads a
        // unit's rows into registers early (the loads' latency hides behind the wait
        // for PV); prepare writes them to the tile once the slot is free.
        uint4 qreg[4];
        int qreg_bg = -1;
        auto fetch_q = [&](int i) {
            const DecUnit d = dec_unit(dm, u_begin + i);
            const int bg = d.b * a.n_kv_heads + d.g;
            if (bg == q_bg || bg == qreg_bg) return;
#pragma unroll
            for (int half = 0; half < 2; ++half)
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    uint4 v = make_uint4(0, 0, 0, 0);
                    if (valid)
                        v = *reinterpret_cast<const uint4*>(a.q + (size_t)d.b * a.n_heads * 128 +
                                                            (size_t)(d.g * n_rep + r) * 128 + half * 64 +
                                                            (q * 2 + cc) * 8);
                    qreg[half * 2 + cc] = v;
                }
            qreg_bg = bg;
        };
        auto prepare = [&](int i) {
            const DecUnit d = dec_unit(dm, u_begin + i);
            const int bg = d.b * a.n_kv_heads + d.g;
            if (bg != q_bg) {
                fetch_q(i);
#pragma unroll
                for (int half = 0; half < 2; ++half)
#pragma unroll
                    for (int cc = 0; cc < 2; ++cc)
                        *reinterpret_cast<uint4*>(qs + half * 1024 + sw_off(r, q * 2 + cc)) = qreg[half * 2 + cc];
                q_bg = bg;
                ptx::fence_proxy_async_smem();
            }
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&slot_ready[slot]);
        };
        if (slot < n_iter) prepare(slot);
        for (int i = slot, k = 0; i < n_iter; i += kDecSlots, ++k) {
            const DecUnit d = dec_unit(dm, u_begin + i);
            const int st = i % kDecStagesV;   // the unit's V stage
            if (ok) ok = ptx::mbar_wait(&s_full[slot], k & 1, err);
            ptx::tc_fence_after();
            const int jmax = min(kAttnChunk - 1, d.pos - d.c * kAttnChunk);   // the same for every row
            float sv[32];
            tmem_ld_quarter(taddr, q, sv);
            float m = quarter_max_raw(sv, q * 32, jmax);
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
            m = __fmul_rn(m, a.scale_log2);
            uint32_t packed[16];
            float lq;
            softmax_quarter(sv, q * 32, jmax, a.scale_log2, m, packed, lq);
            store_p_quarter(ps, 1024, r, q, packed);
            const float l0 = __shfl_sync(0xffffffffu, lq, r), l1 = __shfl_sync(0xffffffffu, lq, r + 8);
            const float l2 = __shfl_sync(0xffffffffu, lq, r + 16), l3 = __shfl_sync(0xffffffffu, lq, r + 24);
            const float l = __fadd_rn(__fadd_rn(__fadd_rn(l0, l1), l2), l3);
            ptx::tc_fence_before();
            // value rows past the position hold anything (NaN included): zero them once
            // the chunk's V has landed
            if (d.c == d.nt - 1) {
                if (ok) ok = ptx::mbar_wait(&v_full[st], (i / kDecStagesV) & 1, err);
#pragma unroll
                for (int r4 = 0; r4 < 4; ++r4) {
                    const int vr = lane + 32 * r4;
                    if (d.c * kAttnChunk + vr > d.pos) {
                        uint8_t* vrow = sm + D_OFF_V + st * 2 * kSub + vr * 128;
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
            if (i + kDecSlots < n_iter) fetch_q(i + kDecSlots);
            if (ok) ok = ptx::mbar_wait(&o_full[slot], k & 1, err);
            ptx::tc_fence_after();
            float ov[32];
            tmem_ld_quarter(taddr, q, ov);   // row r, output columns 32q..32q+31
            ptx::tc_fence_before();
            // the slot is free again: prepare it for this warp's next unit before storing
            if (i + kDecSlots < n_iter) prepare(i + kDecSlots);
            if (valid) {
                float* dst =
                    a.partial + ((((size_t)d.b * a.n_kv_heads + d.g) * a.n_chunks + d.c) * n_rep + r) * kPartStride;
#pragma unroll
                for (int q4 = 0; q4 < 8; ++q4)
                    *reinterpret_cast<float4*>(dst + q * 32 + 4 * q4) =
                        make_float4(ov[4 * q4], ov[4 * q4 + 1], ov[4 * q4 + 2], ov[4 * q4 + 3]);
                if (q == 0) {
                    dst[128] = m;
                    dst[129] = l;
                }
            }
        }
    }
    __syncthreads();
    if (warp == kDecSlots + 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 512);
    }
    TRACE(trace_cta(TR_ATTN_DEC, tr0, s_tr_release);)
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::atomic<PFN_cuTensorMapEncodeTiled_v12000> fn{nullptr};
    PFN_cuTensorMapEncodeTiled_v12000 f = fn.load(std::memory_order_acquire);
    if (!f) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult qr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &qr) !=
                cudaSuccess ||
            qr != cudaDriverEntryPointSuccess)
            return nullptr;
        f = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        fn.store(f, std::memory_order_release);
    }
    return f;
}

// K or V cache [rows][128] bf16 as [2][rows][64] (see tma_load_chunk).
bool make_tmap_kv_chunk(CUtensorMap* map, const void* base, uint64_t rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {64, rows, 2};
    cuuint64_t strides[2] = {128 * 2, 64 * 2};
    cuuint32_t box[3] = {64, 128, 2};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_tmap_q3d(CUtensorMap* map, const void* q, int n_heads, int tokens, int n_rep, int tq) {
    auto fn = encode_fn();
    if (!fn) return false;
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
    k.pos_seq = a.pos_seq;
    k.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)a.head_dim));
    k.q = (const bf16*)a.q;
    k.o = (bf16*)a.o;
    k.partial = a.partial;
    k.n_chunks = a.n_chunks;
    k.err = a.err;
    return k;
}

}  // namespace

LLAMA_TRACE_UNIT(attn_tc)

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
    cudaError_t r = kernel_setup_once((const void*)k_attn_pf, [](const void* kern) {
        // the register split inside the kernel must fit the block's launch allocation
        cudaFuncAttributes fa;
        cudaError_t e = cudaFuncGetAttributes(&fa, kern);
        if (e != cudaSuccess) return e;
        if (fa.numRegs * kPfThreads < kPfRegsNeeded) return cudaErrorInvalidConfiguration;
        return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, PF_SMEM_BYTES);
    });
    if (r != cudaSuccess) return r;
    // persistent: one CTA per SM at most, each walking its tiles
    const long n_tiles = (long)a.n_kv_heads * a.batch * ((a.tokens + k.tq - 1) / k.tq);
    if (n_tiles > INT32_MAX) return cudaErrorInvalidValue;
    const dim3 grid((unsigned)std::min(n_tiles, (long)device_sm_count()));
    return launch_pdl(k_attn_pf, grid, dim3(kPfThreads), PF_SMEM_BYTES, s, mq, mk, mv, k);
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
        // one copy per 128-key chunk of K or V
        if (!make_tmap_kv_chunk(&mk, a.kc, cache_rows) || !make_tmap_kv_chunk(&mv, a.vc, cache_rows))
            return cudaErrorInvalidValue;
        // persistent: one CTA per SM (units assigned on the device from the position)
        const int n_sm = device_sm_count();
        const long max_units = (long)a.batch * a.n_kv_heads * a.n_chunks;
        cudaError_t r = kernel_setup_once((const void*)k_attn_tc_dec, [](const void* kern) {
            return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, D_SMEM_BYTES);
        });
        if (r != cudaSuccess) return r;
        dim3 grid((unsigned)std::min<long>(max_units, n_sm));
        r = launch_pdl(k_attn_tc_dec, grid, dim3(kDecThreads), D_SMEM_BYTES, s, mk, mv, k);
        if (r != cudaSuccess) return r;
        return launch_attention_combine(a, s);
    }
    if (chunks_per_cta <= 0) chunks_per_cta = 2;
    k.chunks_per_cta = chunks_per_cta;
    auto kern = k_attn_tc_wide;
    cudaError_t r = kernel_setup_once((const void*)kern, [](const void* kf) {
        return cudaFuncSetAttribute(kf, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    });
    if (r != cudaSuccess) return r;
    dim3 grid((a.n_chunks + chunks_per_cta - 1) / chunks_per_cta, a.n_kv_heads, a.batch);
    r = launch_pdl(kern, grid, dim3(kThreads), SMEM_BYTES, s, mk, mv, k);
    if (r != cudaSuccess) return r;
    return launch_attention_combine(a, s);
}

}  // namespace llama
