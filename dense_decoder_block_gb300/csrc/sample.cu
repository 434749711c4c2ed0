// Next-token sampling on the device: temperature, softmax over the vocabulary,
// top-k / top-p truncation, renormalisation and one draw per row from a
// caller-supplied uniform ("How Llama 3.1 Generates the Next Token": Temperature,
// Softmax, Top-k and top-p sampling).
//
// One CTA per row.  Token order is by decreasing logit, equal logits by
// increasing index (the greedy tie rule).  Each token's softmax weight
// e^{(z - max)/T} is evaluated in fp32 and held as a 2^-40 fixed-point integer,
// so every sum of weights -- the normaliser, the mass of a set of tokens, the
// cumulative mass up to a token -- is an exact integer sum whatever order the
// threads add in: the kept set and the drawn token do not depend on scheduling.
//
// The kept set and the draw are found without sorting.  "The first token (in
// order) at which the running count or mass reaches a target" is found in two
// levels.  Level 0, shared by every search of a row: a 256-bin histogram (token
// count and mass per bin) over bins of one eighth of (max - z) / T each, i.e.
// intervals of logits in decreasing order, kept per warp and then summed (the
// bins follow the distribution, so few threads add to the same bin at once).
// Scanning it from the top gives the bin that holds the boundary.  Then an exact
// radix descent over the logits' order-preserving 32-bit keys, restricted to that
// bin: four rounds, each a 256-bin histogram of the bin's tokens that share the
// key bits fixed so far, scanned from the highest key down.  The boundary key is
// then exact; the tokens equal to it (a tie group) share one weight, so how many
// of them the target needs is a division, and the drawn one is found by its rank
// among them in index order.
#include "internal.h"

namespace llama {
namespace {

constexpr int kSampThreads = 1024;
constexpr int kWarps = kSampThreads / 32;
constexpr int kBins = 256;
constexpr float kBinsPerNat = 8.0f;              // level-0 bins per unit of (max - z) / T
constexpr float kMassScale = 1099511627776.0f;   // 2^40: fixed-point weight of the largest logit

struct SampSmem {
    unsigned int pc[kWarps][kBins];              // level 0, per warp
    unsigned long long pm[kWarps][kBins];
    unsigned int cnt0[kBins];                    // level 0, summed
    unsigned long long mass0[kBins];
    unsigned int cnt[kBins];                     // key rounds
    unsigned long long mass[kBins];
    float red_v[kWarps];
    int red_i[kWarps];
    unsigned int scan[kWarps];
    // search state, written by warp 0
    unsigned int prefix, above_c, tie_c, chosen;
    unsigned long long above_m;
    int found;
};
constexpr size_t kSampSmem = sizeof(SampSmem);

// Order-preserving key: larger logit -> larger key (-0 counted as +0).
__device__ __forceinline__ uint32_t order_key(float z) {
    uint32_t b = z == 0.0f ? 0u : __float_as_uint(z);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_logit(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Softmax weight e^{(z - m)/T} of one logit as a 2^-40 fixed-point integer.
__device__ __forceinline__ unsigned long long weight_of(float z, float m, float t) {
    const float e = expf(__fdiv_rn(__fsub_rn(z, m), t));
    return __float2ull_rn(__fmul_rn(e, kMassScale));
}

// Level-0 bin of a logit: floor(8 (m - z) / T), at most 255 (monotone in z: a bin
// is an interval of logits, bin 0 the highest).
__device__ __forceinline__ int level0_bin(float z, float m, float t) {
    return (int)fminf(__fmul_rn(__fdiv_rn(__fsub_rn(m, z), t), kBinsPerNat), (float)(kBins - 1));
}

// ceil or floor of a * b / 2^24 for a <= 2^24, b < 2^57 (the product needs 81 bits).
__device__ __forceinline__ unsigned long long mul_shift24(unsigned long long a, unsigned long long b, bool ceil_) {
    const unsigned long long lo = a * b, hi = __umul64hi(a, b);
    const unsigned long long q = (hi << 40) | (lo >> 24);
    return q + ((ceil_ && (lo & 0xffffffull)) ? 1ull : 0ull);
}

enum SelMode { SEL_COUNT_GE = 0, SEL_MASS_GE = 1, SEL_MASS_GT = 2 };

struct Sel {
    uint32_t key;                // the boundary key
    uint32_t above_c;            // tokens with a larger key
    unsigned long long above_m;  // their mass
    uint32_t tie_c;              // tokens with exactly this key
};

// Warp 0: scan 256 bins in order (bin o for level 0, where bin 0 is the highest;
// bin 255 - o for key rounds, where the highest key is bin 255) from running
// totals (above_c0, above_m0) to the first non-empty bin at which the running
// count reaches `target` (SEL_COUNT_GE) or the running mass reaches it
// (SEL_MASS_GE) or exceeds it (SEL_MASS_GT).  Writes sm.chosen, sm.above_c,
// sm.above_m (totals before that bin) and sm.tie_c (its count).  The target must
// be reachable; otherwise the last non-empty bin is taken.
template <int MODE, bool ASCENDING>
__device__ void scan_bins(const unsigned int* cnt, const unsigned long long* mass, uint32_t above_c0,
                          unsigned long long above_m0, unsigned long long target, SampSmem& sm) {
    const int lane = threadIdx.x & 31;
    auto bin_at = [](int o) { return ASCENDING ? o : kBins - 1 - o; };
    uint32_t c_l = 0;
    unsigned long long m_l = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int b = bin_at(lane * 8 + j);
        c_l += cnt[b];
        m_l += mass[b];
    }
    uint32_t c_inc = c_l;
    unsigned long long m_inc = m_l;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const uint32_t c_o = __shfl_up_sync(0xffffffffu, c_inc, off);
        const unsigned long long m_o = __shfl_up_sync(0xffffffffu, m_inc, off);
        if (lane >= off) {
            c_inc += c_o;
            m_inc += m_o;
        }
    }
    const uint32_t c_run = above_c0 + c_inc;
    const unsigned long long m_run = above_m0 + m_inc;
    const bool hit = MODE == SEL_COUNT_GE ? c_run >= target : MODE == SEL_MASS_GE ? m_run >= target : m_run > target;
    const unsigned ballot = __ballot_sync(0xffffffffu, hit && c_l > 0);
    // the last lane that holds a non-empty bin, for an unreachable target
    const unsigned nonempty = __ballot_sync(0xffffffffu, c_l > 0);
    const int first = ballot ? __ffs(ballot) - 1 : (nonempty ? 31 - __clz(nonempty) : 0);
    if (lane == first) {
        uint32_t c_acc = above_c0 + c_inc - c_l;
        unsigned long long m_acc = above_m0 + m_inc - m_l;
        int chosen = -1, last = -1;
        uint32_t tie = 0, last_c = 0;
        unsigned long long last_m = 0;
        for (int j = 0; j < 8; ++j) {
            const int b = bin_at(lane * 8 + j);
            const uint32_t c = cnt[b];
            const unsigned long long ms = mass[b];
            if (c == 0) continue;
            const bool h = MODE == SEL_COUNT_GE ? c_acc + c >= target
                           : MODE == SEL_MASS_GE ? m_acc + ms >= target
                                                 : m_acc + ms > target;
            if (h) {
                chosen = b;
                tie = c;
                break;
            }
            last = b;
            last_c = c;
            last_m = ms;
            c_acc += c;
            m_acc += ms;
        }
        if (chosen < 0) {   // unreachable target: stop at the last non-empty bin
            chosen = last < 0 ? bin_at(lane * 8) : last;
            tie = last_c;
            c_acc -= last_c;
            m_acc -= last_m;
        }
        sm.chosen = (unsigned int)chosen;
        sm.above_c = c_acc;
        sm.above_m = m_acc;
        sm.tie_c = tie;
    }
}

// The first token in order at which the running count reaches `target`
// (SEL_COUNT_GE) or the running mass reaches it (SEL_MASS_GE) or exceeds it
// (SEL_MASS_GT): the level-0 bin from the row's level-0 histogram, then the exact
// key by a radix descent over that bin's tokens.
template <int MODE>
__device__ Sel select_boundary(const float* __restrict__ z, int V, float m, float t, unsigned long long target,
                               SampSmem& sm) {
    const int tid = threadIdx.x, warp = tid >> 5;
    if (warp == 0) scan_bins<MODE, true>(sm.cnt0, sm.mass0, 0u, 0ull, target, sm);
    __syncthreads();
    const int b0 = (int)sm.chosen;
    uint32_t prefix = 0;
    for (int r = 0; r < 4; ++r) {
        const int shift = 24 - 8 * r;
        for (int i = tid; i < kBins; i += blockDim.x) {
            sm.cnt[i] = 0;
            sm.mass[i] = 0;
        }
        const uint32_t above_c0 = sm.above_c;
        const unsigned long long above_m0 = sm.above_m;
        __syncthreads();
        for (int i = tid; i < V; i += blockDim.x) {
            const float zi = z[i];
            if (level0_bin(zi, m, t) != b0) continue;
            const uint32_t k = order_key(zi);
            if (r > 0 && ((k ^ prefix) >> (shift + 8)) != 0) continue;
            const uint32_t bin = (k >> shift) & (kBins - 1);
            atomicAdd(&sm.cnt[bin], 1u);
            atomicAdd(&sm.mass[bin], weight_of(zi, m, t));
        }
        __syncthreads();
        if (warp == 0) scan_bins<MODE, false>(sm.cnt, sm.mass, above_c0, above_m0, target, sm);
        __syncthreads();
        prefix |= sm.chosen << shift;
    }
    Sel s;
    s.key = prefix;
    s.above_c = sm.above_c;
    s.above_m = sm.above_m;
    s.tie_c = sm.tie_c;
    __syncthreads();   // sm is reused by the caller's next step
    return s;
}

__global__ void __launch_bounds__(kSampThreads) k_sample(const float* __restrict__ logits, int V, float t,
                                                         int top_k, unsigned int p_q24,
                                                         const float* __restrict__ uniforms,
                                                         int32_t* __restrict__ ids) {
    extern __shared__ __align__(16) uint8_t samp_smem_raw[];
    SampSmem& sm = *reinterpret_cast<SampSmem*>(samp_smem_raw);
    const int row = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n_warps = blockDim.x >> 5;
    const float* z = logits + (size_t)row * V;
    asm volatile("griddepcontrol.wait;" ::: "memory");

    // 1. the largest logit and its first index
    float best = -INFINITY;
    int bi = INT32_MAX;
    for (int i = tid; i < V; i += blockDim.x) {
        const float v = z[i];
        if (v > best) { best = v; bi = i; }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, best, off);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
        if (ov > best || (ov == best && oi < bi)) { best = ov; bi = oi; }
    }
    if (lane == 0) { sm.red_v[warp] = best; sm.red_i[warp] = bi; }
    __syncthreads();
    if (tid == 0) {
        for (int w = 1; w < n_warps; ++w)
            if (sm.red_v[w] > best || (sm.red_v[w] == best && sm.red_i[w] < bi)) { best = sm.red_v[w]; bi = sm.red_i[w]; }
        sm.red_v[0] = best;
        sm.red_i[0] = bi == INT32_MAX ? 0 : bi;
    }
    __syncthreads();
    const float m = sm.red_v[0];
    const int argmax = sm.red_i[0];
    if (t == 0.0f || top_k == 1) {   // the greedy limit
        if (tid == 0) ids[row] = argmax;
        return;
    }
    __syncthreads();

    // 2. the level-0 histogram (per warp, then summed) and the normaliser Z
    for (int i = tid; i < kWarps * kBins; i += blockDim.x) {
        (&sm.pc[0][0])[i] = 0;
        (&sm.pm[0][0])[i] = 0;
    }
    __syncthreads();
    for (int i = tid; i < V; i += blockDim.x) {
        const float zi = z[i];
        const int b = level0_bin(zi, m, t);
        atomicAdd(&sm.pc[warp][b], 1u);
        atomicAdd(&sm.pm[warp][b], weight_of(zi, m, t));
    }
    __syncthreads();
    for (int b = tid; b < kBins; b += blockDim.x) {
        unsigned int c = 0;
        unsigned long long ms = 0;
        for (int w = 0; w < kWarps; ++w) {
            c += sm.pc[w][b];
            ms += sm.pm[w][b];
        }
        sm.cnt0[b] = c;
        sm.mass0[b] = ms;
    }
    __syncthreads();
    unsigned long long Z = 0;   // every warp sums the 256 bins (8 per lane)
#pragma unroll
    for (int j = 0; j < 8; ++j) Z += sm.mass0[lane * 8 + j];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) Z += __shfl_xor_sync(0xffffffffu, Z, off);

    // 3. top-k: the mass of the k first tokens
    uint32_t n_k = (uint32_t)V;
    unsigned long long S_k = Z;
    if (top_k > 0 && top_k < V) {
        const Sel s = select_boundary<SEL_COUNT_GE>(z, V, m, t, (unsigned long long)top_k, sm);
        const unsigned long long w = weight_of(key_logit(s.key), m, t);
        n_k = (uint32_t)top_k;
        S_k = s.above_m + (unsigned long long)(top_k - s.above_c) * w;
    }
    // 4. top-p: the fewest first tokens whose mass reaches p of the total
    uint32_t n_p = (uint32_t)V;
    unsigned long long S_p = Z;
    if (p_q24 < (1u << 24)) {
        unsigned long long target = mul_shift24(p_q24, Z, true);
        if (target == 0) target = 1;
        const Sel s = select_boundary<SEL_MASS_GE>(z, V, m, t, target, sm);
        const unsigned long long w = weight_of(key_logit(s.key), m, t);
        unsigned long long j = w ? (target - s.above_m + w - 1) / w : 1;
        if (j < 1) j = 1;
        if (j > s.tie_c) j = s.tie_c;
        n_p = s.above_c + (uint32_t)j;
        S_p = s.above_m + j * w;
    }
    const unsigned long long S = n_k <= n_p ? S_k : S_p;

    // 5. the draw: the first token whose cumulative mass exceeds u * S
    float u = uniforms[row];
    u = u > 0.0f ? u : 0.0f;
    unsigned long long u_q24 = (unsigned long long)(u * 16777216.0f);
    if (u_q24 > (1ull << 24) - 1) u_q24 = (1ull << 24) - 1;
    const unsigned long long target = mul_shift24(u_q24, S, false);
    const Sel s = select_boundary<SEL_MASS_GT>(z, V, m, t, target, sm);
    const unsigned long long w = weight_of(key_logit(s.key), m, t);
    unsigned long long j = w ? (target - s.above_m) / w + 1 : 1;
    if (j > s.tie_c) j = s.tie_c;
    if (j < 1) j = 1;

    // 6. the j-th token (in index order) among those with the boundary key
    const int len = (V + blockDim.x - 1) / blockDim.x;
    const int lo = min(V, tid * len), hi = min(V, lo + len);
    unsigned int c = 0;
    for (int i = lo; i < hi; ++i) c += order_key(z[i]) == s.key;
    // exclusive scan of c over the block in thread order
    unsigned int inc = c;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const unsigned int o = __shfl_up_sync(0xffffffffu, inc, off);
        if (lane >= off) inc += o;
    }
    if (lane == 31) sm.scan[warp] = inc;
    if (tid == 0) sm.found = argmax;
    __syncthreads();
    unsigned int base = 0;
    for (int w2 = 0; w2 < warp; ++w2) base += sm.scan[w2];
    const unsigned int excl = base + inc - c;
    if (c > 0 && j > excl && j <= excl + c) {
        unsigned int need = (unsigned int)(j - excl);
        for (int i = lo; i < hi; ++i)
            if (order_key(z[i]) == s.key && --need == 0) {
                sm.found = i;
                break;
            }
    }
    __syncthreads();
    if (tid == 0) ids[row] = sm.found;
}

}  // namespace

cudaError_t launch_sample(const float* logits, int batch, int vocab, float temperature, int top_k, float top_p,
                          const float* uniforms, int32_t* ids, cudaStream_t s) {
    if (batch <= 0) return cudaSuccess;
    const double pq = (double)top_p * 16777216.0;
    const unsigned int p_q24 = top_p >= 1.0f ? (1u << 24) : (unsigned int)(pq + 0.5);
    cudaError_t e = kernel_setup_once((const void*)k_sample, [](const void* k) {
        return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSampSmem);
    });
    if (e != cudaSuccess) return e;
    return launch_pdl(k_sample, dim3(batch), dim3(kSampThreads), kSampSmem, s, logits, vocab, temperature, top_k,
                      p_q24, uniforms, ids);
}

}  // namespace llama
