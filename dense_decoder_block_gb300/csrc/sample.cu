// Next-token sampling on the device: temperature, softmax over the vocabulary,
// top-k / top-p truncation, renormalisation and one draw per row from a
// caller-supplied uniform ("How Llama 3.1 Generates the Next Token": Temperature,
// Softmax, Top-k and top-p sampling).
//
// One CTA per row.  Token order is by decreasing logit, equal logits by
// increasing index (the greedy tie rule).  Each token's softmax weight
// e^{(z - max)/T} is evaluated in fp32 (the hardware 2^x, relative error below
// 2^-22) and held as a 2^-40 fixed-point integer,
// so every sum of weights -- the normaliser, the mass of a set of tokens, the
// cumulative mass up to a token -- is an exact integer sum whatever order the
// threads add in: the kept set and the drawn token do not depend on scheduling.
//
// "The first token (in order) at which the running count or mass reaches a
// target" (the top-k boundary, the top-p boundary, the drawn token) is found in
// two levels.  Level 0, computed once per row: a 256-bin histogram (token count
// and mass) over bins of one sixteenth of (max - z) / T, i.e. intervals of logits
// in decreasing order, the last bin holding everything more than 16 units below
// the maximum; it is kept per warp (the tail bin in registers) and then summed.
// A scan from the top gives the bin that holds the boundary and the count and
// mass above it.  Level 1: that bin's tokens are gathered into shared memory,
// sorted by (logit down, index up) with a bitonic sort, and scanned in order --
// the boundary token, its rank and the mass through it are then exact.  A bin
// too large for shared memory (many equal or nearly equal logits) is resolved by
// an exact radix descent over the logits' order-preserving keys within the bin
// instead, and ties by rank in index order.
#include "internal.h"

namespace llama {
namespace {

constexpr int kSampThreads = 1024;
constexpr int kWarps = kSampThreads / 32;
constexpr int kBins = 256;
constexpr int kTailBin = kBins - 1;
constexpr float kBinsPerNat = 16.0f;             // level-0 bins per unit of (max - z) / T
constexpr float kMassScale = 1099511627776.0f;   // 2^40: fixed-point weight of the largest logit
constexpr int kListCap = 16384;                  // tokens of one level-0 bin sorted in shared memory

struct SampSmem {
    union {
        struct {
            // histograms kept per warp; a bin's mass in three 32-bit parts of 14, 14 and 13
            // bits (native 32-bit shared atomics; a warp adds at most 2^15 weights of at
            // most 2^40, so no part overflows)
            unsigned int pc[kWarps][kBins];
            unsigned int pm[kWarps][kBins][3];
            unsigned long long tail_m[kWarps];   // the tail bin's mass, summed in registers
        } h;
        unsigned long long list[kListCap];       // one bin's tokens: key << 32 | (~index)
    } u;
    unsigned int cnt0[kBins];                    // level 0, summed
    unsigned long long mass0[kBins];
    unsigned int cnt[kBins];                     // key rounds of the large-bin path
    unsigned long long mass[kBins];
    float red_v[kWarps];
    int red_i[kWarps];
    unsigned int scan_c[kWarps];
    unsigned long long scan_m[kWarps];
    // search state, written by one thread or warp 0
    unsigned int prefix, above_c, tie_c, chosen, n_list, rank;
    unsigned long long above_m, mass_through;
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

// Per-row constants: the largest logit m, c = log2(e) / T for the weights and
// 16 / T for the level-0 bins.
struct RowScale {
    float m, c, bin;
};

// Softmax weight e^{(z - m)/T} = 2^{(z - m) c} of one logit as a 2^-40 fixed-point
// integer.  ex2.approx (relative error below 2^-22) on the special-function unit:
// the same value wherever it is evaluated, which is all the searches below need.
__device__ __forceinline__ unsigned long long weight_of(float z, const RowScale& r) {
    float e;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(__fmul_rn(__fsub_rn(z, r.m), r.c)));
    return __float2ull_rn(__fmul_rn(e, kMassScale));
}

// Level-0 bin of a logit: floor(16 (m - z) / T), at most 255 (monotone in z: a bin
// is an interval of logits, bin 0 the highest).
__device__ __forceinline__ int level0_bin(float z, const RowScale& r) {
    return (int)fminf(__fmul_rn(__fsub_rn(r.m, z), r.bin), (float)(kBins - 1));
}

// ceil or floor of a * b / 2^24 for a <= 2^24, b < 2^57 (the product needs 81 bits).
__device__ __forceinline__ unsigned long long mul_shift24(unsigned long long a, unsigned long long b, bool ceil_) {
    const unsigned long long lo = a * b, hi = __umul64hi(a, b);
    const unsigned long long q = (hi << 40) | (lo >> 24);
    return q + ((ceil_ && (lo & 0xffffffull)) ? 1ull : 0ull);
}

// f(i, z[i]) for this thread's share of the row (i = tid, tid + blockDim, ... in
// increasing order), eight loads in flight per thread: a pass over a row is
// otherwise bound by the latency of one load after another.
constexpr int kRowUnroll = 8;
template <typename F>
__device__ __forceinline__ void for_row(const float* __restrict__ z, int V, F&& f) {
    const int step = blockDim.x;
    if ((V & 3) == 0 && ((uintptr_t)z & 15) == 0) {
        // 16-byte loads: thread t takes elements 4t .. 4t + 3, then 4(t + step) ..
        const float4* z4 = reinterpret_cast<const float4*>(z);
        const int V4 = V >> 2;
        int i = threadIdx.x;
        for (; i + (kRowUnroll - 1) * step < V4; i += kRowUnroll * step) {
            float4 v[kRowUnroll];
#pragma unroll
            for (int u = 0; u < kRowUnroll; ++u) v[u] = __ldg(z4 + i + u * step);
#pragma unroll
            for (int u = 0; u < kRowUnroll; ++u) {
                const int e = 4 * (i + u * step);
                f(e, v[u].x);
                f(e + 1, v[u].y);
                f(e + 2, v[u].z);
                f(e + 3, v[u].w);
            }
        }
        for (; i < V4; i += step) {
            const float4 v = __ldg(z4 + i);
            f(4 * i, v.x);
            f(4 * i + 1, v.y);
            f(4 * i + 2, v.z);
            f(4 * i + 3, v.w);
        }
        return;
    }
    int i = threadIdx.x;
    for (; i + (kRowUnroll - 1) * step < V; i += kRowUnroll * step) {
        float v[kRowUnroll];
#pragma unroll
        for (int u = 0; u < kRowUnroll; ++u) v[u] = __ldg(z + i + u * step);
#pragma unroll
        for (int u = 0; u < kRowUnroll; ++u) f(i + u * step, v[u]);
    }
    for (; i < V; i += step) f(i, __ldg(z + i));
}

enum SelMode { SEL_COUNT_GE = 0, SEL_MASS_GE = 1, SEL_MASS_GT = 2 };

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

// Per-warp histograms of the threads' (bin, weight) pairs summed into cnt / mass.
__device__ __forceinline__ void sum_warp_histograms(SampSmem& sm, unsigned int* cnt, unsigned long long* mass) {
    for (int b = threadIdx.x; b < kBins; b += blockDim.x) {
        unsigned int c = 0;
        unsigned long long ms = 0;
        for (int w = 0; w < kWarps; ++w) {
            c += sm.u.h.pc[w][b];
            ms += (unsigned long long)sm.u.h.pm[w][b][0] + ((unsigned long long)sm.u.h.pm[w][b][1] << 14) +
                  ((unsigned long long)sm.u.h.pm[w][b][2] << 28);
            if (b == kTailBin) ms += sm.u.h.tail_m[w];
        }
        cnt[b] = c;
        mass[b] = ms;
    }
}

__device__ __forceinline__ void zero_warp_histograms(SampSmem& sm) {
    for (int i = threadIdx.x; i < kWarps * kBins; i += blockDim.x) {
        (&sm.u.h.pc[0][0])[i] = 0;
        (&sm.u.h.pm[0][0][0])[3 * i] = 0;
        (&sm.u.h.pm[0][0][0])[3 * i + 1] = 0;
        (&sm.u.h.pm[0][0][0])[3 * i + 2] = 0;
    }
    if (threadIdx.x < kWarps) sm.u.h.tail_m[threadIdx.x] = 0;
}

// One token into warp `w`'s histogram: its count and its weight's three parts.
__device__ __forceinline__ void add_to_warp_histogram(SampSmem& sm, int w, int bin, unsigned long long weight) {
    atomicAdd(&sm.u.h.pc[w][bin], 1u);
    atomicAdd(&sm.u.h.pm[w][bin][0], (unsigned int)(weight & 0x3fffull));
    atomicAdd(&sm.u.h.pm[w][bin][1], (unsigned int)((weight >> 14) & 0x3fffull));
    atomicAdd(&sm.u.h.pm[w][bin][2], (unsigned int)(weight >> 28));
}

template <int MODE>
__device__ __forceinline__ bool reached(uint32_t count, unsigned long long mass, unsigned long long target) {
    return MODE == SEL_COUNT_GE ? count >= target : MODE == SEL_MASS_GE ? mass >= target : mass > target;
}

// The boundary token: the first token in order at which the running count
// reaches `target` (SEL_COUNT_GE), or the running mass reaches it (SEL_MASS_GE) or
// exceeds it (SEL_MASS_GT).  Leaves in sm its 0-based rank (sm.rank), the mass of
// the tokens up to and including it (sm.mass_through) and its index (sm.found).
template <int MODE>
__device__ void find_boundary(const float* __restrict__ z, int V, const RowScale& rs, unsigned long long target,
                              SampSmem& sm) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (warp == 0) scan_bins<MODE, true>(sm.cnt0, sm.mass0, 0u, 0ull, target, sm);
    if (tid == 0) sm.n_list = 0;
    __syncthreads();
    const int b0 = (int)sm.chosen;
    const uint32_t above_c = sm.above_c;
    const unsigned long long above_m = sm.above_m;
    const uint32_t n_bin = sm.cnt0[b0];
    if (n_bin <= (uint32_t)kListCap) {
        // ---- level 1: gather the bin's tokens, sort them, scan in order
        // append one token (warp-collective: every lane calls it the same number of times)
        auto append = [&](int i, float zi, bool valid) {
            const bool in = valid && level0_bin(zi, rs) == b0;
            const unsigned ballot = __ballot_sync(0xffffffffu, in);
            if (ballot) {
                unsigned int base = 0;
                if (lane == __ffs(ballot) - 1) base = atomicAdd(&sm.n_list, (unsigned int)__popc(ballot));
                base = __shfl_sync(0xffffffffu, base, __ffs(ballot) - 1);
                if (in) {
                    const unsigned int at = base + __popc(ballot & ((1u << lane) - 1u));
                    sm.u.list[at] = ((unsigned long long)order_key(zi) << 32) | (unsigned long long)(~(uint32_t)i);
                }
            }
        };
        if ((V & 3) == 0 && ((uintptr_t)z & 15) == 0) {
            const float4* z4 = reinterpret_cast<const float4*>(z);
            const int V4 = V >> 2;
            for (int i0 = 0; i0 < V4; i0 += kRowUnroll * blockDim.x) {   // the same trip count in every warp
                float4 v[kRowUnroll];
#pragma unroll
                for (int u = 0; u < kRowUnroll; ++u) {
                    const int i = i0 + u * blockDim.x + tid;
                    v[u] = i < V4 ? __ldg(z4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
                for (int u = 0; u < kRowUnroll; ++u) {
                    const int i = i0 + u * blockDim.x + tid;
                    const bool valid = i < V4;
                    append(4 * i, v[u].x, valid);
                    append(4 * i + 1, v[u].y, valid);
                    append(4 * i + 2, v[u].z, valid);
                    append(4 * i + 3, v[u].w, valid);
                }
            }
        } else {
            for (int i0 = 0; i0 < V; i0 += kRowUnroll * blockDim.x) {   // the same trip count in every warp
                float v[kRowUnroll];
#pragma unroll
                for (int u = 0; u < kRowUnroll; ++u) {
                    const int i = i0 + u * blockDim.x + tid;
                    v[u] = i < V ? __ldg(z + i) : 0.f;
                }
#pragma unroll
                for (int u = 0; u < kRowUnroll; ++u) {
                    const int i = i0 + u * blockDim.x + tid;
                    append(i, v[u], i < V);
                }
            }
        }
        __syncthreads();
        const int n = (int)sm.n_list;
        int n2 = 1;
        while (n2 < n) n2 <<= 1;
        for (int i = n + tid; i < n2; i += blockDim.x) sm.u.list[i] = 0ull;   // sorts after every token
        __syncthreads();
        for (int k = 2; k <= n2; k <<= 1)
            for (int j = k >> 1; j > 0; j >>= 1) {
                for (int p = tid; p < (n2 >> 1); p += blockDim.x) {   // pair p: (i, i + j), bit j of i clear
                    const int i = ((p & ~(j - 1)) << 1) | (p & (j - 1));
                    const int ixj = i | j;
                    const unsigned long long a = sm.u.list[i], b = sm.u.list[ixj];
                    const bool down = (i & k) == 0;   // descending overall
                    if (down ? (a < b) : (a > b)) {
                        sm.u.list[i] = b;
                        sm.u.list[ixj] = a;
                    }
                }
                __syncthreads();
            }
        // running mass in order: contiguous segments per thread, block scan of the segment sums
        const int seg = (n + blockDim.x - 1) / blockDim.x;
        const int lo = min(n, tid * seg), hi = min(n, lo + seg);
        unsigned long long ms = 0;
        for (int i = lo; i < hi; ++i) ms += weight_of(key_logit((uint32_t)(sm.u.list[i] >> 32)), rs);
        unsigned long long inc = ms;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const unsigned long long o = __shfl_up_sync(0xffffffffu, inc, off);
            if (lane >= off) inc += o;
        }
        if (lane == 31) sm.scan_m[warp] = inc;
        if (tid == 0) {   // an unreachable target ends at the bin's last token
            sm.rank = above_c + (uint32_t)max(n - 1, 0);
            sm.found = n > 0 ? (int)~(uint32_t)(sm.u.list[n - 1] & 0xffffffffull) : 0;
        }
        __syncthreads();
        unsigned long long run = above_m + inc - ms;
        for (int w = 0; w < warp; ++w) run += sm.scan_m[w];
        if (tid == 0) {
            unsigned long long total = above_m;
            for (int w = 0; w < kWarps; ++w) total += sm.scan_m[w];
            sm.mass_through = total;
        }
        __syncthreads();
        for (int i = lo; i < hi; ++i) {
            const unsigned long long e = sm.u.list[i];
            const unsigned long long w = weight_of(key_logit((uint32_t)(e >> 32)), rs);
            const bool before = reached<MODE>(above_c + (uint32_t)i, run, target);
            run += w;
            if (!before && reached<MODE>(above_c + (uint32_t)i + 1, run, target)) {
                sm.rank = above_c + (uint32_t)i;
                sm.mass_through = run;
                sm.found = (int)~(uint32_t)(e & 0xffffffffull);
                break;
            }
        }
        __syncthreads();
        return;
    }
    // ---- a bin too large to sort: radix descent over the keys of the bin's tokens
    uint32_t prefix = 0;
    for (int r = 0; r < 4; ++r) {
        const int shift = 24 - 8 * r;
        zero_warp_histograms(sm);
        const uint32_t above_c0 = sm.above_c;
        const unsigned long long above_m0 = sm.above_m;
        __syncthreads();
        for_row(z, V, [&](int, float zi) {
            if (level0_bin(zi, rs) != b0) return;
            const uint32_t k = order_key(zi);
            if (r > 0 && ((k ^ prefix) >> (shift + 8)) != 0) return;
            const uint32_t bin = (k >> shift) & (kBins - 1);
            add_to_warp_histogram(sm, warp, bin, weight_of(zi, rs));
        });
        __syncthreads();
        sum_warp_histograms(sm, sm.cnt, sm.mass);
        __syncthreads();
        if (warp == 0) scan_bins<MODE, false>(sm.cnt, sm.mass, above_c0, above_m0, target, sm);
        __syncthreads();
        prefix |= sm.chosen << shift;
    }
    const unsigned long long wk = weight_of(key_logit(prefix), rs);
    const uint32_t ac = sm.above_c, tie = sm.tie_c;
    const unsigned long long am = sm.above_m;
    unsigned long long j;   // how many tokens of the tie group the target needs (1-based)
    if (MODE == SEL_COUNT_GE) j = target - ac;
    else if (MODE == SEL_MASS_GE) j = wk ? (target - am + wk - 1) / wk : 1;
    else j = wk ? (target - am) / wk + 1 : 1;
    if (j < 1) j = 1;
    if (j > tie) j = tie;
    // the j-th token (in index order) with the boundary key
    const int len = (V + blockDim.x - 1) / blockDim.x;
    const int lo = min(V, tid * len), hi = min(V, lo + len);
    unsigned int c = 0;
    for (int i = lo; i < hi; ++i) c += order_key(z[i]) == prefix;
    unsigned int inc = c;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const unsigned int o = __shfl_up_sync(0xffffffffu, inc, off);
        if (lane >= off) inc += o;
    }
    if (lane == 31) sm.scan_c[warp] = inc;
    if (tid == 0) {
        sm.rank = ac + (uint32_t)j - 1;
        sm.mass_through = am + j * wk;
        sm.found = 0;
    }
    __syncthreads();
    unsigned int base = 0;
    for (int w = 0; w < warp; ++w) base += sm.scan_c[w];
    const unsigned int excl = base + inc - c;
    if (c > 0 && j > excl && j <= excl + c) {
        unsigned int need = (unsigned int)(j - excl);
        for (int i = lo; i < hi; ++i)
            if (order_key(z[i]) == prefix && --need == 0) {
                sm.found = i;
                break;
            }
    }
    __syncthreads();
}

__global__ void __launch_bounds__(kSampThreads) k_sample(const float* __restrict__ logits, int V, float t,
                                                         int top_k, unsigned int p_q24,
                                                         const float* __restrict__ uniforms,
                                                         int32_t* __restrict__ ids) {
    extern __shared__ __align__(16) uint8_t samp_smem_raw[];
    SampSmem& sm = *reinterpret_cast<SampSmem*>(samp_smem_raw);
    const int row = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float* z = logits + (size_t)row * V;
    asm volatile("griddepcontrol.wait;" ::: "memory");

    // 1. the largest logit and its first index
    float best = -INFINITY;
    int bi = INT32_MAX;
    for_row(z, V, [&](int i, float v) {
        if (v > best) { best = v; bi = i; }   // increasing i: the first maximum stays
    });
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, best, off);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
        if (ov > best || (ov == best && oi < bi)) { best = ov; bi = oi; }
    }
    if (lane == 0) { sm.red_v[warp] = best; sm.red_i[warp] = bi; }
    __syncthreads();
    if (tid == 0) {
        for (int w = 1; w < kWarps; ++w)
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

    RowScale rs;
    rs.m = m;
    rs.c = __fdiv_rn(1.4426950408889634f, t);
    rs.bin = __fdiv_rn(kBinsPerNat, t);

    // 2. the level-0 histogram (per warp, the tail bin in registers) and the normaliser Z
    zero_warp_histograms(sm);
    __syncthreads();
    unsigned int tail_c = 0;
    unsigned long long tail_m = 0;
    for_row(z, V, [&](int, float zi) {
        const int b = level0_bin(zi, rs);
        const unsigned long long w = weight_of(zi, rs);
        if (b == kTailBin) {
            ++tail_c;
            tail_m += w;
        } else {
            add_to_warp_histogram(sm, warp, b, w);
        }
    });
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        tail_c += __shfl_xor_sync(0xffffffffu, tail_c, off);
        tail_m += __shfl_xor_sync(0xffffffffu, tail_m, off);
    }
    if (lane == 0) {
        sm.u.h.pc[warp][kTailBin] += tail_c;
        sm.u.h.tail_m[warp] = tail_m;
    }
    __syncthreads();
    sum_warp_histograms(sm, sm.cnt0, sm.mass0);
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
        find_boundary<SEL_COUNT_GE>(z, V, rs, (unsigned long long)top_k, sm);
        n_k = (uint32_t)top_k;
        S_k = sm.mass_through;
        __syncthreads();
    }
    // 4. top-p: the fewest first tokens whose mass reaches p of the total
    uint32_t n_p = (uint32_t)V;
    unsigned long long S_p = Z;
    if (p_q24 < (1u << 24)) {
        unsigned long long target = mul_shift24(p_q24, Z, true);
        if (target == 0) target = 1;
        find_boundary<SEL_MASS_GE>(z, V, rs, target, sm);
        n_p = sm.rank + 1;
        S_p = sm.mass_through;
        __syncthreads();
    }
    const unsigned long long S = n_k <= n_p ? S_k : S_p;

    // 5. the draw: the first token whose cumulative mass exceeds u * S
    float u = uniforms[row];
    u = u > 0.0f ? u : 0.0f;
    unsigned long long u_q24 = (unsigned long long)(u * 16777216.0f);
    if (u_q24 > (1ull << 24) - 1) u_q24 = (1ull << 24) - 1;
    find_boundary<SEL_MASS_GT>(z, V, rs, mul_shift24(u_q24, S, false), sm);
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
