// Next-token sampling on the device: temperature, softmax over the vocabulary,
// top-k / top-p truncation, renormalisation and one draw per row from a
// caller-supplied uniform ("How Llama 3.1 Generates the Next Token": Temperature,
// Softmax, Top-k and top-p sampling).
//
// One cluster of kCl CTAs per row; CTA c owns the c-th contiguous slice of the
// row.  Token order is by decreasing logit, equal logits by increasing index (the
// greedy tie rule).  Each token's softmax weight e^{(z - max)/T} is evaluated in
// fp32 (the hardware 2^x, relative error below 2^-22) and held as a 2^-40
// fixed-point integer, so every sum of weights -- the normaliser, the mass of a
// set of tokens, the cumulative mass up to a token -- is an exact integer sum
// whatever order the threads and CTAs add in: the kept set and the drawn token do
// not depend on scheduling.
//
// "The first token (in order) at which the running count or mass reaches a
// target" (the top-k boundary, the top-p boundary, the drawn token) is found in
// three levels.  Level 0, computed once per row: a 256-bin histogram (token count
// and mass) over bins of one sixteenth of (max - z) / T, i.e. intervals of logits
// in decreasing order, the last bin holding everything more than 16 units below
// the maximum; each CTA histograms its slice (per warp, the tail bin in
// registers) and the cluster adds the slices' histograms through distributed
// shared memory.  A scan from the top gives the bin that holds the boundary and
// the count and mass above it.  Level 1: the CTAs send that bin's tokens to CTA 0,
// which histograms them over 256 sub-bins of 1/4096 of (max - z) / T (the same
// product scaled by 2^8, so a sub-bin is again an interval of logits) and scans
// to the sub-bin of the boundary.  Level 2: CTA 0 sorts that sub-bin's tokens by
// (logit down, index up) and scans them in order -- the boundary token, its rank
// and the mass through it are then exact.  A sub-bin too large to sort is handled
// by sorting the whole bin; a bin too large to gather, by an exact radix descent
// over the logits' order-preserving keys across the cluster, ties by rank in
// index order.
//
// Every cluster barrier is reached by every CTA the same number of times: each
// branch around one depends only on the arguments or on cluster-wide sums that
// every CTA computes alike.
#include "internal.h"

namespace llama {
namespace {

constexpr int kCl = 8;                           // CTAs per row
constexpr int kSampThreads = 512;
constexpr int kWarps = kSampThreads / 32;
constexpr int kBins = 256;
constexpr int kTailBin = kBins - 1;
constexpr float kBinsPerNat = 16.0f;             // level-0 bins per unit of (max - z) / T
constexpr float kMassScale = 1099511627776.0f;   // 2^40: fixed-point weight of the largest logit
constexpr int kListCap = 8192;                   // tokens of one level-0 bin gathered in CTA 0
constexpr int kSortCap = 2048;                   // tokens of one sub-bin sorted on their own

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
    unsigned long long sub[kSortCap];            // CTA 0: one sub-bin's tokens, sorted
    unsigned int loc_cnt[kBins];                 // this slice's level-0 histogram (read by the cluster)
    unsigned long long loc_mass[kBins];
    unsigned int rnd_cnt[kBins];                 // this slice's histogram of a radix round
    unsigned long long rnd_mass[kBins];
    unsigned int cnt0[kBins];                    // level 0 over the row (the same in every CTA)
    unsigned long long mass0[kBins];
    unsigned int cnt[kBins];                     // sub-bins (CTA 0) or a radix round, over the row
    unsigned long long mass[kBins];
    float red_v[kWarps];
    int red_i[kWarps];
    float cl_v[kCl];                             // slice maxima, written by every CTA of the cluster
    int cl_i[kCl];
    unsigned int cl_n[kCl];                      // slice counts of the boundary key (radix ties)
    unsigned int scan_c[kWarps];
    unsigned long long scan_m[kWarps];
    // a bin scan's result (scan_bins), and a boundary search's result (the same in every CTA)
    unsigned int above_c, tie_c, chosen, n_list, n_sub;
    unsigned long long above_m;
    unsigned int res_rank;
    unsigned long long res_mass;
    int res_found;
};
constexpr size_t kSampSmem = sizeof(SampSmem);

// ---------------------------------------------------------------- cluster helpers
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// Every thread of every CTA of the cluster; orders the shared-memory writes before
// it (local and remote) before every read after it.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t remote_addr(const void* local, uint32_t rank) {
    uint32_t a = (uint32_t)__cvta_generic_to_shared(local), r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
    return r;
}
__device__ __forceinline__ void st_remote_u32(const void* local, uint32_t rank, uint32_t v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(remote_addr(local, rank)), "r"(v) : "memory");
}
__device__ __forceinline__ void st_remote_u64(const void* local, uint32_t rank, unsigned long long v) {
    asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(remote_addr(local, rank)), "l"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_remote_u32(const void* local, uint32_t rank) {
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(remote_addr(local, rank)) : "memory");
    return v;
}
__device__ __forceinline__ unsigned long long ld_remote_u64(const void* local, uint32_t rank) {
    unsigned long long v;
    asm volatile("ld.shared::cluster.u64 %0, [%1];" : "=l"(v) : "r"(remote_addr(local, rank)) : "memory");
    return v;
}

// ---------------------------------------------------------------- the weights and the bins
// Order-preserving key: larger logit -> larger key (-0 counted as +0).
__device__ __forceinline__ uint32_t order_key(float z) {
    uint32_t b = z == 0.0f ? 0u : __float_as_uint(z);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_logit(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Per-row constants: the largest logit m, c = log2(e) / T for the weights, 16 / T
// for the level-0 bins and 4096 / T (= 2^8 * 16 / T exactly) for the sub-bins.
struct RowScale {
    float m, c, bin, sub;
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
// Sub-bin of a logit of level-0 bin b0: floor(4096 (m - z) / T) - 256 b0.  The
// product is the level-0 product times 2^8 exactly, so for b0 < 255 the result
// lies in 0..255; clamped, it stays monotone in z in the tail bin too.
__device__ __forceinline__ int sub_bin(float z, const RowScale& r, int b0) {
    const float x = fminf(__fmul_rn(__fsub_rn(r.m, z), r.sub), 16777216.0f);
    return min(max((int)x - 256 * b0, 0), kBins - 1);
}

// ceil or floor of a * b / 2^24 for a <= 2^24, b < 2^57 (the product needs 81 bits).
__device__ __forceinline__ unsigned long long mul_shift24(unsigned long long a, unsigned long long b, bool ceil_) {
    const unsigned long long lo = a * b, hi = __umul64hi(a, b);
    const unsigned long long q = (hi << 40) | (lo >> 24);
    return q + ((ceil_ && (lo & 0xffffffull)) ? 1ull : 0ull);
}

// f(i, z[i]) over the slice [lo, hi) of a row (i = lo + tid, lo + tid + blockDim, ...
// in increasing order per thread), eight loads in flight per thread.  lo is a
// multiple of 4, and so is hi when V is.
constexpr int kRowUnroll = 8;
template <typename F>
__device__ __forceinline__ void for_slice(const float* __restrict__ z, int V, int lo, int hi, F&& f) {
    const int step = blockDim.x;
    if ((V & 3) == 0 && ((uintptr_t)z & 15) == 0) {
        // 16-byte loads: thread t takes elements lo + 4t .. lo + 4t + 3, then 4 step further
        const float4* z4 = reinterpret_cast<const float4*>(z);
        const int e4 = hi >> 2;
        int i = (lo >> 2) + threadIdx.x;
        for (; i + (kRowUnroll - 1) * step < e4; i += kRowUnroll * step) {
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
        for (; i < e4; i += step) {
            const float4 v = __ldg(z4 + i);
            f(4 * i, v.x);
            f(4 * i + 1, v.y);
            f(4 * i + 2, v.z);
            f(4 * i + 3, v.w);
        }
        return;
    }
    int i = lo + threadIdx.x;
    for (; i + (kRowUnroll - 1) * step < hi; i += kRowUnroll * step) {
        float v[kRowUnroll];
#pragma unroll
        for (int u = 0; u < kRowUnroll; ++u) v[u] = __ldg(z + i + u * step);
#pragma unroll
        for (int u = 0; u < kRowUnroll; ++u) f(i + u * step, v[u]);
    }
    for (; i < hi; i += step) f(i, __ldg(z + i));
}

enum SelMode { SEL_COUNT_GE = 0, SEL_MASS_GE = 1, SEL_MASS_GT = 2 };

template <int MODE>
__device__ __forceinline__ bool reached(unsigned long long count, unsigned long long mass, unsigned long long target) {
    return MODE == SEL_COUNT_GE ? count >= target : MODE == SEL_MASS_GE ? mass >= target : mass > target;
}

// Warp 0: scan 256 bins in order (bin o when ASCENDING, where bin 0 holds the
// highest logits; bin 255 - o for key rounds, where the highest key is bin 255)
// from running totals (above_c0, above_m0) to the first non-empty bin at which the
// running count reaches `target` (SEL_COUNT_GE) or the running mass reaches it
// (SEL_MASS_GE) or exceeds it (SEL_MASS_GT).  Writes sm.chosen, sm.above_c,
// sm.above_m (totals before that bin) and sm.tie_c (its count).  An unreachable
// target takes the last non-empty bin.
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
    const bool hit = reached<MODE>((unsigned long long)above_c0 + c_inc, above_m0 + m_inc, target);
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
            if (reached<MODE>((unsigned long long)c_acc + c, m_acc + ms, target)) {
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

// The per-warp histograms summed into this CTA's (cnt, mass).
__device__ __forceinline__ void sum_warp_histograms(const SampSmem& sm, unsigned int* cnt, unsigned long long* mass) {
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

// The slice histograms of every CTA of the cluster (after a cluster barrier)
// added into this CTA's (cnt, mass): integer sums, the same in every CTA.
__device__ __forceinline__ void sum_cluster_histograms(const unsigned int* loc_cnt, const unsigned long long* loc_mass,
                                                       unsigned int* cnt, unsigned long long* mass) {
    for (int b = threadIdx.x; b < kBins; b += blockDim.x) {
        unsigned int c = 0;
        unsigned long long ms = 0;
#pragma unroll
        for (int r = 0; r < kCl; ++r) {
            c += ld_remote_u32(&loc_cnt[b], (uint32_t)r);
            ms += ld_remote_u64(&loc_mass[b], (uint32_t)r);
        }
        cnt[b] = c;
        mass[b] = ms;
    }
}

// Bitonic sort of list[0, n) in shared memory into descending order of the 64-bit
// entries (key << 32 | ~index: logit down, then index up); n <= the list's length,
// a power of two.  The whole CTA.
__device__ void sort_desc(unsigned long long* list, int n) {
    int n2 = 1;
    while (n2 < n) n2 <<= 1;
    for (int i = n + (int)threadIdx.x; i < n2; i += blockDim.x) list[i] = 0ull;   // sorts after every token
    __syncthreads();
    for (int k = 2; k <= n2; k <<= 1)
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int p = threadIdx.x; p < (n2 >> 1); p += blockDim.x) {   // pair p: (i, i + j), bit j of i clear
                const int i = ((p & ~(j - 1)) << 1) | (p & (j - 1));
                const int ixj = i | j;
                const unsigned long long a = list[i], b = list[ixj];
                const bool down = (i & k) == 0;   // descending overall
                if (down ? (a < b) : (a > b)) {
                    list[i] = b;
                    list[ixj] = a;
                }
            }
            __syncthreads();
        }
}

// Scan the sorted tokens list[0, n) in order, from the totals (above_c, above_m)
// of the tokens before them, to the first at which the running count or mass
// reaches the target; an unreachable target ends at the last token.  Writes
// sm.res_rank, sm.res_mass (the mass through that token) and sm.res_found.  The
// whole CTA.
template <int MODE>
__device__ void scan_sorted(const unsigned long long* list, int n, uint32_t above_c, unsigned long long above_m,
                            unsigned long long target, const RowScale& rs, SampSmem& sm) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int seg = (n + (int)blockDim.x - 1) / (int)blockDim.x;
    const int lo = min(n, tid * seg), hi = min(n, lo + seg);
    unsigned long long ms = 0;
    for (int i = lo; i < hi; ++i) ms += weight_of(key_logit((uint32_t)(list[i] >> 32)), rs);
    unsigned long long inc = ms;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const unsigned long long o = __shfl_up_sync(0xffffffffu, inc, off);
        if (lane >= off) inc += o;
    }
    if (lane == 31) sm.scan_m[warp] = inc;
    __syncthreads();
    if (tid == 0) {   // an unreachable target ends at the last token
        unsigned long long total = above_m;
        for (int w = 0; w < kWarps; ++w) total += sm.scan_m[w];
        sm.res_mass = total;
        sm.res_rank = above_c + (uint32_t)max(n - 1, 0);
        sm.res_found = n > 0 ? (int)~(uint32_t)(list[n - 1] & 0xffffffffull) : 0;
    }
    __syncthreads();
    unsigned long long run = above_m + inc - ms;
    for (int w = 0; w < warp; ++w) run += sm.scan_m[w];
    for (int i = lo; i < hi; ++i) {
        const unsigned long long e = list[i];
        const unsigned long long w = weight_of(key_logit((uint32_t)(e >> 32)), rs);
        const bool before = reached<MODE>((unsigned long long)above_c + (uint32_t)i, run, target);
        run += w;
        if (!before && reached<MODE>((unsigned long long)above_c + (uint32_t)i + 1, run, target)) {
            sm.res_rank = above_c + (uint32_t)i;   // exactly one token crosses the target
            sm.res_mass = run;
            sm.res_found = (int)~(uint32_t)(e & 0xffffffffull);
            break;
        }
    }
    __syncthreads();
}

// CTA 0: the boundary within the gathered level-0 bin b0 (list[0, n), with totals
// (above_c, above_m) of the tokens above it): level 1 over the sub-bins, level 2
// sorting one sub-bin.
template <int MODE>
__device__ void resolve_bin(int n, int b0, uint32_t above_c, unsigned long long above_m, unsigned long long target,
                            const RowScale& rs, SampSmem& sm) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int b = tid; b < kBins; b += blockDim.x) {
        sm.cnt[b] = 0;
        sm.mass[b] = 0;
    }
    if (tid == 0) sm.n_sub = 0;
    __syncthreads();
    for (int i = tid; i < n; i += blockDim.x) {
        const float z = key_logit((uint32_t)(sm.u.list[i] >> 32));
        const int s = sub_bin(z, rs, b0);
        atomicAdd(&sm.cnt[s], 1u);
        atomicAdd(&sm.mass[s], weight_of(z, rs));
    }
    __syncthreads();
    if (warp == 0) scan_bins<MODE, true>(sm.cnt, sm.mass, above_c, above_m, target, sm);
    __syncthreads();
    const int s0 = (int)sm.chosen;
    const uint32_t n_s = sm.cnt[s0];
    if (n_s > (uint32_t)kSortCap) {   // a crowded sub-bin: sort the whole bin
        sort_desc(sm.u.list, n);
        scan_sorted<MODE>(sm.u.list, n, above_c, above_m, target, rs, sm);
        return;
    }
    const uint32_t ac = sm.above_c;
    const unsigned long long am = sm.above_m;
    // the sub-bin's tokens, in any order (whole warps: every lane takes the same steps)
    for (int i0 = 0; i0 < n; i0 += blockDim.x) {
        const int i = i0 + tid;
        unsigned long long e = 0;
        bool in = false;
        if (i < n) {
            e = sm.u.list[i];
            in = sub_bin(key_logit((uint32_t)(e >> 32)), rs, b0) == s0;
        }
        const unsigned ballot = __ballot_sync(0xffffffffu, in);
        if (ballot) {
            unsigned int base = 0;
            if (lane == __ffs(ballot) - 1) base = atomicAdd(&sm.n_sub, (unsigned int)__popc(ballot));
            base = __shfl_sync(0xffffffffu, base, __ffs(ballot) - 1);
            if (in) sm.sub[base + __popc(ballot & ((1u << lane) - 1u))] = e;
        }
    }
    __syncthreads();
    sort_desc(sm.sub, (int)n_s);
    scan_sorted<MODE>(sm.sub, (int)n_s, ac, am, target, rs, sm);
}

// The boundary token of the row for one target: its rank (sm.res_rank), the mass
// of the tokens through it (sm.res_mass) and its index (sm.res_found), the same in
// every CTA of the cluster on return.  Every CTA calls it with the same arguments.
template <int MODE>
__device__ void find_boundary(const float* __restrict__ z, int V, int lo, int hi, const RowScale& rs,
                              unsigned long long target, uint32_t c, SampSmem& sm) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (warp == 0) scan_bins<MODE, true>(sm.cnt0, sm.mass0, 0u, 0ull, target, sm);
    if (tid == 0) sm.n_list = 0;
    __syncthreads();
    const int b0 = (int)sm.chosen;
    const uint32_t above_c = sm.above_c;
    const unsigned long long above_m = sm.above_m;
    const uint32_t n_bin = sm.cnt0[b0];   // over the row: the same in every CTA
    if (n_bin <= (uint32_t)kListCap) {
        // ---- this slice's tokens of bin b0 into the local list, then into CTA 0's
        auto append = [&](int i, float zi, bool valid) {
            const bool in = valid && level0_bin(zi, rs) == b0;
            const unsigned ballot = __ballot_sync(0xffffffffu, in);
            if (ballot) {
                unsigned int base = 0;
                if (lane == __ffs(ballot) - 1) base = atomicAdd(&sm.n_list, (unsigned int)__popc(ballot));
                base = __shfl_sync(0xffffffffu, base, __ffs(ballot) - 1);
                if (in)
                    sm.u.list[base + __popc(ballot & ((1u << lane) - 1u))] =
                        ((unsigned long long)order_key(zi) << 32) | (unsigned long long)(~(uint32_t)i);
            }
        };
        const int step = blockDim.x;
        if ((V & 3) == 0 && ((uintptr_t)z & 15) == 0) {
            const float4* z4 = reinterpret_cast<const float4*>(z);
            const int s4 = lo >> 2, e4 = hi >> 2;
            for (int i0 = s4; i0 < e4; i0 += kRowUnroll * step) {   // the same trip count in every warp
                float4 v[kRowUnroll];
#pragma unroll
                for (int u = 0; u < kRowUnroll; ++u) {
                    const int i = i0 + u * step + tid;
                    v[u] = i < e4 ? __ldg(z4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
                for (int u = 0; u < kRowUnroll; ++u) {
                    const int i = i0 + u * step + tid;
                    const bool valid = i < e4;
                    append(4 * i, v[u].x, valid);
                    append(4 * i + 1, v[u].y, valid);
                    append(4 * i + 2, v[u].z, valid);
                    append(4 * i + 3, v[u].w, valid);
                }
            }
        } else {
            for (int i0 = lo; i0 < hi; i0 += kRowUnroll * step) {   // the same trip count in every warp
                float v[kRowUnroll];
#pragma unroll
                for (int u = 0; u < kRowUnroll; ++u) {
                    const int i = i0 + u * step + tid;
                    v[u] = i < hi ? __ldg(z + i) : 0.f;
                }
#pragma unroll
                for (int u = 0; u < kRowUnroll; ++u) {
                    const int i = i0 + u * step + tid;
                    append(i, v[u], i < hi);
                }
            }
        }
        __syncthreads();
        if (c != 0) {
            // behind CTA 0's own tokens and those of the CTAs before this one
            uint32_t off = 0;
            for (uint32_t r = 0; r < c; ++r) off += ld_remote_u32(&sm.loc_cnt[b0], r);
            const int n_c = (int)sm.n_list;
            for (int i = tid; i < n_c; i += blockDim.x) st_remote_u64(&sm.u.list[off + i], 0u, sm.u.list[i]);
        }
        cluster_sync();   // CTA 0 holds the bin's n_bin tokens
        if (c == 0) {
            resolve_bin<MODE>((int)n_bin, b0, above_c, above_m, target, rs, sm);
            if (tid > 0 && tid < kCl) {
                st_remote_u32(&sm.res_rank, (uint32_t)tid, sm.res_rank);
                st_remote_u64(&sm.res_mass, (uint32_t)tid, sm.res_mass);
                st_remote_u32(&sm.res_found, (uint32_t)tid, (uint32_t)sm.res_found);
            }
        }
        cluster_sync();   // every CTA holds the result; CTA 0's list is free again
        return;
    }
    // ---- a bin too large to gather: radix descent over the keys of its tokens, by the cluster
    uint32_t prefix = 0;
    uint32_t ac = above_c;
    unsigned long long am = above_m;
    for (int r = 0; r < 4; ++r) {
        const int shift = 24 - 8 * r;
        zero_warp_histograms(sm);
        __syncthreads();
        for_slice(z, V, lo, hi, [&](int, float zi) {
            if (level0_bin(zi, rs) != b0) return;
            const uint32_t k = order_key(zi);
            if (r > 0 && ((k ^ prefix) >> (shift + 8)) != 0) return;
            add_to_warp_histogram(sm, warp, (k >> shift) & (kBins - 1), weight_of(zi, rs));
        });
        __syncthreads();
        sum_warp_histograms(sm, sm.rnd_cnt, sm.rnd_mass);
        cluster_sync();   // every slice's round histogram complete
        sum_cluster_histograms(sm.rnd_cnt, sm.rnd_mass, sm.cnt, sm.mass);
        __syncthreads();
        if (warp == 0) scan_bins<MODE, false>(sm.cnt, sm.mass, ac, am, target, sm);
        cluster_sync();   // every CTA has read the round histograms before the next round rewrites them
        prefix |= sm.chosen << shift;
        ac = sm.above_c;
        am = sm.above_m;
    }
    const unsigned long long wk = weight_of(key_logit(prefix), rs);
    const uint32_t tie = sm.tie_c;
    unsigned long long j;   // how many tokens of the tie group the target needs (1-based)
    if (MODE == SEL_COUNT_GE) j = target - ac;
    else if (MODE == SEL_MASS_GE) j = wk ? (target - am + wk - 1) / wk : 1;
    else j = wk ? (target - am) / wk + 1 : 1;
    if (j < 1) j = 1;
    if (j > tie) j = tie;
    // the j-th token (in index order) with the boundary key: the slices in CTA
    // order, within a slice contiguous runs per thread in thread order
    const int len = (hi - lo + (int)blockDim.x - 1) / (int)blockDim.x;
    const int tlo = min(hi, lo + tid * len), thi = min(hi, tlo + len);
    unsigned int cnt_t = 0;
    for (int i = tlo; i < thi; ++i) cnt_t += order_key(z[i]) == prefix;
    unsigned int inc = cnt_t;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const unsigned int o = __shfl_up_sync(0xffffffffu, inc, off);
        if (lane >= off) inc += o;
    }
    if (lane == 31) sm.scan_c[warp] = inc;
    __syncthreads();
    if (tid == 0) {
        unsigned int total = 0;
        for (int w = 0; w < kWarps; ++w) total += sm.scan_c[w];
        for (int q = 0; q < kCl; ++q) st_remote_u32(&sm.cl_n[c], (uint32_t)q, total);
        sm.res_rank = ac + (uint32_t)j - 1;
        sm.res_mass = am + j * wk;
        sm.res_found = 0;
    }
    cluster_sync();   // every slice's count of the boundary key
    unsigned int base = 0;
    for (uint32_t q = 0; q < c; ++q) base += sm.cl_n[q];
    for (int w = 0; w < warp; ++w) base += sm.scan_c[w];
    const unsigned int excl = base + inc - cnt_t;
    if (cnt_t > 0 && j > excl && j <= excl + cnt_t) {   // exactly one thread of the cluster
        unsigned int need = (unsigned int)(j - excl);
        for (int i = tlo; i < thi; ++i)
            if (order_key(z[i]) == prefix && --need == 0) {
                for (int q = 0; q < kCl; ++q) st_remote_u32(&sm.res_found, (uint32_t)q, (uint32_t)i);
                break;
            }
    }
    cluster_sync();   // every CTA holds the index
}

__global__ void __launch_bounds__(kSampThreads, 2) k_sample(const float* __restrict__ logits, int V, float t,
                                                            int top_k, unsigned int p_q24,
                                                            const float* __restrict__ uniforms,
                                                            int32_t* __restrict__ ids) {
    extern __shared__ __align__(16) uint8_t samp_smem_raw[];
    SampSmem& sm = *reinterpret_cast<SampSmem*>(samp_smem_raw);
    const uint32_t c = cluster_rank();
    const int row = blockIdx.x / kCl, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float* z = logits + (size_t)row * V;
    const int per = (V + 4 * kCl - 1) / (4 * kCl) * 4;   // slice length, a multiple of 4
    const int lo = min(V, (int)c * per), hi = min(V, lo + per);
    asm volatile("griddepcontrol.wait;" ::: "memory");

    // 1. the largest logit and its first index: per slice, then over the cluster
    float best = -INFINITY;
    int bi = INT32_MAX;
    for_slice(z, V, lo, hi, [&](int i, float v) {
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
        for (int q = 0; q < kCl; ++q) {
            st_remote_u32(&sm.cl_v[c], (uint32_t)q, __float_as_uint(best));
            st_remote_u32(&sm.cl_i[c], (uint32_t)q, (uint32_t)bi);
        }
    }
    cluster_sync();
    float m = sm.cl_v[0];
    int argmax = sm.cl_i[0];
    for (int q = 1; q < kCl; ++q)
        if (sm.cl_v[q] > m || (sm.cl_v[q] == m && sm.cl_i[q] < argmax)) { m = sm.cl_v[q]; argmax = sm.cl_i[q]; }
    if (argmax == INT32_MAX) argmax = 0;
    if (t == 0.0f || top_k == 1) {   // the greedy limit (the same branch in every CTA)
        if (c == 0 && tid == 0) ids[row] = argmax;
        return;
    }

    RowScale rs;
    rs.m = m;
    rs.c = __fdiv_rn(1.4426950408889634f, t);
    rs.bin = __fdiv_rn(kBinsPerNat, t);
    rs.sub = __fmul_rn(rs.bin, 256.0f);

    // 2. the level-0 histogram (per warp, the tail bin in registers), over the cluster, and Z
    zero_warp_histograms(sm);
    __syncthreads();
    unsigned int tail_c = 0;
    unsigned long long tail_m = 0;
    for_slice(z, V, lo, hi, [&](int, float zi) {
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
    sum_warp_histograms(sm, sm.loc_cnt, sm.loc_mass);
    cluster_sync();   // every slice's histogram complete
    sum_cluster_histograms(sm.loc_cnt, sm.loc_mass, sm.cnt0, sm.mass0);
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
        find_boundary<SEL_COUNT_GE>(z, V, lo, hi, rs, (unsigned long long)top_k, c, sm);
        n_k = (uint32_t)top_k;
        S_k = sm.res_mass;
    }
    // 4. top-p: the fewest first tokens whose mass reaches p of the total
    uint32_t n_p = (uint32_t)V;
    unsigned long long S_p = Z;
    if (p_q24 < (1u << 24)) {
        unsigned long long target = mul_shift24(p_q24, Z, true);
        if (target == 0) target = 1;
        find_boundary<SEL_MASS_GE>(z, V, lo, hi, rs, target, c, sm);
        n_p = sm.res_rank + 1;
        S_p = sm.res_mass;
    }
    const unsigned long long S = n_k <= n_p ? S_k : S_p;

    // 5. the draw: the first token whose cumulative mass exceeds u * S
    float u = uniforms[row];
    u = u > 0.0f ? u : 0.0f;
    unsigned long long u_q24 = (unsigned long long)(u * 16777216.0f);
    if (u_q24 > (1ull << 24) - 1) u_q24 = (1ull << 24) - 1;
    find_boundary<SEL_MASS_GT>(z, V, lo, hi, rs, mul_shift24(u_q24, S, false), c, sm);
    if (c == 0 && tid == 0) ids[row] = sm.res_found;
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
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)batch * kCl);
    cfg.blockDim = dim3(kSampThreads);
    cfg.dynamicSmemBytes = kSampSmem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = kCl;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, k_sample, logits, vocab, temperature, top_k, p_q24, uniforms, ids);
}

}  // namespace llama
