// Host side of the tcgen05 projection kernel: TMA descriptors, schedule choice, launch.
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>
#include <set>
#include <utility>

#include "gemm_tc.cuh"

namespace llama {

namespace {
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}
}  // namespace

bool make_tmap_bf16(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                    std::string* why) {
    auto fn = encode_fn();
    if (!fn) {
        if (why) *why = "cuTensorMapEncodeTiled unavailable from the driver";
        return false;
    }
    if (((uintptr_t)base & 15) != 0 || (cols * 2) % 16 != 0) {
        if (why) *why = "TMA needs a 16-byte aligned base and rows that are a multiple of 16 bytes";
        return false;
    }
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        if (why) *why = "cuTensorMapEncodeTiled failed (code " + std::to_string((int)r) + ")";
        return false;
    }
    return true;
}

int pick_gemm_path(const GemmProblem& p, int path) {
    if (path == PATH_AUTO) return p.M <= 32 ? PATH_WEIGHT_STREAM : PATH_TOKEN_TILED;
    return path;
}

static int seg_kb_of(const GemmProblem& p) { return p.seg_kb > 0 ? p.seg_kb : kSegK / kBlockK; }
static int n_segments(const GemmProblem& p) {
    const int kb = p.K / kBlockK, s = seg_kb_of(p);
    return (kb + s - 1) / s;
}

int choose_seg_kb(int n_tiles, int total_kb, int n_sm) {
    // The fewest segments whose (tile, segment) units keep at least 70% of the SMs
    // streaming in a single wave: HBM is saturated well before every SM streams,
    // and each extra segment costs its fp32 partials and, from two segments on, a
    // reduction kernel (8B decode: the gate/up pair in one segment on 112 SMs and
    // the down projection in four on 128 took the step from 120.8 to 116.8 us; two
    // segments for QKV or three for O, 96 units each, were slower).
    for (int s = 1; s <= total_kb; ++s) {
        const int seg = (total_kb + s - 1) / s;
        const long units = (long)n_tiles * ((total_kb + seg - 1) / seg);
        if (units > n_sm) break;
        if (10 * units >= 7L * n_sm) return seg;
    }
    // Otherwise the segment length with the shortest schedule of equal units.
    int best = total_kb;
    long best_span = -1;
    for (int s = 1; s <= total_kb; ++s) {
        const int seg = (total_kb + s - 1) / s;
        if (seg < 8 && s > 1) break;
        const int segs = (total_kb + seg - 1) / seg;
        const long units = (long)n_tiles * segs;
        const long span = ((units + n_sm - 1) / n_sm) * seg;
        if (best_span < 0 || span < best_span) {
            best_span = span;
            best = seg;
        }
    }
    return best;
}

namespace {
constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];
std::mutex g_setup_lock;
std::set<std::pair<const void*, int>> g_setup_done;
}  // namespace

int device_sm_count() {
    int dev = 0, n = 0;
    cudaGetDevice(&dev);
    const bool cached = dev >= 0 && dev < kMaxDevices;
    if (cached && (n = g_sm_count[dev].load(std::memory_order_relaxed)) > 0) return n;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) return 148;
    if (cached) g_sm_count[dev].store(n, std::memory_order_relaxed);
    return n;
}

cudaError_t kernel_setup_once(const void* kern, cudaError_t (*setup)(const void* kern)) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(g_setup_lock);
    const auto key = std::make_pair(kern, dev);
    if (g_setup_done.count(key)) return cudaSuccess;
    e = setup(kern);
    if (e == cudaSuccess) g_setup_done.insert(key);
    return e;
}

cudaError_t setup_prefer_shared(const void* kern) {
    return cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
}

bool gemm_tt_split(const GemmProblem& p, int path) {
    // A token-tiled projection whose 256-token tiles would keep under 70% of the SMs
    // busy runs its K-segments on separate CTAs (split mode of gemm_tt.cuh) and
    // leaves them to the reduction kernels, as the weight-streaming schedule does --
    // when K is at least twice F, so that the MMA time saved outweighs writing and
    // reading the fp32 segment results (8B prefill at 512 tokens: the down projection
    // 72 -> 61 us with its reduction; QKV and O, K <= F, measured slower split).
    // An M = 128 MMA takes as long at N = 128 as at N = 256 (a microbenchmark of the
    // kernels' MMA shapes), so narrower token tiles would add tiles, not throughput.
    if (pick_gemm_path(p, path) != PATH_TOKEN_TILED || p.dual || n_segments(p) <= 1) return false;
    if (p.K < 2 * p.F) return false;
    const long tiles = (long)(p.F / kTileF) * ((p.M + 255) / 256);
    return 10 * tiles < 7L * device_sm_count();
}

size_t gemm_partial_bytes(const GemmProblem& p, int path) {
    const int segs = n_segments(p);
    if (gemm_tt_split(p, path)) return (size_t)segs * p.M * p.F * sizeof(float);
    if (pick_gemm_path(p, path) != PATH_WEIGHT_STREAM) return 0;
    if (segs <= 1) return 0;
    const int bn = p.M <= 16 ? 16 : 32;   // the weight-streaming tile width for this M
    return (size_t)segs * bn * (p.dual ? 2 : 1) * p.F * sizeof(float);
}

int gemm_num_segments(const GemmProblem& p) { return n_segments(p); }

bool gemm_needs_reduce(const GemmProblem& p, int path) {
    return (pick_gemm_path(p, path) == PATH_WEIGHT_STREAM && n_segments(p) > 1) || gemm_tt_split(p, path);
}

// Instantiated in gemm_token_tiled.cu / gemm_weight_stream.cu
cudaError_t launch_token_tiled(const GemmProblem& p, const GemmKArgs& ka, const CUtensorMap& a0,
                               const CUtensorMap& a1, const CUtensorMap& a2, const bf16* x, cudaStream_t s);
cudaError_t launch_weight_stream(const GemmProblem& p, const GemmKArgs& ka, const CUtensorMap& a0,
                                 const CUtensorMap& a1, const CUtensorMap& a2, const bf16* x, cudaStream_t s);

cudaError_t launch_gemm(const GemmProblem& p, const GemmEpi& e, int path, float* partial, cudaStream_t s) {
    if (p.M <= 0) return cudaSuccess;
    if (p.F % kTileF != 0 || p.K % kBlockK != 0) return cudaErrorInvalidValue;
    GemmKArgs ka{};
    ka.M = p.M;
    ka.F = p.F;
    ka.K = p.K;
    ka.seg_kb = seg_kb_of(p);
    ka.n_segs = n_segments(p);
    ka.e = e;
    ka.partial = partial;
    const CUtensorMap& a0 = *p.a_maps[0];
    const CUtensorMap& a1 = p.a_maps[1] ? *p.a_maps[1] : a0;
    const CUtensorMap& a2 = p.a_maps[2] ? *p.a_maps[2] : a0;
    if (e.kind == EPI_QKV) {
        ka.q_tiles = e.n_heads;
        ka.k_tiles = e.n_kv_heads;
    }
    const int chosen = pick_gemm_path(p, path);
    if (chosen == PATH_WEIGHT_STREAM) {
        if (p.M > 32) return cudaErrorInvalidValue;
        if (ka.n_segs > 1 && !partial) return cudaErrorInvalidValue;
        return launch_weight_stream(p, ka, a0, a1, a2, p.x, s);
    }
    ka.split = gemm_tt_split(p, path) ? 1 : 0;
    if (ka.split && !partial) return cudaErrorInvalidValue;
    return launch_token_tiled(p, ka, a0, a1, a2, p.x, s);
}

cudaError_t launch_gemm_single_segment(const GemmProblem& p, const GemmEpi& e, cudaStream_t s) {
    if (p.M <= 0) return cudaSuccess;
    if (p.F % kTileF != 0 || p.K % kBlockK != 0 || p.M > 32 || p.dual) return cudaErrorInvalidValue;
    GemmKArgs ka{};
    ka.M = p.M;
    ka.F = p.F;
    ka.K = p.K;
    ka.seg_kb = p.K / kBlockK;
    ka.n_segs = 1;
    ka.e = e;
    const CUtensorMap& a0 = *p.a_maps[0];
    return launch_weight_stream(p, ka, a0, a0, a0, p.x, s);
}

}  // namespace llama
