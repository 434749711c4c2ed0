// LM head + greedy choice for callers that cannot allocate device memory.
//
// llama_lmhead_argmax needs a caller-provided workspace for the normalised rows
// it feeds to the tensor cores.  Some callers have no way to provide one: code
// that runs where cudaMalloc is not allowed (inside a memory-pool-less runtime,
// a plugin handed only its input and output buffers) or that must not allocate
// on its hot path.  llama_lmhead_argmax_noalloc runs the same three kernels
// (final RMSNorm, weight-streaming LM-head projection, row argmax) with that
// scratch held in a file-scope device array instead.
#include <atomic>
#include <mutex>

#include "internal.h"

namespace llama {
namespace {

// Normalised rows of the no-alloc LM head: up to kNoAllocRows x kNoAllocDim bf16
// (512 KiB, held by every GPU that loads the library until the process exits).
constexpr int kNoAllocRows = 32;
constexpr int kNoAllocDim = 8192;
static __device__ __align__(256) __nv_bfloat16 g_lmhead_rows[kNoAllocRows * kNoAllocDim];
// Error word of the projection's bounded waits (cleared by every call, reported through ids).
static __device__ __align__(16) int g_lmhead_err;

constexpr int kMaxDevices = 64;
struct Scratch {
    void* rows;
    int* err;
};
std::atomic<void*> g_rows_addr[kMaxDevices];
std::atomic<int*> g_err_addr[kMaxDevices];
std::mutex g_setup;

// The arrays' device addresses on the current device.  The host-side symbols are
// stand-ins, not device addresses, so they are looked up once per device (with
// that device current) and cached.
cudaError_t scratch_address(Scratch* out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    void* p = g_rows_addr[dev].load(std::memory_order_acquire);
    int* q = g_err_addr[dev].load(std::memory_order_acquire);
    if (!p || !q) {
        std::lock_guard<std::mutex> lock(g_setup);
        p = g_rows_addr[dev].load(std::memory_order_relaxed);
        q = g_err_addr[dev].load(std::memory_order_relaxed);
        if (!p || !q) {
            e = cudaGetSymbolAddress(&p, g_lmhead_rows);
            if (e != cudaSuccess) return e;
            void* qv = nullptr;
            e = cudaGetSymbolAddress(&qv, g_lmhead_err);
            if (e != cudaSuccess) return e;
            q = (int*)qv;
            g_err_addr[dev].store(q, std::memory_order_release);
            g_rows_addr[dev].store(p, std::memory_order_release);
        }
    }
    out->rows = p;
    out->err = q;
    return cudaSuccess;
}

}  // namespace
}  // namespace llama

using namespace llama;

extern "C" int llama_lmhead_argmax_noalloc(const void* h, int batch, int h_stride, const void* g_final,
                                           const void* w_out, int vocab, int d_model, float eps, int32_t* ids,
                                           float* logits, void* stream) {
    if (batch < 0 || vocab <= 0 || d_model <= 0 || d_model % 128 || vocab % 128) return LLAMA_ERR_INVALID_ARG;
    if (batch == 0) return LLAMA_OK;
    if (!h || !g_final || !w_out || !ids || !logits || h_stride < d_model) return LLAMA_ERR_INVALID_ARG;
    if (batch > kNoAllocRows || d_model > kNoAllocDim) return LLAMA_ERR_WORKSPACE;   // beyond the static scratch
    Scratch sc{};
    if (scratch_address(&sc) != cudaSuccess) return LLAMA_ERR_CUDA;
    void* rows = sc.rows;
    cudaStream_t s = (cudaStream_t)stream;
    if (cudaMemsetAsync(sc.err, 0, sizeof(int), s) != cudaSuccess) return LLAMA_ERR_CUDA;
    if (h_stride == d_model) {
        if (launch_rmsnorm(h, g_final, rows, batch, d_model, eps, LLAMA_BF16, s) != cudaSuccess) return LLAMA_ERR_CUDA;
    } else {
        for (int r = 0; r < batch; ++r)
            if (launch_rmsnorm((const uint8_t*)h + (size_t)r * h_stride * 2, g_final,
                               (uint8_t*)rows + (size_t)r * d_model * 2, 1, d_model, eps, LLAMA_BF16, s) != cudaSuccess)
                return LLAMA_ERR_CUDA;
    }
    CUtensorMap mw;
    std::string why;
    if (!make_tmap_bf16(&mw, w_out, vocab, d_model, 128, &why)) return LLAMA_ERR_INVALID_ARG;
    GemmProblem p;
    p.M = batch;
    p.F = vocab;
    p.K = d_model;
    p.a_maps[0] = &mw;
    p.x = (const bf16*)rows;
    GemmEpi e;
    e.kind = EPI_LOGITS;
    e.out_f32 = logits;
    e.err = sc.err;
    if (launch_gemm_single_segment(p, e, s) != cudaSuccess) return LLAMA_ERR_CUDA;
    if (launch_argmax_rows(logits, batch, vocab, ids, sc.err, s) != cudaSuccess) return LLAMA_ERR_CUDA;
    return LLAMA_OK;
}
