// noalloc.cu -- fp8_gemm for callers that must not allocate device memory.
//
// Some callers cannot hand the library a workspace: code that runs inside a
// memory pool's or allocator's own callback (allocating there re-enters the
// allocator), plugin hosts that give a library only its input and output
// buffers, and latency-critical paths where a device allocation, which may
// synchronise the device, is not allowed.  fp8bs_gemm_noalloc serves them by
// taking the split-K scratch of the small-M plan from a fixed array that
// lives in the library's own device image instead of from the caller.
//
// The array below is a host-side stand-in in host code: its address is only
// valid on the device.  The first call on each device looks up the real
// device address with cudaGetSymbolAddress (with that device current) and
// caches it; that first call should therefore happen before any stream
// capture.  Every call on a device shares the same array and leaves its
// partial sums there; calls whose kernels overlap on the GPU (two streams,
// or two threads) race on it and must be serialised by the caller.  Nothing
// in it needs clearing: each call's reduction reads only partial sums that
// the same call's GEMM kernel has just written.
#include <mutex>

#include "../../include/fp8bs.h"
#include "internal.h"

namespace {

// Split-K partial sums for fp8bs_gemm_noalloc.  Every device that loads the
// library holds this array until the process exits.
static __device__ __align__(256) unsigned char g_gemm_scratch[FP8BS_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_dev[kMaxDevices];  // device address of g_gemm_scratch, per device

fp8bs_status scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FP8BS_ERR_CUDA;
    std::lock_guard<std::mutex> g(g_mu);
    if (g_scratch_dev[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_gemm_scratch) != cudaSuccess || p == nullptr) return FP8BS_ERR_CUDA;
        g_scratch_dev[dev] = p;
    }
    *out = g_scratch_dev[dev];
    return FP8BS_OK;
}

}  // namespace

extern "C" fp8bs_status fp8bs_gemm_noalloc(const uint8_t* xq, const float* sx, int64_t lds, const uint8_t* wq,
                                           const float* sw, int64_t M, int64_t N, int64_t K, uint16_t* y,
                                           int64_t ldy, fp8bs_stream_t stream) {
    if (M < 0 || N < 0 || K < 0) return FP8BS_ERR_INVALID_ARG;
    // Scratch the fastest plan wants for this shape (0: no split, none used).
    const size_t need = fp8bs_gemm_workspace_size(M, N, K);
    if (need > FP8BS_NOALLOC_SCRATCH_BYTES) return FP8BS_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    if (need > 0) {
        if (fp8bs_status st = scratch_address(&scratch)) return st;
    }
    // Argument checks and the launch are those of fp8bs_gemm.
    return fp8bs_gemm(xq, sx, lds, wq, sw, M, N, K, y, ldy, scratch, need > 0 ? FP8BS_NOALLOC_SCRATCH_BYTES : 0,
                      stream);
}
