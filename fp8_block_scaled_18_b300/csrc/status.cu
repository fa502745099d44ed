// status.cu -- per-device facts and the device status word that kernels set
// when a bounded wait gives up.
#include <cstdlib>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace fp8bs {

// One word per device (every device that loads the library holds its own copy).
__device__ unsigned g_status_word;

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_lock;
bool g_ready[kMaxDevices];
DeviceInfo g_info[kMaxDevices];
}  // namespace

cudaError_t device_info(DeviceInfo* out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> g(g_lock);
    if (!g_ready[dev]) {
        DeviceInfo d{};
        d.device = dev;
        if ((e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return e;
        void* p = nullptr;
        if ((e = cudaGetSymbolAddress(&p, g_status_word)) != cudaSuccess) return e;
        d.err = static_cast<unsigned*>(p);
        g_info[dev] = d;
        g_ready[dev] = true;
    }
    *out = g_info[dev];
    return cudaSuccess;
}

uint64_t wait_timeout_ns() {
    static const uint64_t v = [] {
        const char* s = std::getenv("FP8BS_WAIT_TIMEOUT_NS");
        if (s && *s) {
            char* end = nullptr;
            unsigned long long t = std::strtoull(s, &end, 10);
            if (end != s && t > 0) return static_cast<uint64_t>(t);
        }
        return static_cast<uint64_t>(2000000000ull);  // 2 s: kernels here run for milliseconds at most
    }();
    return v;
}

}  // namespace fp8bs
