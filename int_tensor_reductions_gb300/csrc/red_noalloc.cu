// red_noalloc.cu -- red_full_noalloc, the full reduction for callers that
// cannot allocate device memory (a device-synchronising cudaMalloc is not
// acceptable to them, or their own allocator owns the device's memory).
//
// The scratch that red_full keeps in its cudaMalloc'd workspace (one fp32
// partial per CTA and the last-block arrival counter) lives here in a fixed
// device array instead.  Host code must not pass the array's name to a
// kernel: on the host that name is only a stand-in for the symbol, not a
// device address (a kernel given it would fault, or on a GPU that can reach
// host memory silently use the wrong memory).  The device address is looked
// up once per device with cudaGetSymbolAddress, with that device current,
// and cached; a cudaDeviceReset unloads the module and makes the cached
// address stale, so the call must not be used on that device afterwards
// (red.h states this limit for the caller).
#include <mutex>

#include "red.h"
#include "red_internal.h"

namespace {

constexpr int64_t kMaxPartials = RED_NOALLOC_MAX_PARTIALS;
constexpr size_t kTickOffset = (size_t)kMaxPartials * sizeof(float);  // 256-byte aligned
constexpr size_t kScratchBytes = kTickOffset + 256;
constexpr int kMaxDevices = 64;

std::mutex g_mu;
unsigned char *g_addr[kMaxDevices];

}  // namespace

// Partials in bytes [0, kTickOffset), the arrival counter at kTickOffset.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

namespace {

// Device address of the scratch on the current device (looked up on the
// first call on that device).
int scratch_on(int dev, unsigned char **addr)
{
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_addr[dev]) {
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess)
            return red::cuda_fail(e, "red_full_noalloc: cudaGetSymbolAddress");
        if (!p)
            return red::fail(RED_ECUDA, "red_full_noalloc: cudaGetSymbolAddress gave NULL");
        g_addr[dev] = static_cast<unsigned char *>(p);
    }
    *addr = g_addr[dev];
    return RED_OK;
}

}  // namespace

extern "C" int red_full_noalloc(int op, const float *x, int64_t n, float *out, red_stream_t stream)
{
    if (op < RED_SUM || op > RED_MIN)
        return red::fail(RED_EINVAL, "red_full_noalloc: unknown op %d", op);
    if (n < 0 || n > (int64_t(1) << 44))
        return red::fail(RED_EINVAL, "red_full_noalloc: n = %lld out of range", (long long)n);
    if (!out || ((uintptr_t)out) % 4)
        return red::fail(RED_EINVAL, "red_full_noalloc: out is NULL or not 4-byte aligned");
    if (n > 0 && (!x || ((uintptr_t)x) % 4))
        return red::fail(RED_EINVAL, "red_full_noalloc: x is NULL or not 4-byte aligned");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (n == 0) {
        if (op != RED_SUM)
            return red::fail(RED_EINVAL, "red_full_noalloc: max/min of an empty vector");
        return red::cuda_fail(cudaMemsetAsync(out, 0, sizeof(float), s), "red_full_noalloc: cudaMemsetAsync");
    }
    red::DeviceInfo di;
    int st = red::device_info(&di);
    if (st != RED_OK)
        return st;
    if (di.dev >= kMaxDevices)
        return red::fail(RED_ECUDA, "red_full_noalloc: device ordinal %d out of range", di.dev);
    unsigned char *base = nullptr;
    st = scratch_on(di.dev, &base);
    if (st != RED_OK)
        return st;
    unsigned *tick = reinterpret_cast<unsigned *>(base + kTickOffset);
    // The array keeps the previous call's contents: the counter must start
    // at zero (the partials are always written before they are read).
    st = red::cuda_fail(cudaMemsetAsync(tick, 0, sizeof(unsigned), s), "red_full_noalloc: cudaMemsetAsync");
    if (st != RED_OK)
        return st;
    return red::launch_full_scratch(op, x, n, out, s, reinterpret_cast<float *>(base), tick, kMaxPartials);
}
