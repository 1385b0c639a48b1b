// red_internal.h -- host-side plumbing shared by the library's translation
// units: device facts, the per-device workspace, error reporting, knobs and
// the kernel launchers behind the C entry points.
#pragma once

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace red {

// Workspace held once per device: fp32/uint32 partials of the multi-CTA
// stages and the arrival counters of the last-block stages.
constexpr size_t WS_PART_BYTES = size_t(16) << 20;        // 16 MiB
constexpr size_t WS_PART_ELEMS = WS_PART_BYTES / 4;       // 4 Mi 32-bit words
constexpr int WS_TICKETS = 65536;

struct Workspace {
    void *part = nullptr;        // WS_PART_BYTES bytes
    unsigned *tick = nullptr;    // WS_TICKETS counters, zero between calls
};

struct DeviceInfo {
    int dev = 0;
    int sms = 0;
};

// Status helpers (codes of red.h).  fail() records a printf-style message
// for red_last_error() and returns `code`.
int fail(int code, const char *fmt, ...);
int cuda_fail(cudaError_t e, const char *where);

int device_info(DeviceInfo *info);
int get_workspace(Workspace *ws);

int knob(int which);        // 0 = automatic
void count_launches(int n); // adds n to red_launch_count()
int full_stage(int op);    // grid stage red_full uses for op (1, 2 or 3)

// Launchers: arguments have been validated by the entry points.
int launch_full(int op, const float *x, int64_t n, float *out, cudaStream_t s);
// Last-block full reduction with caller-provided scratch (max_parts partial
// slots and one counter that is zero on entry); allocates nothing.
int launch_full_scratch(int op, const float *x, int64_t n, float *out, cudaStream_t s, float *part,
                        unsigned *tick, int64_t max_parts);
int launch_rows_split(int op, const float *x, int64_t rows, int64_t len, int accum, float *out,
                      cudaStream_t s, const DeviceInfo &di);
int launch_full_stats(const float *x, int64_t n, float *out, cudaStream_t s);
int launch_rows_stats(const float *x, int64_t rows, int64_t len, float *out, cudaStream_t s);
int launch_rows_thread(int op, const float *x, int64_t rows, int len, int accum, float *out, cudaStream_t s);
int launch_rows(int op, const float *x, int64_t rows, int64_t len, int accum, float *out,
                cudaStream_t s);
int launch_ragged(int op, const float *x, const int64_t *off, int64_t rows, int64_t nnz, int accum,
                  float *out, cudaStream_t s);
int launch_typed(bool full, int op, int dtype, const void *x, int64_t rows, int64_t len, int accum, void *out,
                 cudaStream_t s);
// Ragged rows through shared-memory tiles (short rows).
int launch_ragged_staged(int op, const float *x, const int64_t *off, int64_t rows, int64_t nnz, int accum,
                         float *out, cudaStream_t s, int sms);
// Rows of 2..32 bytes (len * element size dividing 32) from a 32-byte aligned x.
int launch_typed_tiny(int op, int dtype, const void *x, int64_t rows, int len, int accum, void *out, cudaStream_t s,
                      int sms);
// Column reductions of the R x C region of a row-major matrix with row stride ld >= C.
int launch_cols(int op, int dtype, const void *x, int64_t R, int64_t C, int64_t ld, void *out, cudaStream_t s);


// Kernel launch on stream s with the programmatic-serialization attribute
// (the kernel's pdl_enter() waits for its predecessors before any global
// access, so the order of effects is that of a plain launch).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, cudaStream_t s, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Resident CTAs per SM of a kernel at `threads` threads and no dynamic shared
// memory; 0 if the query fails.
int occupancy(const void *kernel, int threads);

// occupancy() cached in `cache` (one per kernel instantiation) after the
// first successful query; concurrent first calls may both query, which is
// harmless, and a failed query is not cached.
inline int cached_occupancy(std::atomic<int> &cache, const void *kernel, int threads)
{
    int v = cache.load(std::memory_order_relaxed);
    if (v <= 0) {
        v = occupancy(kernel, threads);
        if (v > 0)
            cache.store(v, std::memory_order_relaxed);
    }
    return v;
}

}  // namespace red
