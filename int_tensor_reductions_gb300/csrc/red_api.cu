// red_api.cu -- the extern "C" entry points of libred.so (declared and
// documented in red.h): host-side argument checks before any launch, the
// per-device workspace, error messages and tuning knobs.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <mutex>

#include "red.h"
#include "red_internal.h"

namespace red {
namespace {

constexpr int MAX_DEVICES = 64;
constexpr int64_t MAX_ELEMS = int64_t(1) << 44;  // guards index arithmetic

thread_local char g_err[512] = "";
std::mutex g_mu;
Workspace g_ws[MAX_DEVICES];
std::atomic<int> g_sms[MAX_DEVICES];

std::atomic<int> g_full_mode{RED_MODE_AUTO};
std::atomic<uint64_t> g_launches{0};
std::atomic<int> g_knobs[16];


bool misaligned(const void *p, uintptr_t a) { return ((uintptr_t)p) % a != 0; }

}  // namespace

int fail(int code, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return code;
}

int cuda_fail(cudaError_t e, const char *where)
{
    if (e == cudaSuccess)
        return RED_OK;
    return fail(RED_ECUDA, "%s: %s (%s)", where, cudaGetErrorName(e), cudaGetErrorString(e));
}

int device_info(DeviceInfo *info)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= MAX_DEVICES)
        return fail(RED_ECUDA, "device ordinal %d out of range", dev);
    int sms = g_sms[dev].load(std::memory_order_relaxed);
    if (sms == 0) {
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaDeviceGetAttribute");
        g_sms[dev].store(sms, std::memory_order_relaxed);
    }
    info->dev = dev;
    info->sms = sms;
    return RED_OK;
}

int get_workspace(Workspace *ws)
{
    DeviceInfo di;
    int st = device_info(&di);
    if (st != RED_OK)
        return st;
    std::lock_guard<std::mutex> lock(g_mu);
    Workspace &w = g_ws[di.dev];
    if (!w.part) {
        void *part = nullptr, *tick = nullptr;
        cudaError_t e = cudaMalloc(&part, WS_PART_BYTES);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return fail(RED_ENOMEM, "workspace allocation: %s", cudaGetErrorString(e));
        }
        e = cudaMalloc(&tick, WS_TICKETS * sizeof(unsigned));
        if (e != cudaSuccess) {
            cudaGetLastError();
            cudaFree(part);
            return fail(RED_ENOMEM, "workspace allocation: %s", cudaGetErrorString(e));
        }
        e = cudaMemset(tick, 0, WS_TICKETS * sizeof(unsigned));
        if (e == cudaSuccess)
            e = cudaDeviceSynchronize();
        if (e != cudaSuccess) {
            cudaFree(part);
            cudaFree(tick);
            return cuda_fail(e, "workspace initialisation");
        }
        w.part = part;
        w.tick = static_cast<unsigned *>(tick);
    }
    *ws = w;
    return RED_OK;
}

int knob(int which)
{
    if (which <= 0 || which >= 16)
        return 0;
    return g_knobs[which].load(std::memory_order_relaxed);
}

void count_launches(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

int full_stage(int op)
{
    // Automatic choice, by measurement (the three stages tie on inputs far
    // larger than L2; on small ones a second launch, overlapped by
    // programmatic dependent launch, costs less than the last-block fence
    // and partials read, and one atomic per CTA less than either): sums take
    // the two-pass stage, which is deterministic; max / min the atomic stage,
    // exact in any order.
    const int m = g_full_mode.load(std::memory_order_relaxed);
    if (m != RED_MODE_AUTO)
        return m;
    return op == RED_SUM ? RED_MODE_TWO_PASS : RED_MODE_ATOMIC;
}

int occupancy(const void *kernel, int threads)
{
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, 0) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

}  // namespace red

using namespace red;

extern "C" {

int red_full(int op, const float *x, int64_t n, float *out, red_stream_t stream)
{
    if (op < RED_SUM || op > RED_MIN)
        return fail(RED_EINVAL, "red_full: unknown op %d", op);
    if (n < 0 || n > MAX_ELEMS)
        return fail(RED_EINVAL, "red_full: n = %lld out of range", (long long)n);
    if (!out || misaligned(out, 4))
        return fail(RED_EINVAL, "red_full: out is NULL or not 4-byte aligned");
    if (n > 0 && (!x || misaligned(x, 4)))
        return fail(RED_EINVAL, "red_full: x is NULL or not 4-byte aligned");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (n == 0) {
        if (op != RED_SUM)
            return fail(RED_EINVAL, "red_full: max/min of an empty vector");
        return cuda_fail(cudaMemsetAsync(out, 0, sizeof(float), s), "red_full: cudaMemsetAsync");
    }
    return launch_full(op, x, n, out, s);
}

int red_full_stats(const float *x, int64_t n, float *out, red_stream_t stream)
{
    if (n <= 0 || n > MAX_ELEMS)
        return fail(RED_EINVAL, "red_full_stats: n = %lld out of range (max/min need n >= 1)", (long long)n);
    if (!out || misaligned(out, 4))
        return fail(RED_EINVAL, "red_full_stats: out is NULL or not 4-byte aligned");
    if (!x || misaligned(x, 4))
        return fail(RED_EINVAL, "red_full_stats: x is NULL or not 4-byte aligned");
    return launch_full_stats(x, n, out, reinterpret_cast<cudaStream_t>(stream));
}

int red_rows_stats(const float *x, int64_t rows, int64_t len, float *out, red_stream_t stream)
{
    if (rows < 0 || len < 0 || rows > MAX_ELEMS || len > MAX_ELEMS || (len > 0 && rows > MAX_ELEMS / len))
        return fail(RED_EINVAL, "red_rows_stats: rows = %lld, len = %lld out of range", (long long)rows,
                    (long long)len);
    if (rows == 0)
        return RED_OK;
    if (len == 0)
        return fail(RED_EINVAL, "red_rows_stats: empty rows have no max or min");
    if (!out || misaligned(out, 16))
        return fail(RED_EINVAL, "red_rows_stats: out is NULL or not 16-byte aligned");
    if (!x || misaligned(x, 4))
        return fail(RED_EINVAL, "red_rows_stats: x is NULL or not 4-byte aligned");
    return launch_rows_stats(x, rows, len, out, reinterpret_cast<cudaStream_t>(stream));
}

int red_rows(int op, const float *x, int64_t rows, int64_t len, int accum, float *out, red_stream_t stream)
{
    if (op < RED_SUM || op > RED_MIN)
        return fail(RED_EINVAL, "red_rows: unknown op %d", op);
    if (rows < 0 || len < 0 || rows > MAX_ELEMS || len > MAX_ELEMS ||
        (len > 0 && rows > MAX_ELEMS / len))
        return fail(RED_EINVAL, "red_rows: rows = %lld, len = %lld out of range", (long long)rows,
                    (long long)len);
    if (rows == 0)
        return RED_OK;
    if (!out || misaligned(out, 4))
        return fail(RED_EINVAL, "red_rows: out is NULL or not 4-byte aligned");
    if (len > 0 && (!x || misaligned(x, 4)))
        return fail(RED_EINVAL, "red_rows: x is NULL or not 4-byte aligned");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (len == 0) {
        if (op != RED_SUM)
            return fail(RED_EINVAL, "red_rows: max/min of empty rows");
        if (accum)
            return RED_OK;
        return cuda_fail(cudaMemsetAsync(out, 0, (size_t)rows * sizeof(float), s),
                         "red_rows: cudaMemsetAsync");
    }
    return launch_rows(op, x, rows, len, accum ? 1 : 0, out, s);
}

int red_rows_thread(int op, const float *x, int64_t rows, int len, int accum, float *out, red_stream_t stream)
{
    if (op < RED_SUM || op > RED_MIN)
        return fail(RED_EINVAL, "red_rows_thread: unknown op %d", op);
    if (len < 1 || len > RED_THREAD_MAX_LEN)
        return fail(RED_EINVAL, "red_rows_thread: len = %d outside 1..%d", len, RED_THREAD_MAX_LEN);
    if (rows < 0 || rows > MAX_ELEMS / len)
        return fail(RED_EINVAL, "red_rows_thread: rows = %lld out of range", (long long)rows);
    if (rows == 0)
        return RED_OK;
    if (!out || misaligned(out, 4))
        return fail(RED_EINVAL, "red_rows_thread: out is NULL or not 4-byte aligned");
    if (!x || misaligned(x, 4))
        return fail(RED_EINVAL, "red_rows_thread: x is NULL or not 4-byte aligned");
    return launch_rows_thread(op, x, rows, len, accum ? 1 : 0, out, reinterpret_cast<cudaStream_t>(stream));
}

int red_rows_ragged(int op, const float *x, const int64_t *offsets, int64_t rows, int64_t nnz, int accum,
                    float *out, red_stream_t stream)
{
    if (op < RED_SUM || op > RED_MIN)
        return fail(RED_EINVAL, "red_rows_ragged: unknown op %d", op);
    if (rows < 0 || nnz < 0 || rows > MAX_ELEMS || nnz > MAX_ELEMS)
        return fail(RED_EINVAL, "red_rows_ragged: rows = %lld, nnz = %lld out of range", (long long)rows,
                    (long long)nnz);
    if (rows == 0)
        return RED_OK;
    if (!offsets || misaligned(offsets, 8))
        return fail(RED_EINVAL, "red_rows_ragged: offsets is NULL or not 8-byte aligned");
    if (!out || misaligned(out, 4))
        return fail(RED_EINVAL, "red_rows_ragged: out is NULL or not 4-byte aligned");
    if (nnz > 0 && (!x || misaligned(x, 4)))
        return fail(RED_EINVAL, "red_rows_ragged: x is NULL or not 4-byte aligned");
    return launch_ragged(op, x, offsets, rows, nnz, accum ? 1 : 0, out,
                         reinterpret_cast<cudaStream_t>(stream));
}

int red_cols_ld(int op, int dtype, const void *x, int64_t R, int64_t C, int64_t ld, void *out,
                red_stream_t stream)
{
    if (op < RED_SUM || op > RED_PROD)
        return fail(RED_EINVAL, "red_cols: unknown op %d", op);
    if (dtype < RED_F32 || dtype > RED_U32)
        return fail(RED_EINVAL, "red_cols: unknown dtype %d", dtype);
    if (R < 0 || C < 0 || R > MAX_ELEMS || C > MAX_ELEMS)
        return fail(RED_EINVAL, "red_cols: R = %lld, C = %lld out of range", (long long)R, (long long)C);
    if (ld < C || ld > MAX_ELEMS || (ld > 0 && R > MAX_ELEMS / ld))
        return fail(RED_EINVAL, "red_cols: row stride ld = %lld must be >= C = %lld and R * ld in range",
                    (long long)ld, (long long)C);
    if (R == 0 || C == 0)
        return RED_OK;  // TCOLPROD returns early on an empty valid region; dst untouched
    const uintptr_t esz = (dtype == RED_F32 || dtype == RED_I32 || dtype == RED_U32) ? 4 : 2;
    if (!x || misaligned(x, esz))
        return fail(RED_EINVAL, "red_cols: x is NULL or not aligned to its element size");
    if (!out || misaligned(out, esz))
        return fail(RED_EINVAL, "red_cols: out is NULL or not aligned to its element size");
    return launch_cols(op, dtype, x, R, C, ld, out, reinterpret_cast<cudaStream_t>(stream));
}

int red_cols(int op, int dtype, const void *x, int64_t R, int64_t C, void *out, red_stream_t stream)
{
    return red_cols_ld(op, dtype, x, R, C, C, out, stream);
}

namespace {
uintptr_t elem_bytes(int dtype) { return (dtype == RED_F32 || dtype == RED_I32 || dtype == RED_U32) ? 4 : 2; }
}  // namespace

int red_full_typed(int op, int dtype, const void *x, int64_t n, void *out, red_stream_t stream)
{
    if (op < RED_SUM || op > RED_PROD)
        return fail(RED_EINVAL, "red_full_typed: unknown op %d", op);
    if (dtype < RED_F32 || dtype > RED_U32)
        return fail(RED_EINVAL, "red_full_typed: unknown dtype %d", dtype);
    if (n < 0 || n > MAX_ELEMS)
        return fail(RED_EINVAL, "red_full_typed: n = %lld out of range", (long long)n);
    if (n == 0 && (op == RED_MAX || op == RED_MIN))
        return fail(RED_EINVAL, "red_full_typed: max/min of an empty vector");
    if (!out || misaligned(out, elem_bytes(dtype)))
        return fail(RED_EINVAL, "red_full_typed: out is NULL or not aligned to its element size");
    if (n > 0 && (!x || misaligned(x, elem_bytes(dtype))))
        return fail(RED_EINVAL, "red_full_typed: x is NULL or not aligned to its element size");
    return launch_typed(true, op, dtype, x, 1, n, 0, out, reinterpret_cast<cudaStream_t>(stream));
}

int red_rows_typed(int op, int dtype, const void *x, int64_t rows, int64_t len, int accum, void *out,
                   red_stream_t stream)
{
    if (op < RED_SUM || op > RED_PROD)
        return fail(RED_EINVAL, "red_rows_typed: unknown op %d", op);
    if (dtype < RED_F32 || dtype > RED_U32)
        return fail(RED_EINVAL, "red_rows_typed: unknown dtype %d", dtype);
    if (rows < 0 || len < 0 || rows > MAX_ELEMS || len > MAX_ELEMS || (len > 0 && rows > MAX_ELEMS / len))
        return fail(RED_EINVAL, "red_rows_typed: rows = %lld, len = %lld out of range", (long long)rows,
                    (long long)len);
    if (rows == 0)
        return RED_OK;
    if (len == 0 && (op == RED_MAX || op == RED_MIN))
        return fail(RED_EINVAL, "red_rows_typed: max/min of empty rows");
    if (!out || misaligned(out, elem_bytes(dtype)))
        return fail(RED_EINVAL, "red_rows_typed: out is NULL or not aligned to its element size");
    if (len > 0 && (!x || misaligned(x, elem_bytes(dtype))))
        return fail(RED_EINVAL, "red_rows_typed: x is NULL or not aligned to its element size");
    return launch_typed(false, op, dtype, x, rows, len, accum ? 1 : 0, out, reinterpret_cast<cudaStream_t>(stream));
}

int red_colprod(int dtype, const void *x, int64_t R, int64_t C, void *out, red_stream_t stream)
{
    if (dtype < RED_F32 || dtype > RED_U32)
        return fail(RED_EINVAL, "red_colprod: unknown dtype %d", dtype);
    return red_cols(RED_PROD, dtype, x, R, C, out, stream);
}

int red_set_full_mode(int mode)
{
    if (mode < RED_MODE_AUTO || mode > RED_MODE_ATOMIC)
        return fail(RED_EINVAL, "red_set_full_mode: unknown mode %d", mode);
    g_full_mode.store(mode, std::memory_order_relaxed);
    return RED_OK;
}

int red_get_full_mode(void) { return g_full_mode.load(std::memory_order_relaxed); }

int red_set_knob(int k, int value)
{
    switch (k) {
    case RED_KNOB_ROWS_GROUP:
    case RED_KNOB_RAGGED_GROUP:
        if (!(value == 0 || value == 1 || value == 2 || value == 4 || value == 8 || value == 16 || value == 32))
            return fail(RED_EINVAL, "red_set_knob: lanes per row must be 0 or a power of two <= 32");
        break;
    case RED_KNOB_COLPROD_SPLITS:
        if (value < 0 || value > 65535)
            return fail(RED_EINVAL, "red_set_knob: colprod splits must be in 0..65535");
        break;
    case RED_KNOB_FULL_CTAS_PER_SM:
        if (value < 0 || value > 32)
            return fail(RED_EINVAL, "red_set_knob: CTAs per SM must be in 0..32");
        break;
    case RED_KNOB_RAGGED_STAGED:
        if (value < 0 || value > 2)
            return fail(RED_EINVAL, "red_set_knob: ragged mapping must be 0 (auto), 1 (staged) or 2 (direct)");
        break;
    case RED_KNOB_ROWS_ALIGNED:
        if (value < 0 || value > 2)
            return fail(RED_EINVAL, "red_set_knob: aligned-rows setting must be 0, 1 or 2");
        break;
    case RED_KNOB_COLS_LANES:
        if (!(value == 0 || value == 1 || value == 2 || value == 4 || value == 8 || value == 16 || value == 32))
            return fail(RED_EINVAL, "red_set_knob: lanes per row must be 0 or a power of two <= 32");
        break;
    default:
        return fail(RED_EINVAL, "red_set_knob: unknown knob %d", k);
    }
    g_knobs[k].store(value, std::memory_order_relaxed);
    return RED_OK;
}

int red_get_knob(int k)
{
    if (k < RED_KNOB_ROWS_GROUP || k > RED_KNOB_COLS_LANES)
        return fail(RED_EINVAL, "red_get_knob: unknown knob %d", k);
    return knob(k);
}

const char *red_last_error(void) { return g_err; }

int red_release_workspace(void)
{
    DeviceInfo di;
    const int st = device_info(&di);
    if (st != RED_OK)
        return st;
    std::lock_guard<std::mutex> lock(g_mu);
    Workspace &w = g_ws[di.dev];
    cudaError_t e = cudaSuccess, e2 = cudaSuccess;
    if (w.part)
        e = cudaFree(w.part);
    if (w.tick)
        e2 = cudaFree(w.tick);
    w.part = nullptr;
    w.tick = nullptr;
    if (e != cudaSuccess)
        return cuda_fail(e, "red_release_workspace");
    return cuda_fail(e2, "red_release_workspace");
}

uint64_t red_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int red_version(void) { return 2; }

}  // extern "C"
