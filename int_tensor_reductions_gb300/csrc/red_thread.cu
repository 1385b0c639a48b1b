// red_thread.cu -- red_rows_thread: one thread per row, each row reduced by
// the thread-scope fold of the public device header red_device.cuh (Apache
// TVM docs, "reduction -> sm100_packed", "Algorithm"), so the rounding order
// of every row's sum is the page's and depends on the row length alone.
//
// The row length is a template parameter (the register array of the fold
// has a static size, like the page's local buffer), instantiated for
// 1..RED_THREAD_MAX_LEN.  A CTA of 128 threads folds tiles of 128
// consecutive rows (one tile per CTA, or a persistent grid looping over the
// tiles when rows hold at most 8 floats);
// their values (128 x len floats, contiguous) are staged through shared
// memory with coalesced loads (256-bit when the tile starts on a 32-byte
// boundary, else one float per thread per load), at an odd row stride so
// that the threads' row reads hit distinct banks, then each thread copies
// its row into registers.
#include "red_device.cuh"
#include "red_internal.h"
#include "red_prims.cuh"
#include "red.h"

namespace red {
namespace {

constexpr int TH_NT = 128;
// 256-bit staging loads in flight per thread: 4 (a 16 KB tile of rows of 32
// in one batch), 8 for rows of 44 floats or more (measured: from 33 to 40
// floats the extra registers cost more than the second batch)
template <int N>
__host__ __device__ constexpr int th_u() { return N >= 44 ? 8 : 4; }

template <int OP, int N>
__global__ void __launch_bounds__(TH_NT)
thread_rows_kernel(const float *__restrict__ x, int64_t rows, int accum, float *__restrict__ out)
{
    constexpr int STRIDE = N | 1;  // odd row stride in shared memory
    __shared__ float s_val[TH_NT * STRIDE];
    pdl_enter();
    const int64_t ntiles = (rows + TH_NT - 1) / TH_NT;
    for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
        const int64_t r0 = tile * TH_NT;
        const int nr = (int)((rows - r0) < TH_NT ? (rows - r0) : TH_NT);
        const float *src = x + r0 * N;
        const int tot = nr * N;
        int g0 = 0;  // elements below g0 are staged by the 256-bit loop
        __syncthreads();  // the previous tile's reads of s_val are done
        if ((((uintptr_t)src) & 31u) == 0) {
            // 256-bit loads, TH_U in flight per thread before any shared store
            constexpr int TH_U = th_u<N>();
            const int nv = tot >> 3;
            for (int c0 = threadIdx.x; c0 < nv; c0 += TH_U * TH_NT) {
                float v[TH_U][8];
#pragma unroll
                for (int u = 0; u < TH_U; ++u)
                    if (c0 + u * TH_NT < nv)
                        ld8(src + 8 * (c0 + u * TH_NT), v[u]);
#pragma unroll
                for (int u = 0; u < TH_U; ++u)
                    if (c0 + u * TH_NT < nv)
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            const int g = 8 * (c0 + u * TH_NT) + k;
                            const int t = g / N, i = g - t * N;
                            s_val[t * STRIDE + i] = v[u][k];
                        }
            }
            g0 = nv << 3;
        }
        for (int g = g0 + threadIdx.x; g < tot; g += TH_NT) {
            const int t = g / N, i = g - t * N;
            s_val[t * STRIDE + i] = __ldg(src + g);
        }
        __syncthreads();
        if (threadIdx.x < nr) {
            float a[N];
#pragma unroll
            for (int i = 0; i < N; ++i)
                a[i] = s_val[threadIdx.x * STRIDE + i];
            const int64_t r = r0 + threadIdx.x;
            const float old = accum ? out[r] : 0.0f;
            float v;
            if (OP == RED_SUM)
                v = red_dev::thread_sum<N>(a, accum != 0, old);
            else if (OP == RED_MAX)
                v = red_dev::thread_max<N>(a, accum != 0, old);
            else
                v = red_dev::thread_min<N>(a, accum != 0, old);
            out[r] = v;
        }
    }
}

// Rows of N = 1, 2, 4 or 8 floats from a 32-byte aligned base: a 32-byte
// block holds 8/N whole rows, so each thread folds the rows of its blocks
// straight from registers (256-bit loads, TINY_U in flight, no shared memory)
// with the same thread-scope fold; the rows past the last whole block (fewer
// than 8/N) are read element by element.
constexpr int TINY_NT = 256;
constexpr int TINY_U = 4;

template <int OP, int N>
__device__ __forceinline__ float fold_row(const float (&a)[N], int accum, float old)
{
    if (OP == RED_SUM)
        return red_dev::thread_sum<N>(a, accum != 0, old);
    else if (OP == RED_MAX)
        return red_dev::thread_max<N>(a, accum != 0, old);
    else
        return red_dev::thread_min<N>(a, accum != 0, old);
}

// RPB consecutive floats at p (RPB = 2: 8-byte aligned; 4 or 8: 16-byte
// aligned), as float2 / float4 accesses.
template <int RPB>
__device__ __forceinline__ void tiny_ld(const float *p, float (&v)[RPB])
{
    if constexpr (RPB == 2) {
        const float2 t = *reinterpret_cast<const float2 *>(p);
        v[0] = t.x;
        v[1] = t.y;
    } else {
#pragma unroll
        for (int k = 0; k < RPB; k += 4) {
            const float4 t = *reinterpret_cast<const float4 *>(p + k);
            v[k] = t.x;
            v[k + 1] = t.y;
            v[k + 2] = t.z;
            v[k + 3] = t.w;
        }
    }
}

template <int RPB>
__device__ __forceinline__ void tiny_st(float *p, const float (&v)[RPB])
{
    if constexpr (RPB == 2) {
        *reinterpret_cast<float2 *>(p) = make_float2(v[0], v[1]);
    } else {
#pragma unroll
        for (int k = 0; k < RPB; k += 4)
            *reinterpret_cast<float4 *>(p + k) = make_float4(v[k], v[k + 1], v[k + 2], v[k + 3]);
    }
}

template <int OP, int N>
__global__ void __launch_bounds__(TINY_NT)
tiny_rows_kernel(const float *__restrict__ x, int64_t rows, int accum, float *__restrict__ out)
{
    pdl_enter();
    constexpr int RPB = 8 / N;  // rows per block
    const int64_t nblk = rows / RPB;
    const bool vec_out = RPB > 1 && (((uintptr_t)out) & (uintptr_t)(4 * (RPB < 4 ? RPB : 4) - 1)) == 0;
    const int64_t tid = (int64_t)blockIdx.x * TINY_NT + threadIdx.x;
    const int64_t nth = (int64_t)gridDim.x * TINY_NT;
    for (int64_t c0 = tid; c0 < nblk; c0 += TINY_U * nth) {
        float v[TINY_U][8];
#pragma unroll
        for (int u = 0; u < TINY_U; ++u)
            if (c0 + u * nth < nblk)
                ld8(x + 8 * (c0 + u * nth), v[u]);
#pragma unroll
        for (int u = 0; u < TINY_U; ++u)
            if (c0 + u * nth < nblk) {
                // the block's RPB results are consecutive in out: one vector
                // access when out allows it (a lane per row would touch a
                // separate sector with every 4-byte store)
                float *o = out + (c0 + u * nth) * RPB;
                float old[RPB], res[RPB];
#pragma unroll
                for (int q = 0; q < RPB; ++q)
                    old[q] = 0.0f;
                if (accum) {
                    if (vec_out)
                        tiny_ld<RPB>(o, old);
                    else
#pragma unroll
                        for (int q = 0; q < RPB; ++q)
                            old[q] = o[q];
                }
#pragma unroll
                for (int q = 0; q < RPB; ++q) {
                    float a[N];
#pragma unroll
                    for (int i = 0; i < N; ++i)
                        a[i] = v[u][q * N + i];
                    res[q] = fold_row<OP, N>(a, accum, old[q]);
                }
                if (vec_out)
                    tiny_st<RPB>(o, res);
                else
#pragma unroll
                    for (int q = 0; q < RPB; ++q)
                        o[q] = res[q];
            }
    }
    const int64_t r = nblk * RPB + tid;
    if (r < rows) {
        float a[N];
#pragma unroll
        for (int i = 0; i < N; ++i)
            a[i] = __ldg(x + r * N + i);
        out[r] = fold_row<OP, N>(a, accum, accum ? out[r] : 0.0f);
    }
}

template <int OP, int N>
int launch_n(const float *x, int64_t rows, int accum, float *out, cudaStream_t s)
{
    if constexpr (N == 1 || N == 2 || N == 4 || N == 8) {
        if ((((uintptr_t)x) & 31u) == 0) {
            DeviceInfo di;
            const int st = device_info(&di);
            if (st != RED_OK)
                return st;
            static std::atomic<int> occ_cache{0};
            const int occ = cached_occupancy(occ_cache, (const void *)tiny_rows_kernel<OP, N>, TINY_NT);
            if (occ <= 0)
                return fail(RED_ECUDA, "red_rows_thread: kernel cannot be resident on this device");
            const int64_t need = (rows / (8 / N) + (int64_t)TINY_NT * TINY_U - 1) / ((int64_t)TINY_NT * TINY_U) + 1;
            int64_t ctas = (int64_t)di.sms * occ;
            if (need < ctas)
                ctas = need;
            const cudaError_t e =
                launch_pdl(tiny_rows_kernel<OP, N>, dim3((unsigned)ctas), dim3(TINY_NT), s, x, rows, accum, out);
            count_launches(1);
            return cuda_fail(e != cudaSuccess ? e : cudaGetLastError(), "red_rows_thread launch");
        }
    }
    // Rows of at most 8 floats: a persistent grid of resident CTAs loops over
    // the tiles of 128 rows (a tile is only 4 KB, and launching one CTA per
    // tile costs more than the work); longer rows: one CTA per tile, whose
    // staging overlaps other CTAs' folds (measured faster from 12 floats up).
    DeviceInfo di;
    const int st = device_info(&di);
    if (st != RED_OK)
        return st;
    static std::atomic<int> occ_cache{0};
    const int occ = cached_occupancy(occ_cache, (const void *)thread_rows_kernel<OP, N>, TH_NT);
    if (occ <= 0)
        return fail(RED_ECUDA, "red_rows_thread: kernel cannot be resident on this device");
    int64_t ctas = (rows + TH_NT - 1) / TH_NT;
    if (N <= 8 && ctas > (int64_t)di.sms * occ)
        ctas = (int64_t)di.sms * occ;
    if (ctas > 0x7fffffffLL)
        return fail(RED_EINVAL, "red_rows_thread: too many rows");
    const cudaError_t e = launch_pdl(thread_rows_kernel<OP, N>, dim3((unsigned)ctas), dim3(TH_NT), s, x, rows, accum, out);
    count_launches(1);
    return cuda_fail(e != cudaSuccess ? e : cudaGetLastError(), "red_rows_thread launch");
}

// Dispatch a runtime length 1..RED_THREAD_MAX_LEN onto the instantiations.
template <int OP, int N = 1>
int dispatch(int len, const float *x, int64_t rows, int accum, float *out, cudaStream_t s)
{
    if constexpr (N > RED_THREAD_MAX_LEN) {
        return fail(RED_EINVAL, "red_rows_thread: len %d out of range", len);
    } else {
        if (len == N)
            return launch_n<OP, N>(x, rows, accum, out, s);
        return dispatch<OP, N + 1>(len, x, rows, accum, out, s);
    }
}

}  // namespace

int launch_rows_thread(int op, const float *x, int64_t rows, int len, int accum, float *out, cudaStream_t s)
{
    switch (op) {
    case RED_SUM: return dispatch<RED_SUM>(len, x, rows, accum, out, s);
    case RED_MAX: return dispatch<RED_MAX>(len, x, rows, accum, out, s);
    default: return dispatch<RED_MIN>(len, x, rows, accum, out, s);
    }
}

}  // namespace red
