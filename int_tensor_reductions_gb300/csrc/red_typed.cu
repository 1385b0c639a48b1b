// red_typed.cu -- full-vector and per-row sum / max / min / product for the
// element types of the column reductions (float, int32, half, bfloat16,
// int16, uint16, uint32), with the accum fold of Apache TVM docs, "reduction
// -> sm100_packed", "How inputs change the algorithm" (the old dst value is
// one more operand).  Arithmetic as red_types.cuh states: a 32-bit
// accumulator per type, one narrowing at the end.
//
// Rows: a group of G lanes owns a row; lane l folds elements l, l+G, ... of
// it (consecutive lanes read consecutive elements), 4 loads in flight; the
// group combines through a butterfly.  Full vector: every thread of the grid
// folds elements tid, tid+nthreads, ..., the CTA combines through a warp
// butterfly and shared memory, and the last CTA to finish folds the CTA
// partials (last-block grid stage, workspace partials).
#include "red_internal.h"
#include "red_prims.cuh"
#include "red_types.cuh"
#include "red.h"

namespace red {
namespace {

constexpr int TY_NT = 256;
constexpr int TY_U = 4;

template <typename A>
__device__ __forceinline__ A shfl_xor(A v, int off)
{
    return __shfl_xor_sync(0xffffffffu, v, off);
}

template <int OP, typename A, int W>
__device__ __forceinline__ A tree(A v)
{
#pragma unroll
    for (int off = W / 2; off > 0; off >>= 1)
        v = Comb<OP, A>::op(v, shfl_xor(v, off));
    return v;
}

template <int OP, int DT, int G>
__global__ void __launch_bounds__(TY_NT)
typed_rows_kernel(const typename Elem<DT>::T *__restrict__ x, int64_t rows, int64_t len, int accum,
                  typename Elem<DT>::T *__restrict__ out)
{
    using E = Elem<DT>;
    using A = typename E::A;
    using K = Comb<OP, A>;
    constexpr int GPW = 32 / G;
    const int lane = threadIdx.x & 31, gl = lane & (G - 1), gw = lane / G;
    const int64_t warp = ((int64_t)blockIdx.x * TY_NT + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * TY_NT) >> 5;
    for (int64_t r0 = warp * GPW; r0 < rows; r0 += nwarps * GPW) {  // warp-uniform
        const int64_t r = r0 + gw;
        const bool live = r < rows;
        A acc = K::identity();
        if (live) {
            const typename E::T *p = x + r * len;
            int64_t k = gl;
            for (; k + (TY_U - 1) * G < len; k += TY_U * G) {
                uint32_t b[TY_U];
#pragma unroll
                for (int u = 0; u < TY_U; ++u)
                    b[u] = load_bits<DT>(p + k + u * G);
#pragma unroll
                for (int u = 0; u < TY_U; ++u)
                    acc = K::op(acc, E::widen(b[u]));
            }
            for (; k < len; k += G)
                acc = K::op(acc, E::widen(load_bits<DT>(p + k)));
            if (accum && gl == 0)
                acc = K::op(E::widen(bits_of<DT>(out[r])), acc);
        }
        acc = tree<OP, A, G>(acc);
        if (live && gl == 0)
            out[r] = E::narrow(acc);
    }
}

template <int OP, int DT>
__global__ void __launch_bounds__(TY_NT)
typed_full_kernel(const typename Elem<DT>::T *__restrict__ x, int64_t n, typename Elem<DT>::A *__restrict__ part,
                  unsigned *__restrict__ tick, typename Elem<DT>::T *__restrict__ out)
{
    using E = Elem<DT>;
    using A = typename E::A;
    using K = Comb<OP, A>;
    __shared__ A s_red[TY_NT / 32];
    __shared__ int s_last;
    const int64_t tid = (int64_t)blockIdx.x * TY_NT + threadIdx.x;
    const int64_t nth = (int64_t)gridDim.x * TY_NT;
    A acc = K::identity();
    int64_t k = tid;
    for (; k + (TY_U - 1) * nth < n; k += TY_U * nth) {
        uint32_t b[TY_U];
#pragma unroll
        for (int u = 0; u < TY_U; ++u)
            b[u] = load_bits<DT>(x + k + u * nth);
#pragma unroll
        for (int u = 0; u < TY_U; ++u)
            acc = K::op(acc, E::widen(b[u]));
    }
    for (; k < n; k += nth)
        acc = K::op(acc, E::widen(load_bits<DT>(x + k)));

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    acc = tree<OP, A, 32>(acc);
    if (lane == 0)
        s_red[warp] = acc;
    __syncthreads();
    if (warp == 0) {
        acc = lane < TY_NT / 32 ? s_red[lane] : K::identity();
        acc = tree<OP, A, TY_NT / 32>(acc);
    }
    if (gridDim.x == 1) {
        if (threadIdx.x == 0)
            out[0] = E::narrow(acc);
        return;
    }
    if (threadIdx.x == 0) {
        part[blockIdx.x] = acc;
        __threadfence();
        s_last = (atomicAdd(tick, 1u) == gridDim.x - 1);
    }
    __syncthreads();
    if (!s_last)
        return;
    __threadfence();
    A w = K::identity();
    for (unsigned i = threadIdx.x; i < gridDim.x; i += TY_NT)
        w = K::op(w, ldcg_a<A>(part + i));
    w = tree<OP, A, 32>(w);
    if (lane == 0)
        s_red[warp] = w;
    __syncthreads();
    if (threadIdx.x == 0) {
        A t = K::identity();
        for (int i = 0; i < TY_NT / 32; ++i)
            t = K::op(t, s_red[i]);
        out[0] = E::narrow(t);
        *tick = 0;
    }
}

// Identity of the operator in the element type (written for empty sums and
// products).
template <int OP, int DT>
__global__ void typed_fill_kernel(typename Elem<DT>::T *out, int64_t n)
{
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n)
        out[i] = Elem<DT>::narrow(Comb<OP, typename Elem<DT>::A>::identity());
}

template <int OP, int DT>
int typed_rows_dt(const void *xv, int64_t rows, int64_t len, int accum, void *outv, cudaStream_t s, int sms)
{
    using T = typename Elem<DT>::T;
    const T *x = static_cast<const T *>(xv);
    T *out = static_cast<T *>(outv);
    if (len == 0) {
        if (!accum) {
            typed_fill_kernel<OP, DT><<<(unsigned)((rows + 255) / 256), 256, 0, s>>>(out, rows);
            count_launches(1);
        }
        return cuda_fail(cudaGetLastError(), "red_rows_typed launch");
    }
    int g = 1;
    while (g < 32 && (int64_t)g * 32 <= len)
        g *= 2;
    const int64_t rows_per_cta = (int64_t)(TY_NT / 32) * (32 / g);
    int64_t ctas = (rows + rows_per_cta - 1) / rows_per_cta;
    if (ctas > (int64_t)sms * 8)
        ctas = (int64_t)sms * 8;
    switch (g) {
    case 1: typed_rows_kernel<OP, DT, 1><<<(unsigned)ctas, TY_NT, 0, s>>>(x, rows, len, accum, out); break;
    case 2: typed_rows_kernel<OP, DT, 2><<<(unsigned)ctas, TY_NT, 0, s>>>(x, rows, len, accum, out); break;
    case 4: typed_rows_kernel<OP, DT, 4><<<(unsigned)ctas, TY_NT, 0, s>>>(x, rows, len, accum, out); break;
    case 8: typed_rows_kernel<OP, DT, 8><<<(unsigned)ctas, TY_NT, 0, s>>>(x, rows, len, accum, out); break;
    case 16: typed_rows_kernel<OP, DT, 16><<<(unsigned)ctas, TY_NT, 0, s>>>(x, rows, len, accum, out); break;
    default: typed_rows_kernel<OP, DT, 32><<<(unsigned)ctas, TY_NT, 0, s>>>(x, rows, len, accum, out); break;
    }
    count_launches(1);
    return cuda_fail(cudaGetLastError(), "red_rows_typed launch");
}

template <int OP, int DT>
int typed_full_dt(const void *xv, int64_t n, void *outv, cudaStream_t s, int sms)
{
    using T = typename Elem<DT>::T;
    using A = typename Elem<DT>::A;
    const T *x = static_cast<const T *>(xv);
    T *out = static_cast<T *>(outv);
    if (n == 0) {
        typed_fill_kernel<OP, DT><<<1, 32, 0, s>>>(out, 1);
        count_launches(1);
        return cuda_fail(cudaGetLastError(), "red_full_typed launch");
    }
    static int occ = 0;
    if (occ == 0)
        occ = occupancy((const void *)typed_full_kernel<OP, DT>, TY_NT);
    if (occ <= 0)
        return fail(RED_ECUDA, "red_full_typed: kernel cannot be resident on this device");
    const int64_t want = (n + (int64_t)TY_NT * TY_U - 1) / ((int64_t)TY_NT * TY_U);
    int64_t ctas = (int64_t)sms * occ;
    if (want < ctas)
        ctas = want;
    if (ctas < 1)
        ctas = 1;
    Workspace ws;
    if (ctas > 1) {
        const int st = get_workspace(&ws);
        if (st != RED_OK)
            return st;
    }
    typed_full_kernel<OP, DT><<<(unsigned)ctas, TY_NT, 0, s>>>(x, n, static_cast<A *>(ws.part), ws.tick, out);
    count_launches(1);
    return cuda_fail(cudaGetLastError(), "red_full_typed launch");
}

template <int OP>
int typed_op(bool full, int dtype, const void *x, int64_t rows, int64_t len, int accum, void *out, cudaStream_t s,
             int sms)
{
#define RED_TYPED_CASE(DT)                                                                                      \
    case DT:                                                                                                     \
        return full ? typed_full_dt<OP, DT>(x, len, out, s, sms) : typed_rows_dt<OP, DT>(x, rows, len, accum, out, s, sms);
    switch (dtype) {
        RED_TYPED_CASE(RED_F32)
        RED_TYPED_CASE(RED_I32)
        RED_TYPED_CASE(RED_F16)
        RED_TYPED_CASE(RED_BF16)
        RED_TYPED_CASE(RED_I16)
        RED_TYPED_CASE(RED_U16)
    default:
        return full ? typed_full_dt<OP, RED_U32>(x, len, out, s, sms)
                    : typed_rows_dt<OP, RED_U32>(x, rows, len, accum, out, s, sms);
    }
#undef RED_TYPED_CASE
}

}  // namespace

int launch_typed(bool full, int op, int dtype, const void *x, int64_t rows, int64_t len, int accum, void *out,
                 cudaStream_t s)
{
    DeviceInfo di;
    const int st = device_info(&di);
    if (st != RED_OK)
        return st;
    switch (op) {
    case RED_SUM: return typed_op<RED_SUM>(full, dtype, x, rows, len, accum, out, s, di.sms);
    case RED_MAX: return typed_op<RED_MAX>(full, dtype, x, rows, len, accum, out, s, di.sms);
    case RED_MIN: return typed_op<RED_MIN>(full, dtype, x, rows, len, accum, out, s, di.sms);
    default: return typed_op<RED_PROD>(full, dtype, x, rows, len, accum, out, s, di.sms);
    }
}

}  // namespace red
