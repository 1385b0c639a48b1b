// red_typed.cu -- full-vector and per-row sum / max / min / product for the
// element types of the column reductions (float, int32, half, bfloat16,
// int16, uint16, uint32), with the accum fold of Apache TVM docs, "reduction
// -> sm100_packed", "How inputs change the algorithm" (the old dst value is
// one more operand).  Arithmetic as red_types.cuh states: a 32-bit
// accumulator per type, one narrowing at the end.
//
// Both read the span (a row, or the whole vector) as its 32-byte aligned
// interior in 256-bit blocks (8 or 16 elements each, widened), 4 blocks in
// flight per thread, plus its unaligned head and tail as naturally aligned
// pieces of 1, 2, 4 and 8 elements, so every load lies inside the span.
// Rows: a group of G lanes owns a row and splits its blocks; the group
// combines through a butterfly.  Full vector: the grid splits the blocks, the
// CTA combines through a warp butterfly and shared memory, and the last CTA
// to finish folds the CTA partials (last-block grid stage, workspace
// partials).  Rows whose byte length is a power of two up to 256 bytes,
// from a 32-byte aligned base, go to red_typed_tiny.cu instead.
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

// Elements per 32-byte block.
template <int DT>
__host__ __device__ constexpr int epb() { return 32 / (int)sizeof(typename Elem<DT>::T); }

// Fold the K naturally aligned elements at p (K * element size = 2, 4, 8, 16
// or 32 bytes) into acc, widened.
template <int OP, int DT, int K>
__device__ __forceinline__ void fold_piece(const typename Elem<DT>::T *p, typename Elem<DT>::A &acc)
{
    using E = Elem<DT>;
    using K_ = Comb<OP, typename E::A>;
    constexpr int SZ = (int)sizeof(typename E::T);
    constexpr int BYTES = K * SZ;
    static_assert(BYTES == 2 || BYTES == 4 || BYTES == 8 || BYTES == 16 || BYTES == 32, "piece size");
    if constexpr (BYTES == 2) {
        acc = K_::op(acc, E::widen(__ldg(reinterpret_cast<const unsigned short *>(p))));
    } else {
        constexpr int W = BYTES / 4;
        uint32_t w[W];
        if constexpr (W == 1) {
            w[0] = __ldg(reinterpret_cast<const unsigned int *>(p));
        } else if constexpr (W == 2) {
            const uint2 t = __ldg(reinterpret_cast<const uint2 *>(p));
            w[0] = t.x;
            w[1] = t.y;
        } else if constexpr (W == 4) {
            uint32_t (&w4)[4] = w;
            ld4u(reinterpret_cast<const uint32_t *>(p), w4);
        } else {
            uint32_t (&w8)[8] = w;
            ld8u(reinterpret_cast<const uint32_t *>(p), w8);
        }
#pragma unroll
        for (int k = 0; k < W; ++k) {
            if constexpr (SZ == 4) {
                acc = K_::op(acc, E::widen(w[k]));
            } else {
                acc = K_::op(acc, E::widen(w[k] & 0xffffu));
                acc = K_::op(acc, E::widen(w[k] >> 16));
            }
        }
    }
}

// Fold one 32-byte block already loaded as 8 words.
template <int OP, int DT>
__device__ __forceinline__ void fold_words(const uint32_t (&w)[8], typename Elem<DT>::A &acc)
{
    using E = Elem<DT>;
    using K_ = Comb<OP, typename E::A>;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        if constexpr (sizeof(typename E::T) == 4) {
            acc = K_::op(acc, E::widen(w[k]));
        } else {
            acc = K_::op(acc, E::widen(w[k] & 0xffffu));
            acc = K_::op(acc, E::widen(w[k] >> 16));
        }
    }
}

// The unaligned head [b, a) of a span (h = a - b < epb elements, a on a
// 32-byte boundary) as at most one piece of each power-of-two size, each
// naturally aligned: sizes ascend with the address.
template <int OP, int DT>
__device__ __forceinline__ void fold_head(const typename Elem<DT>::T *pb, int h, typename Elem<DT>::A &acc)
{
    if (h & 1)
        fold_piece<OP, DT, 1>(pb, acc);
    if (h & 2)
        fold_piece<OP, DT, 2>(pb + (h & 1), acc);
    if (h & 4)
        fold_piece<OP, DT, 4>(pb + (h & 3), acc);
    if constexpr (epb<DT>() > 8)
        if (h & 8)
            fold_piece<OP, DT, 8>(pb + (h & 7), acc);
}

// The tail [z, e) (t = e - z < epb elements, z on a 32-byte boundary):
// sizes descend with the address.
template <int OP, int DT>
__device__ __forceinline__ void fold_tail(const typename Elem<DT>::T *pz, int t, typename Elem<DT>::A &acc)
{
    int o = 0;
    if constexpr (epb<DT>() > 8) {
        if (t & 8) {
            fold_piece<OP, DT, 8>(pz, acc);
            o = 8;
        }
    }
    if (t & 4) {
        fold_piece<OP, DT, 4>(pz + o, acc);
        o += 4;
    }
    if (t & 2) {
        fold_piece<OP, DT, 2>(pz + o, acc);
        o += 2;
    }
    if (t & 1)
        fold_piece<OP, DT, 1>(pz + o, acc);
}

// Element index (relative to x) of the first 32-byte boundary at or after
// element i, for a base x that is element-aligned.
template <int DT>
__device__ __forceinline__ int64_t up_to_block(const typename Elem<DT>::T *x, int64_t i)
{
    constexpr int SZ = (int)sizeof(typename Elem<DT>::T);
    const int64_t mis = (int64_t)(((uintptr_t)x & 31u) / SZ);  // x's offset from a boundary, in elements
    return ((i + mis + epb<DT>() - 1) & ~int64_t(epb<DT>() - 1)) - mis;
}

template <int DT>
__device__ __forceinline__ int64_t down_to_block(const typename Elem<DT>::T *x, int64_t i)
{
    constexpr int SZ = (int)sizeof(typename Elem<DT>::T);
    const int64_t mis = (int64_t)(((uintptr_t)x & 31u) / SZ);
    return ((i + mis) & ~int64_t(epb<DT>() - 1)) - mis;
}

template <int OP, int DT, int G>
__global__ void __launch_bounds__(TY_NT)
typed_rows_kernel(const typename Elem<DT>::T *__restrict__ x, int64_t rows, int64_t len, int accum,
                  typename Elem<DT>::T *__restrict__ out)
{
    pdl_enter();
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
            // Row [b, e): aligned interior [a, z) in 32-byte blocks spread
            // over the group's lanes (TY_U in flight per lane); head and tail
            // as naturally aligned pieces by lane 0 and the last lane.  Every
            // load lies inside the row.
            const int64_t b = r * len, e = b + len;
            const int64_t a = up_to_block<DT>(x, b), z = down_to_block<DT>(x, e);
            if (a <= z) {
                if (gl == 0)
                    fold_head<OP, DT>(x + b, (int)(a - b), acc);
                if (gl == G - 1)
                    fold_tail<OP, DT>(x + z, (int)(e - z), acc);
                const int64_t nblk = (z - a) / epb<DT>();
                const typename E::T *q = x + a;
                for (int64_t c0 = gl; c0 < nblk; c0 += (int64_t)TY_U * G) {
                    uint32_t w[TY_U][8];  // all loads out before any fold
#pragma unroll
                    for (int u = 0; u < TY_U; ++u)
                        if (c0 + u * G < nblk)
                            ld8u(reinterpret_cast<const uint32_t *>(q + (c0 + u * G) * epb<DT>()), w[u]);
#pragma unroll
                    for (int u = 0; u < TY_U; ++u)
                        if (c0 + u * G < nblk)
                            fold_words<OP, DT>(w[u], acc);
                }
            } else {
                for (int64_t k = b + gl; k < e; k += G)  // the row inside one block
                    acc = K::op(acc, E::widen(load_bits<DT>(x + k)));
            }
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
    pdl_enter();
    using E = Elem<DT>;
    using A = typename E::A;
    using K = Comb<OP, A>;
    __shared__ A s_red[TY_NT / 32];
    __shared__ int s_last;
    const int64_t tid = (int64_t)blockIdx.x * TY_NT + threadIdx.x;
    const int64_t nth = (int64_t)gridDim.x * TY_NT;
    A acc = K::identity();
    const int64_t a = up_to_block<DT>(x, 0), z = down_to_block<DT>(x, n);
    if (a <= z) {
        // aligned interior as 32-byte blocks, grid-stride, TY_U in flight per
        // thread; the head and tail pieces by the first and the last thread
        if (tid == 0)
            fold_head<OP, DT>(x, (int)a, acc);
        if (tid == nth - 1)
            fold_tail<OP, DT>(x + z, (int)(n - z), acc);
        const int64_t nblk = (z - a) / epb<DT>();
        const typename E::T *q = x + a;
        for (int64_t c0 = tid; c0 < nblk; c0 += (int64_t)TY_U * nth) {
            uint32_t w[TY_U][8];  // all loads out before any fold
#pragma unroll
            for (int u = 0; u < TY_U; ++u)
                if (c0 + u * nth < nblk)
                    ld8u(reinterpret_cast<const uint32_t *>(q + (c0 + u * nth) * epb<DT>()), w[u]);
#pragma unroll
            for (int u = 0; u < TY_U; ++u)
                if (c0 + u * nth < nblk)
                    fold_words<OP, DT>(w[u], acc);
        }
    } else {
        for (int64_t k = tid; k < n; k += nth)  // the whole vector inside one block
            acc = K::op(acc, E::widen(load_bits<DT>(x + k)));
    }

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
    pdl_enter();
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
        cudaError_t e = cudaSuccess;
        if (!accum) {
            e = launch_pdl(typed_fill_kernel<OP, DT>, dim3((unsigned)((rows + 255) / 256)), dim3(256), s, out, rows);
            count_launches(1);
        }
        return cuda_fail(e != cudaSuccess ? e : cudaGetLastError(), "red_rows_typed launch");
    }
    // From a 32-byte aligned base: rows of 2, 4, 8, 16 or 32 bytes (whole
    // blocks per thread, several rows each), and rows of 2, 4 or 8 whole
    // blocks (consecutive lanes on consecutive blocks of the matrix; measured
    // against lanes per row: bf16 rows of 64 6.65 vs 5.69 TB/s, fp32 rows of
    // 64 6.67 vs 6.52, int32 rows of 256 (32 blocks) 6.68 vs 6.83).
    if ((((uintptr_t)x) & 31u) == 0) {
        const bool tiny = len <= epb<DT>() && epb<DT>() % len == 0;
        const int64_t rb = len % epb<DT>() == 0 ? len / epb<DT>() : 0;
        if (tiny || rb == 2 || rb == 4 || rb == 8)
            return launch_typed_tiny(OP, DT, x, rows, (int)len, accum, out, s, sms);
    }
    // Lanes per row: the largest power of two (<= 32) that still leaves each
    // lane TY_U whole 32-byte blocks of the row, so a lane keeps TY_U loads
    // in flight (bf16 rows of 64 elements: 1 lane, not 4 lanes of one block).
    int g = 1;
    while (g < 32 && (int64_t)(2 * g) * TY_U * epb<DT>() <= len)
        g *= 2;
    const int64_t rows_per_cta = (int64_t)(TY_NT / 32) * (32 / g);
    int64_t ctas = (rows + rows_per_cta - 1) / rows_per_cta;
    if (ctas > (int64_t)sms * 8)
        ctas = (int64_t)sms * 8;
    const dim3 grid((unsigned)ctas), block(TY_NT);
    cudaError_t e;
    switch (g) {
    case 1: e = launch_pdl(typed_rows_kernel<OP, DT, 1>, grid, block, s, x, rows, len, accum, out); break;
    case 2: e = launch_pdl(typed_rows_kernel<OP, DT, 2>, grid, block, s, x, rows, len, accum, out); break;
    case 4: e = launch_pdl(typed_rows_kernel<OP, DT, 4>, grid, block, s, x, rows, len, accum, out); break;
    case 8: e = launch_pdl(typed_rows_kernel<OP, DT, 8>, grid, block, s, x, rows, len, accum, out); break;
    case 16: e = launch_pdl(typed_rows_kernel<OP, DT, 16>, grid, block, s, x, rows, len, accum, out); break;
    default: e = launch_pdl(typed_rows_kernel<OP, DT, 32>, grid, block, s, x, rows, len, accum, out); break;
    }
    count_launches(1);
    return cuda_fail(e != cudaSuccess ? e : cudaGetLastError(), "red_rows_typed launch");
}

template <int OP, int DT>
int typed_full_dt(const void *xv, int64_t n, void *outv, cudaStream_t s, int sms)
{
    using T = typename Elem<DT>::T;
    using A = typename Elem<DT>::A;
    const T *x = static_cast<const T *>(xv);
    T *out = static_cast<T *>(outv);
    if (n == 0) {
        const cudaError_t e = launch_pdl(typed_fill_kernel<OP, DT>, dim3(1), dim3(32), s, out, (int64_t)1);
        count_launches(1);
        return cuda_fail(e != cudaSuccess ? e : cudaGetLastError(), "red_full_typed launch");
    }
    static std::atomic<int> occ_cache{0};
    const int occ = cached_occupancy(occ_cache, (const void *)typed_full_kernel<OP, DT>, TY_NT);
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
    const cudaError_t e = launch_pdl(typed_full_kernel<OP, DT>, dim3((unsigned)ctas), dim3(TY_NT), s, x, n,
                                     static_cast<A *>(ws.part), ws.tick, out);
    count_launches(1);
    return cuda_fail(e != cudaSuccess ? e : cudaGetLastError(), "red_full_typed launch");
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
