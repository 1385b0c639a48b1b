// red_typed_tiny.cu -- per-row sum / max / min / product (with accum) of
// short typed rows from a 32-byte aligned base.  Rows of 2, 4, 8, 16 or 32
// bytes: several whole rows per 256-bit block, so a thread keeps four
// 32-byte loads in flight however short the rows are, and the results of a
// block leave as one vector store.  Rows of 2, 4 or 8 whole blocks (64 to
// 256 bytes): the blocks of the matrix read in order across the lanes, a
// row's blocks meeting in a butterfly over the lanes that hold them.  Same operation and arithmetic as the row
// kernel of red_typed.cu (Apache TVM docs, "reduction -> sm100_packed", "How
// inputs change the algorithm": the old dst value is one more operand); a
// 32-bit accumulator per element type, one narrowing at the end.
#include "red_internal.h"
#include "red_prims.cuh"
#include "red_types.cuh"
#include "red.h"

namespace red {
namespace {

constexpr int TY_NT = 256;
constexpr int TY_U = 4;

// Elements per 32-byte block.
template <int DT>
__host__ __device__ constexpr int epb() { return 32 / (int)sizeof(typename Elem<DT>::T); }

// Element j (0 <= j < epb) of a 32-byte block loaded as 8 words, widened.
template <int DT>
__device__ __forceinline__ typename Elem<DT>::A block_elem(const uint32_t (&w)[8], int j)
{
    using E = Elem<DT>;
    if constexpr (sizeof(typename E::T) == 4)
        return E::widen(w[j]);
    else
        return E::widen((j & 1) ? (w[j >> 1] >> 16) : (w[j >> 1] & 0xffffu));
}

// Store the RPB consecutive results of one block at o (RPB * element size =
// 32 / NE bytes): as 16-, 8- or 4-byte words when the destination allows
// it (a lane per element would touch a sector per 2- or 4-byte store).
template <int DT, int RPB>
__device__ __forceinline__ void store_results(typename Elem<DT>::T *o, const typename Elem<DT>::T (&res)[RPB], bool vec)
{
    using T = typename Elem<DT>::T;
    constexpr int BYTES = RPB * (int)sizeof(T);
    if constexpr (BYTES >= 4) {
        if (vec) {
            constexpr int NW = BYTES / 4;
            uint32_t w[NW];
#pragma unroll
            for (int k = 0; k < NW; ++k) {
                if constexpr (sizeof(T) == 4)
                    w[k] = bits_of<DT>(res[k]);  // the bits, not the value (T may be float)
                else
                    w[k] = bits_of<DT>(res[2 * k]) | (bits_of<DT>(res[2 * k + 1]) << 16);
            }
            uint32_t *ow = reinterpret_cast<uint32_t *>(o);
            if constexpr (NW == 1) {
                ow[0] = w[0];
            } else if constexpr (NW == 2) {
                *reinterpret_cast<uint2 *>(ow) = make_uint2(w[0], w[1]);
            } else {
#pragma unroll
                for (int k = 0; k < NW; k += 4)
                    *reinterpret_cast<uint4 *>(ow + k) = make_uint4(w[k], w[k + 1], w[k + 2], w[k + 3]);
            }
            return;
        }
    }
#pragma unroll
    for (int q = 0; q < RPB; ++q)
        o[q] = res[q];
}

// Rows of NE elements where one row is 32 / RPB bytes (RPB = 1, 2, 4, 8 or
// 16 rows per 32-byte block) and x is 32-byte aligned: each thread loads
// whole blocks (TY_U in flight, grid-stride) and folds the RPB rows of each
// from registers, in element order, accum first as in the row kernel; the
// RPB results are written together.  The last rows - RPB * (rows / RPB)
// rows (fewer than one block) go one per thread.
template <int OP, int DT, int NE>
__global__ void __launch_bounds__(TY_NT)
typed_tiny_kernel(const typename Elem<DT>::T *__restrict__ x, int64_t rows, int accum,
                  typename Elem<DT>::T *__restrict__ out)
{
    pdl_enter();
    using E = Elem<DT>;
    using T = typename E::T;
    using A = typename E::A;
    using K = Comb<OP, A>;
    constexpr int RPB = epb<DT>() / NE;
    static_assert(RPB * NE == epb<DT>() && RPB >= 1, "row size divides a block");
    constexpr int OB = RPB * (int)sizeof(T);  // result bytes per block
    const bool vec = ((uintptr_t)out & (uintptr_t)((OB < 16 ? OB : 16) - 1)) == 0;
    const int64_t nblk = rows / RPB;
    const int64_t tid = (int64_t)blockIdx.x * TY_NT + threadIdx.x;
    const int64_t nth = (int64_t)gridDim.x * TY_NT;
    for (int64_t c0 = tid; c0 < nblk; c0 += (int64_t)TY_U * nth) {
        uint32_t w[TY_U][8];  // all loads out before any fold
#pragma unroll
        for (int u = 0; u < TY_U; ++u)
            if (c0 + u * nth < nblk)
                ld8u(reinterpret_cast<const uint32_t *>(x + (c0 + u * nth) * epb<DT>()), w[u]);
#pragma unroll
        for (int u = 0; u < TY_U; ++u)
            if (c0 + u * nth < nblk) {
                T *o = out + (c0 + u * nth) * RPB;
                T res[RPB];
#pragma unroll
                for (int q = 0; q < RPB; ++q) {
                    A acc = K::identity();
#pragma unroll
                    for (int j = 0; j < NE; ++j)
                        acc = K::op(acc, block_elem<DT>(w[u], q * NE + j));
                    if (accum)
                        acc = K::op(E::widen(bits_of<DT>(o[q])), acc);
                    res[q] = E::narrow(acc);
                }
                store_results<DT, RPB>(o, res, vec);
            }
    }
    const int64_t r = nblk * RPB + tid;
    if (r < rows) {
        A acc = K::identity();
#pragma unroll
        for (int j = 0; j < NE; ++j)
            acc = K::op(acc, E::widen(load_bits<DT>(x + r * NE + j)));
        if (accum)
            acc = K::op(E::widen(bits_of<DT>(out[r])), acc);
        out[r] = E::narrow(acc);
    }
}

// Rows of RB whole 32-byte blocks (RB = 2, 4 or 8: 64 to 256 bytes) from a
// 32-byte aligned base: the matrix is one run of rows * RB blocks
// read grid-stride, TY_U blocks in flight per thread, so that consecutive
// lanes read consecutive blocks (every warp load is 1 KB contiguous) and the
// RB blocks of a row sit in RB consecutive lanes (the warp's first block
// index is a multiple of 32, hence of RB).  Each lane folds its block, the RB
// lanes of a row meet in a butterfly, and the row's first lane folds the
// accum value in and writes the result.
template <int OP, int DT, int RB>
__global__ void __launch_bounds__(TY_NT)
typed_blockrows_kernel(const typename Elem<DT>::T *__restrict__ x, int64_t rows, int accum,
                       typename Elem<DT>::T *__restrict__ out)
{
    pdl_enter();
    using E = Elem<DT>;
    using A = typename E::A;
    using K = Comb<OP, A>;
    static_assert(RB == 2 || RB == 4 || RB == 8, "blocks per row");
    const int lane = threadIdx.x & 31;
    const int64_t nblk = rows * RB;
    const int64_t tid = (int64_t)blockIdx.x * TY_NT + threadIdx.x;
    const int64_t nth = (int64_t)gridDim.x * TY_NT;
    for (int64_t c0 = tid; c0 - lane < nblk; c0 += (int64_t)TY_U * nth) {  // warp-uniform
        uint32_t w[TY_U][8];  // all loads out before any fold
#pragma unroll
        for (int u = 0; u < TY_U; ++u)
            if (c0 + u * nth < nblk)
                ld8u(reinterpret_cast<const uint32_t *>(x + (c0 + u * nth) * epb<DT>()), w[u]);
#pragma unroll
        for (int u = 0; u < TY_U; ++u) {
            const int64_t b = c0 + u * nth;
            A acc = K::identity();
            if (b < nblk)
#pragma unroll
                for (int j = 0; j < epb<DT>(); ++j)
                    acc = K::op(acc, block_elem<DT>(w[u], j));
#pragma unroll
            for (int o = 1; o < RB; o <<= 1)
                acc = K::op(acc, __shfl_xor_sync(0xffffffffu, acc, o));
            if (b < nblk && (lane & (RB - 1)) == 0) {
                const int64_t r = b / RB;
                if (accum)
                    acc = K::op(E::widen(bits_of<DT>(out[r])), acc);
                out[r] = E::narrow(acc);
            }
        }
    }
}

template <int OP, int DT, int RB>
int launch_blockrows(const typename Elem<DT>::T *x, int64_t rows, int accum, typename Elem<DT>::T *out, cudaStream_t s,
                     int sms)
{
    static std::atomic<int> occ_cache{0};
    const int occ = cached_occupancy(occ_cache, (const void *)typed_blockrows_kernel<OP, DT, RB>, TY_NT);
    if (occ <= 0)
        return fail(RED_ECUDA, "red_rows_typed: kernel cannot be resident on this device");
    const int64_t need = (rows * RB + (int64_t)TY_NT * TY_U - 1) / ((int64_t)TY_NT * TY_U);
    int64_t ctas = (int64_t)sms * occ;
    if (need < ctas)
        ctas = need;
    if (ctas < 1)
        ctas = 1;
    const cudaError_t e =
        launch_pdl(typed_blockrows_kernel<OP, DT, RB>, dim3((unsigned)ctas), dim3(TY_NT), s, x, rows, accum, out);
    count_launches(1);
    return cuda_fail(e != cudaSuccess ? e : cudaGetLastError(), "red_rows_typed launch");
}

template <int OP, int DT, int NE>
int launch_tiny(const typename Elem<DT>::T *x, int64_t rows, int accum, typename Elem<DT>::T *out, cudaStream_t s,
                int sms)
{
    if constexpr (NE > epb<DT>()) {
        return fail(RED_EINVAL, "red_rows_typed: row longer than a block");
    } else {
        static std::atomic<int> occ_cache{0};
        const int occ = cached_occupancy(occ_cache, (const void *)typed_tiny_kernel<OP, DT, NE>, TY_NT);
        if (occ <= 0)
            return fail(RED_ECUDA, "red_rows_typed: kernel cannot be resident on this device");
        constexpr int RPB = epb<DT>() / NE;
        const int64_t need = (rows / RPB + (int64_t)TY_NT * TY_U - 1) / ((int64_t)TY_NT * TY_U) + 1;
        int64_t ctas = (int64_t)sms * occ;
        if (need < ctas)
            ctas = need;
        const cudaError_t e =
            launch_pdl(typed_tiny_kernel<OP, DT, NE>, dim3((unsigned)ctas), dim3(TY_NT), s, x, rows, accum, out);
        count_launches(1);
        return cuda_fail(e != cudaSuccess ? e : cudaGetLastError(), "red_rows_typed launch");
    }
}

template <int OP, int DT>
int typed_tiny_dt(const typename Elem<DT>::T *x, int64_t rows, int len, int accum, typename Elem<DT>::T *out,
                  cudaStream_t s, int sms)
{
    if (len > epb<DT>()) {  // whole blocks per row
        switch (len / epb<DT>()) {
        case 2: return launch_blockrows<OP, DT, 2>(x, rows, accum, out, s, sms);
        case 4: return launch_blockrows<OP, DT, 4>(x, rows, accum, out, s, sms);
        default: return launch_blockrows<OP, DT, 8>(x, rows, accum, out, s, sms);
        }
    }
    switch (len) {
    case 1: return launch_tiny<OP, DT, 1>(x, rows, accum, out, s, sms);
    case 2: return launch_tiny<OP, DT, 2>(x, rows, accum, out, s, sms);
    case 4: return launch_tiny<OP, DT, 4>(x, rows, accum, out, s, sms);
    case 8: return launch_tiny<OP, DT, 8>(x, rows, accum, out, s, sms);
    default: return launch_tiny<OP, DT, 16>(x, rows, accum, out, s, sms);
    }
}

template <int OP>
int tiny_op(int dtype, const void *x, int64_t rows, int len, int accum, void *out, cudaStream_t s, int sms)
{
#define RED_TINY_CASE(DT)                                                                                     \
    case DT:                                                                                                   \
        return typed_tiny_dt<OP, DT>(static_cast<const typename Elem<DT>::T *>(x), rows, len, accum,            \
                                     static_cast<typename Elem<DT>::T *>(out), s, sms);
    switch (dtype) {
        RED_TINY_CASE(RED_F32)
        RED_TINY_CASE(RED_I32)
        RED_TINY_CASE(RED_F16)
        RED_TINY_CASE(RED_BF16)
        RED_TINY_CASE(RED_I16)
        RED_TINY_CASE(RED_U16)
        RED_TINY_CASE(RED_U32)
    default: return fail(RED_EINVAL, "red_rows_typed: unknown dtype %d", dtype);
    }
#undef RED_TINY_CASE
}

}  // namespace

int launch_typed_tiny(int op, int dtype, const void *x, int64_t rows, int len, int accum, void *out, cudaStream_t s,
                      int sms)
{
    switch (op) {
    case RED_SUM: return tiny_op<RED_SUM>(dtype, x, rows, len, accum, out, s, sms);
    case RED_MAX: return tiny_op<RED_MAX>(dtype, x, rows, len, accum, out, s, sms);
    case RED_MIN: return tiny_op<RED_MIN>(dtype, x, rows, len, accum, out, s, sms);
    default: return tiny_op<RED_PROD>(dtype, x, rows, len, accum, out, s, sms);
    }
}

}  // namespace red
