// red_types.cuh -- element types and operators of the typed reductions
// (red_cols, red_full_typed, red_rows_typed): the element types of pto-isa
// docs, "TCOLPROD", "A2A3 / A5 implementation checks" (float, int32, half,
// bfloat16, int16, uint16, uint32), each widened to a 32-bit accumulator
// (fp32 for floating types, int32 / uint32 for integers) and narrowed back
// once at the end; and sum / max / min / product on those accumulators
// (floating sums and products round to nearest per step, integer sums and
// products wrap modulo 2^32, which the narrowing to 16 bits turns into the
// 16-bit wrap).
#pragma once

#include <cstdint>
#include <cstring>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "red.h"

namespace red {

// ------------------------------------------------------- element types

template <int DT>
struct Elem;

template <>
struct Elem<RED_F32> {
    using T = float;
    using A = float;
    static __device__ __forceinline__ A widen(uint32_t bits) { return __uint_as_float(bits); }
    static __device__ __forceinline__ T narrow(A a) { return a; }
};
template <>
struct Elem<RED_I32> {
    using T = int32_t;
    using A = int32_t;
    static __device__ __forceinline__ A widen(uint32_t bits) { return (int32_t)bits; }
    static __device__ __forceinline__ T narrow(A a) { return a; }
};
template <>
struct Elem<RED_U32> {
    using T = uint32_t;
    using A = uint32_t;
    static __device__ __forceinline__ A widen(uint32_t bits) { return bits; }
    static __device__ __forceinline__ T narrow(A a) { return a; }
};
template <>
struct Elem<RED_F16> {
    using T = uint16_t;  // binary16 bits
    using A = float;
    static __device__ __forceinline__ A widen(uint32_t bits)
    {
        return __half2float(__ushort_as_half((unsigned short)bits));
    }
    static __device__ __forceinline__ T narrow(A a) { return __half_as_ushort(__float2half_rn(a)); }
};
template <>
struct Elem<RED_BF16> {
    using T = uint16_t;  // bfloat16 bits
    using A = float;
    static __device__ __forceinline__ A widen(uint32_t bits) { return __uint_as_float(bits << 16); }
    static __device__ __forceinline__ T narrow(A a) { return __bfloat16_as_ushort(__float2bfloat16_rn(a)); }
};
template <>
struct Elem<RED_I16> {
    using T = int16_t;
    using A = int32_t;
    static __device__ __forceinline__ A widen(uint32_t bits) { return (int32_t)(int16_t)(uint16_t)bits; }
    static __device__ __forceinline__ T narrow(A a) { return (int16_t)(uint16_t)(uint32_t)a; }
};
template <>
struct Elem<RED_U16> {
    using T = uint16_t;
    using A = uint32_t;
    static __device__ __forceinline__ A widen(uint32_t bits) { return bits & 0xffffu; }
    static __device__ __forceinline__ T narrow(A a) { return (uint16_t)a; }
};

// ------------------------------------------------------------ operators

template <int OP, typename A>
struct Comb;

template <int OP>
struct Comb<OP, float> {
    static __device__ __forceinline__ float identity()
    {
        return OP == RED_SUM ? 0.0f
                             : OP == RED_PROD ? 1.0f
                                              : OP == RED_MAX ? __int_as_float(0xff800000) : __int_as_float(0x7f800000);
    }
    static __device__ __forceinline__ float op(float a, float b)
    {
        return OP == RED_SUM ? __fadd_rn(a, b) : OP == RED_PROD ? __fmul_rn(a, b) : OP == RED_MAX ? fmaxf(a, b) : fminf(a, b);
    }
};

template <int OP>
struct Comb<OP, int32_t> {
    static __device__ __forceinline__ int32_t identity()
    {
        return OP == RED_SUM ? 0 : OP == RED_PROD ? 1 : OP == RED_MAX ? INT32_MIN : INT32_MAX;
    }
    static __device__ __forceinline__ int32_t op(int32_t a, int32_t b)
    {
        if (OP == RED_SUM)
            return (int32_t)((uint32_t)a + (uint32_t)b);
        if (OP == RED_PROD)
            return (int32_t)((uint32_t)a * (uint32_t)b);
        return OP == RED_MAX ? (a > b ? a : b) : (a < b ? a : b);
    }
};

template <int OP>
struct Comb<OP, uint32_t> {
    static __device__ __forceinline__ uint32_t identity()
    {
        return OP == RED_SUM ? 0u : OP == RED_PROD ? 1u : OP == RED_MAX ? 0u : 0xffffffffu;
    }
    static __device__ __forceinline__ uint32_t op(uint32_t a, uint32_t b)
    {
        if (OP == RED_SUM)
            return a + b;
        if (OP == RED_PROD)
            return a * b;
        return OP == RED_MAX ? (a > b ? a : b) : (a < b ? a : b);
    }
};

template <typename A>
__device__ __forceinline__ A ldcg_a(const A *p);
template <>
__device__ __forceinline__ float ldcg_a<float>(const float *p) { return __ldcg(p); }
template <>
__device__ __forceinline__ int32_t ldcg_a<int32_t>(const int32_t *p) { return __ldcg(p); }
template <>
__device__ __forceinline__ uint32_t ldcg_a<uint32_t>(const uint32_t *p) { return __ldcg(p); }

// One element's bits through the read-only path (zero-extended for 16-bit
// types), ready for Elem<DT>::widen.
template <int DT>
__device__ __forceinline__ uint32_t load_bits(const typename Elem<DT>::T *p)
{
    if constexpr (sizeof(typename Elem<DT>::T) == 4)
        return __ldg(reinterpret_cast<const unsigned int *>(p));
    else
        return __ldg(reinterpret_cast<const unsigned short *>(p));
}

// The bits of an element value, for the accum operand read from out.
template <int DT>
__device__ __forceinline__ uint32_t bits_of(typename Elem<DT>::T v)
{
    if constexpr (sizeof(typename Elem<DT>::T) == 4) {
        uint32_t b;
        memcpy(&b, &v, 4);
        return b;
    } else {
        uint16_t b;
        memcpy(&b, &v, 2);
        return b;
    }
}

}  // namespace red
