// red_prims.cuh -- device building blocks of the reduction kernels (sm_103a).
//
// * Packed pairwise fp32 add, round-to-nearest, flush-to-zero: the
//   add.rn.ftz.f32x2 instruction of Blackwell, two float lanes per
//   instruction (Apache TVM docs, "reduction -> sm100_packed", sections
//   "Algorithm" and "Generated CUDA").
// * 3-input max / min (the max3 / min3 fold of the same page, "Algorithm":
//   a 4-wide accumulator folded three values at a time), written as the
//   three-operand max.f32 / min.f32 forms.
// * The per-thread fold: an 8-wide sum accumulator fed by chunks of 8
//   (four packed adds per chunk), the scalar remainder, and the final
//   8 -> 4 -> 2 -> 1 collapse; a 4-wide max / min accumulator.
// * Warp butterfly (__shfl_xor_sync) and the shared-memory CTA stage of the
//   block reduce in the Triton vector-accumulation blog post (imxueqiu.com),
//   C version: warp tree, lane 0 of each warp to shared memory, barrier,
//   second warp tree.
// * Streaming vector loads: 256-bit (8 x fp32), 128-bit and 64-bit,
//   read-only path, no L1 allocation (every byte is read once).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "red_device.cuh"

namespace red {

enum : int { OP_SUM = 0, OP_MAX = 1, OP_MIN = 2 };

// Programmatic dependent launch: allow the next kernel on the stream to be
// scheduled now, then wait until every kernel this one depends on has
// completed and its memory is visible.  Called first in a kernel, so that no
// global access precedes the wait; both are no-ops for a launch without the
// programmatic-serialization attribute.
__device__ __forceinline__ void pdl_enter()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ------------------------------------------------------------ packed math

// add.rn.ftz.f32x2 and the three-input max / min live in the public device
// header (the thread-scope API); the kernels use the same instructions.
__device__ __forceinline__ float2 add_f32x2(float2 a, float2 b) { return red_dev::add_f32x2(a, b); }
__device__ __forceinline__ float max3f(float a, float b, float c) { return red_dev::max3(a, b, c); }
__device__ __forceinline__ float min3f(float a, float b, float c) { return red_dev::min3(a, b, c); }

__device__ __forceinline__ float add_ftz(float a, float b)
{
    float d;
    asm("add.rn.ftz.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
    return d;
}

// --------------------------------------------------------------- loads

// 8 consecutive floats from a 32-byte aligned address.
__device__ __forceinline__ void ld8(const float *p, float (&v)[8])
{
    asm volatile("ld.global.nc.L1::no_allocate.v8.f32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]),
                   "=f"(v[4]), "=f"(v[5]), "=f"(v[6]), "=f"(v[7])
                 : "l"(p));
}

// 8 consecutive 32-bit words from a 32-byte aligned address.
__device__ __forceinline__ void ld8u(const uint32_t *p, uint32_t (&v)[8])
{
    asm volatile("ld.global.nc.L1::no_allocate.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]),
                   "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7])
                 : "l"(p));
}

// 4 consecutive 32-bit words from a 16-byte aligned address.
__device__ __forceinline__ void ld4u(const uint32_t *p, uint32_t (&v)[4])
{
    asm volatile("ld.global.nc.L1::no_allocate.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3])
                 : "l"(p));
}

// 4 (16-byte aligned) and 2 (8-byte aligned) consecutive floats.
__device__ __forceinline__ float4 ld4f(const float *p)
{
    float4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ float2 ld2f(const float *p)
{
    float2 v;
    asm volatile("ld.global.nc.L1::no_allocate.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "l"(p));
    return v;
}

__device__ __forceinline__ float ld1(const float *p) { return __ldg(p); }

// ------------------------------------------------------ operator traits

template <int OP>
struct Op;

template <>
struct Op<OP_SUM> {
    static __device__ __forceinline__ float identity() { return 0.0f; }
    static __device__ __forceinline__ float combine(float a, float b) { return add_ftz(a, b); }
};

template <>
struct Op<OP_MAX> {
    static __device__ __forceinline__ float identity() { return __int_as_float(0xff800000); }
    static __device__ __forceinline__ float combine(float a, float b) { return fmaxf(a, b); }
};

template <>
struct Op<OP_MIN> {
    static __device__ __forceinline__ float identity() { return __int_as_float(0x7f800000); }
    static __device__ __forceinline__ float combine(float a, float b) { return fminf(a, b); }
};

// ------------------------------------------------------ per-thread fold

template <int OP>
struct Fold;

// 8-wide fp32 accumulator.  chunk(): four packed adds fold 8 new values in;
// scalar(): remainder (and accum) values go into slot 0; finish(): the
// 8 -> 4 -> 2 -> 1 collapse with three packed adds and one scalar add.
template <>
struct Fold<OP_SUM> {
    float2 a[4];
    __device__ __forceinline__ void init()
    {
#pragma unroll
        for (int k = 0; k < 4; ++k)
            a[k] = make_float2(0.0f, 0.0f);
    }
    __device__ __forceinline__ void chunk(const float (&v)[8])
    {
#pragma unroll
        for (int k = 0; k < 4; ++k)
            a[k] = add_f32x2(a[k], make_float2(v[2 * k], v[2 * k + 1]));
    }
    __device__ __forceinline__ void scalar(float v) { a[0].x = add_ftz(a[0].x, v); }
    // pieces of a row's unaligned head or tail: 2 or 4 values
    __device__ __forceinline__ void pair(float2 v) { a[1] = add_f32x2(a[1], v); }
    __device__ __forceinline__ void quad(float4 v)
    {
        a[2] = add_f32x2(a[2], make_float2(v.x, v.y));
        a[3] = add_f32x2(a[3], make_float2(v.z, v.w));
    }
    __device__ __forceinline__ float finish() const
    {
        float2 s[4] = {a[0], a[1], a[2], a[3]};
        return red_dev::collapse8<true>(s);
    }
};

// 4-wide accumulator; each max3 folds one slot with two new values.
template <>
struct Fold<OP_MAX> {
    float m[4];
    __device__ __forceinline__ void init()
    {
#pragma unroll
        for (int k = 0; k < 4; ++k)
            m[k] = Op<OP_MAX>::identity();
    }
    __device__ __forceinline__ void chunk(const float (&v)[8])
    {
#pragma unroll
        for (int k = 0; k < 4; ++k)
            m[k] = max3f(m[k], v[2 * k], v[2 * k + 1]);
    }
    __device__ __forceinline__ void scalar(float v) { m[0] = fmaxf(m[0], v); }
    __device__ __forceinline__ void pair(float2 v) { m[1] = max3f(m[1], v.x, v.y); }
    __device__ __forceinline__ void quad(float4 v)
    {
        m[2] = max3f(m[2], v.x, v.y);
        m[3] = max3f(m[3], v.z, v.w);
    }
    __device__ __forceinline__ float finish() const { return fmaxf(max3f(m[0], m[1], m[2]), m[3]); }
};

template <>
struct Fold<OP_MIN> {
    float m[4];
    __device__ __forceinline__ void init()
    {
#pragma unroll
        for (int k = 0; k < 4; ++k)
            m[k] = Op<OP_MIN>::identity();
    }
    __device__ __forceinline__ void chunk(const float (&v)[8])
    {
#pragma unroll
        for (int k = 0; k < 4; ++k)
            m[k] = min3f(m[k], v[2 * k], v[2 * k + 1]);
    }
    __device__ __forceinline__ void scalar(float v) { m[0] = fminf(m[0], v); }
    __device__ __forceinline__ void pair(float2 v) { m[1] = min3f(m[1], v.x, v.y); }
    __device__ __forceinline__ void quad(float4 v)
    {
        m[2] = min3f(m[2], v.x, v.y);
        m[3] = min3f(m[3], v.z, v.w);
    }
    __device__ __forceinline__ float finish() const { return fminf(min3f(m[0], m[1], m[2]), m[3]); }
};

// --------------------------------------------------- warp and CTA stages

// Butterfly over groups of W consecutive lanes (W a power of two <= 32);
// every lane of the group ends with the group's result.  All 32 lanes of the
// warp must call it.
template <int OP, int W>
__device__ __forceinline__ float group_tree(float v)
{
#pragma unroll
    for (int off = W / 2; off > 0; off >>= 1)
        v = Op<OP>::combine(v, __shfl_xor_sync(0xffffffffu, v, off));
    return v;
}

// Smallest power of two >= v (v in 1..32).
__host__ __device__ constexpr int pow2ceil(int v) { return v <= 1 ? 1 : 2 * pow2ceil((v + 1) / 2); }

// CTA stage: warp butterfly, lane 0 of each warp to shared memory, barrier,
// warp 0 folds the NW warp results.  The result is valid in warp 0.  The
// caller must place a barrier between two uses of the same `s`.
template <int OP, int NW>
__device__ __forceinline__ float cta_reduce(float v, float *s)
{
    v = group_tree<OP, 32>(v);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0)
        s[warp] = v;
    __syncthreads();
    if (warp == 0) {
        v = lane < NW ? s[lane] : Op<OP>::identity();
        v = group_tree<OP, pow2ceil(NW)>(v);
    }
    return v;
}

// Number of leading elements of p to peel so that the rest is 32-byte
// aligned (0..7), capped at len.
__device__ __forceinline__ int64_t head_to_32B(const float *p, int64_t len)
{
    const int64_t h = (int64_t)(((32u - ((uint32_t)(uintptr_t)p & 31u)) & 31u) >> 2);
    return h < len ? h : len;
}

}  // namespace red
