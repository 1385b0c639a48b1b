// red_device.cuh -- thread-scope reductions of a register-resident fp32
// vector, for use inside CUDA kernels on Blackwell (sm_100 and later; this
// library builds it for sm_103a).  Header-only; include it from .cu files.
//
// This is the granularity of Apache TVM docs, "reduction -> sm100_packed":
// one thread reduces a local 1-D float32 array of static length N to a
// scalar, with an optional accum that folds an old destination value in
// ("Demonstration program": Tx.sum(dst, src, accum); "How inputs change the
// algorithm").  The folds follow that page's "Algorithm":
//
//   red_dev::thread_sum<N>(a, accum, dst)   N >= 8: an 8-wide accumulator
//       loaded from a[0..8); with accum, dst is added into its first slot;
//       every further full chunk of 8 is added with four packed
//       add.rn.ftz.f32x2; a remainder of r < 8 elements is added one at a
//       time into slots 0..r-1; the accumulator then collapses 8 -> 4 -> 2
//       -> 1 (collapse8: three packed adds and one scalar add).  N < 8
//       (below the page's dispatch gate): a left-to-right scalar fold.  The rounding
//       order is therefore fixed by N alone: the same a gives the same bits
//       on every launch configuration.
//   red_dev::thread_max<N>, thread_min<N>  a 4-wide accumulator loaded from
//       a[0..4); each three-input max.f32 / min.f32 folds one slot with two
//       new values; remainder one at a time; exact in any order.
//
// Scalar steps are IEEE round-to-nearest additions (__fadd_rn); the packed
// adds flush denormal results to zero, as the page's add.rn.ftz.f32x2 does.
#pragma once

#include <cuda_runtime.h>

namespace red_dev {

// Packed pairwise add of two fp32 lanes: add.rn.ftz.f32x2.
__device__ __forceinline__ float2 add_f32x2(float2 a, float2 b)
{
    float2 d;
    asm("{\n\t.reg .b64 pa, pb, pd;\n\t"
        "mov.b64 pa, {%2, %3};\n\t"
        "mov.b64 pb, {%4, %5};\n\t"
        "add.rn.ftz.f32x2 pd, pa, pb;\n\t"
        "mov.b64 {%0, %1}, pd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

// The collapse of an 8-wide packed accumulator (four float2 slots) to one
// float: a pairwise tree over the slots, each level adding slot k + h into
// slot k for h = 1, then 2 (the pairing the page's "Algorithm" prescribes:
// lanes (0,1) gain (2,3) and (4,5) gain (6,7), then (0,1) gains (4,5)), and
// a final scalar add of the two lanes left: round-to-nearest, or with FTZ
// also flushing a denormal result to zero (add.rn.ftz.f32).
template <bool FTZ = false>
__device__ __forceinline__ float collapse8(float2 (&s)[4])
{
#pragma unroll
    for (int h = 1; h < 4; h *= 2)
#pragma unroll
        for (int k = 0; k < 4; k += 2 * h)
            s[k] = add_f32x2(s[k], s[k + h]);
    if constexpr (FTZ) {
        float d;
        asm("add.rn.ftz.f32 %0, %1, %2;" : "=f"(d) : "f"(s[0].x), "f"(s[0].y));
        return d;
    } else {
        return __fadd_rn(s[0].x, s[0].y);
    }
}

// Three-input max / min (the max3.f32 / min3.f32 of the page).
__device__ __forceinline__ float max3(float a, float b, float c)
{
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

__device__ __forceinline__ float min3(float a, float b, float c)
{
    float d;
    asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

template <int N>
__device__ __forceinline__ float thread_sum(const float (&a)[N], bool accum = false, float dst = 0.0f)
{
    static_assert(N >= 1, "thread_sum needs at least one element");
    if constexpr (N < 8) {
        float r = a[0];
        if (accum)
            r = __fadd_rn(r, dst);
#pragma unroll
        for (int i = 1; i < N; ++i)
            r = __fadd_rn(r, a[i]);
        return r;
    } else {
        float2 s[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
            s[k] = make_float2(a[2 * k], a[2 * k + 1]);
        if (accum)
            s[0].x = __fadd_rn(s[0].x, dst);
        constexpr int FULL = N / 8 * 8;  // elements in full chunks
#pragma unroll
        for (int c = 8; c < FULL; c += 8)
#pragma unroll
            for (int k = 0; k < 4; ++k)
                s[k] = add_f32x2(s[k], make_float2(a[c + 2 * k], a[c + 2 * k + 1]));
#pragma unroll
        for (int i = FULL; i < N; ++i) {  // remainder: element FULL + j into slot j
            const int j = i - FULL;
            if (j & 1)
                s[j >> 1].y = __fadd_rn(s[j >> 1].y, a[i]);
            else
                s[j >> 1].x = __fadd_rn(s[j >> 1].x, a[i]);
        }
        return collapse8(s);
    }
}

namespace detail {

template <bool MAX, int N>
__device__ __forceinline__ float thread_extreme(const float (&a)[N], bool accum, float dst)
{
    auto two = [](float x, float y) { return MAX ? fmaxf(x, y) : fminf(x, y); };
    auto three = [](float x, float y, float z) { return MAX ? max3(x, y, z) : min3(x, y, z); };
    if constexpr (N < 4) {
        float r = a[0];
        if (accum)
            r = two(r, dst);
#pragma unroll
        for (int i = 1; i < N; ++i)
            r = two(r, a[i]);
        return r;
    } else {
        float m[4] = {a[0], a[1], a[2], a[3]};
        if (accum)
            m[0] = two(m[0], dst);
        constexpr int FULL = 4 + (N - 4) / 8 * 8;
#pragma unroll
        for (int c = 4; c < FULL; c += 8)
#pragma unroll
            for (int k = 0; k < 4; ++k)
                m[k] = three(m[k], a[c + 2 * k], a[c + 2 * k + 1]);
#pragma unroll
        for (int i = FULL; i < N; ++i)
            m[(i - FULL) & 3] = two(m[(i - FULL) & 3], a[i]);
        return two(three(m[0], m[1], m[2]), m[3]);
    }
}

}  // namespace detail

template <int N>
__device__ __forceinline__ float thread_max(const float (&a)[N], bool accum = false, float dst = 0.0f)
{
    return detail::thread_extreme<true, N>(a, accum, dst);
}

template <int N>
__device__ __forceinline__ float thread_min(const float (&a)[N], bool accum = false, float dst = 0.0f)
{
    return detail::thread_extreme<false, N>(a, accum, dst);
}

}  // namespace red_dev
