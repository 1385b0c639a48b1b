// red_colprod.cu -- TCOLPROD column products (pto-isa docs, "TCOLPROD",
// "Math Interpretation": dst[0,j] = prod_{i=0}^{R-1} src[i,j]) for fp32
// (round-to-nearest products) and int32 (products wrap modulo 2^32, done in
// uint32).
//
// Layout of the work: a CTA owns a tile of 32*V adjacent columns and WY warps.
// Lane l of every warp owns columns [32*V*tile + V*l, +V) and keeps V running
// products (per-thread column accumulators); warp w of the CTA walks rows
// i0+w, i0+w+WY, ... of the CTA's row slab, so each warp reads 32*V*4
// contiguous bytes of a row per load (coalesced, row-major order kept).  The
// WY warp products meet in shared memory (fixed order).  gridDim.y CTAs split
// the rows; with more than one, the CTA partials go to the workspace and the
// CTA that arrives last for its column tile multiplies them (in split order)
// into dst.  No CTA ever waits for another.
#include "red_internal.h"
#include "red_prims.cuh"
#include "red.h"

namespace red {
namespace {

constexpr int CP_WY = 16;                // warps per CTA (row interleave)
constexpr int CP_NT = 32 * CP_WY;
constexpr int CP_U = 4;                  // loads in flight per thread

__device__ __forceinline__ float mul(float a, float b) { return __fmul_rn(a, b); }
__device__ __forceinline__ uint32_t mul(uint32_t a, uint32_t b) { return a * b; }

template <typename T>
__device__ __forceinline__ T from_bits(uint32_t w);
template <>
__device__ __forceinline__ float from_bits<float>(uint32_t w) { return __uint_as_float(w); }
template <>
__device__ __forceinline__ uint32_t from_bits<uint32_t>(uint32_t w) { return w; }

template <typename T>
__device__ __forceinline__ T one();
template <>
__device__ __forceinline__ float one<float>() { return 1.0f; }
template <>
__device__ __forceinline__ uint32_t one<uint32_t>() { return 1u; }

// V consecutive elements at p (V = 8: 32-byte aligned, V = 4: 16-byte
// aligned, V = 1: any).
template <typename T, int V>
__device__ __forceinline__ void ldv(const T *p, T (&v)[V])
{
    if constexpr (V == 8) {
        uint32_t w[8];
        ld8u(reinterpret_cast<const uint32_t *>(p), w);
#pragma unroll
        for (int k = 0; k < 8; ++k)
            v[k] = from_bits<T>(w[k]);
    } else if constexpr (V == 4) {
        uint32_t w[4];
        ld4u(reinterpret_cast<const uint32_t *>(p), w);
#pragma unroll
        for (int k = 0; k < 4; ++k)
            v[k] = from_bits<T>(w[k]);
    } else {
        v[0] = __ldg(p);
    }
}

template <typename T, int V>
__global__ void __launch_bounds__(CP_NT)
colprod_kernel(const T *__restrict__ x, int64_t R, int64_t C, int64_t rows_per_split,
               T *__restrict__ part, unsigned *__restrict__ tick, T *__restrict__ out)
{
    __shared__ T s_p[CP_WY][32 * V];
    __shared__ int s_last;

    const int lane = threadIdx.x & 31, wy = threadIdx.x >> 5;
    const int64_t col = ((int64_t)blockIdx.x * 32 + lane) * V;
    const bool live = col < C;  // V > 1 only when C % V == 0
    const int64_t i0 = (int64_t)blockIdx.y * rows_per_split;
    const int64_t i1 = (i0 + rows_per_split < R) ? i0 + rows_per_split : R;

    T p[V];
#pragma unroll
    for (int k = 0; k < V; ++k)
        p[k] = one<T>();
    if (live) {
        const T *q = x + col;
        int64_t i = i0 + wy;
        for (; i + (CP_U - 1) * CP_WY < i1; i += CP_U * CP_WY) {
            T v[CP_U][V];
#pragma unroll
            for (int u = 0; u < CP_U; ++u)
                ldv<T, V>(q + (i + u * CP_WY) * C, v[u]);
#pragma unroll
            for (int u = 0; u < CP_U; ++u)
#pragma unroll
                for (int k = 0; k < V; ++k)
                    p[k] = mul(p[k], v[u][k]);
        }
        for (; i < i1; i += CP_WY) {
            T v[V];
            ldv<T, V>(q + i * C, v);
#pragma unroll
            for (int k = 0; k < V; ++k)
                p[k] = mul(p[k], v[k]);
        }
    }
#pragma unroll
    for (int k = 0; k < V; ++k)
        s_p[wy][lane * V + k] = p[k];
    __syncthreads();
    if (wy == 0) {
#pragma unroll
        for (int w = 1; w < CP_WY; ++w)
#pragma unroll
            for (int k = 0; k < V; ++k)
                p[k] = mul(p[k], s_p[w][lane * V + k]);
    }

    if (gridDim.y == 1) {
        if (wy == 0 && live)
#pragma unroll
            for (int k = 0; k < V; ++k)
                out[col + k] = p[k];
        return;
    }
    if (wy == 0 && live)
#pragma unroll
        for (int k = 0; k < V; ++k)
            part[(int64_t)blockIdx.y * C + col + k] = p[k];
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0)
        s_last = (atomicAdd(tick + blockIdx.x, 1u) == gridDim.y - 1);
    __syncthreads();
    if (!s_last)
        return;
    __threadfence();
    if (wy == 0 && live) {
        T q[V];
#pragma unroll
        for (int k = 0; k < V; ++k)
            q[k] = one<T>();
        for (unsigned sp = 0; sp < gridDim.y; ++sp)
#pragma unroll
            for (int k = 0; k < V; ++k)
                q[k] = mul(q[k], __ldcg(part + (int64_t)sp * C + col + k));
#pragma unroll
        for (int k = 0; k < V; ++k)
            out[col + k] = q[k];
    }
    if (threadIdx.x == 0)
        tick[blockIdx.x] = 0;
}

template <typename T, int V>
int launch_cp(const T *x, int64_t R, int64_t C, T *out, cudaStream_t s, const DeviceInfo &di)
{
    static int occ = 0;
    if (occ == 0)
        occ = occupancy((const void *)colprod_kernel<T, V>, CP_NT);
    if (occ <= 0)
        return fail(RED_ECUDA, "red_colprod: kernel cannot be resident on this device");
    const int64_t tile_cols = 32 * V;
    const int64_t tiles = (C + tile_cols - 1) / tile_cols;
    if (tiles > 0x7fffffffLL)
        return fail(RED_EINVAL, "red_colprod: C too large");
    // Row splits: each warp keeps at least CP_U rows; among those counts take
    // the smallest whose CTAs fill their waves of resident CTAs to at least
    // 90% (more splits add partial-product traffic and per-CTA overhead),
    // else the count with the best wave efficiency.
    int64_t splits = knob(RED_KNOB_COLPROD_SPLITS);
    if (splits <= 0) {
        const int64_t slots = (int64_t)di.sms * occ;
        int64_t smax = R / (CP_WY * CP_U);
        if (smax > 4096)
            smax = 4096;
        if (smax < 1)
            smax = 1;
        splits = 1;
        double best = -1.0;
        for (int64_t sp = 1; sp <= smax; ++sp) {
            const int64_t ctas = tiles * sp;
            const double eff = (double)ctas / (double)(((ctas + slots - 1) / slots) * slots);
            if (eff >= 0.9) {
                splits = sp;
                break;
            }
            if (eff > best) {
                best = eff;
                splits = sp;
            }
        }
    }
    if (splits > R)
        splits = R;
    if (splits > 65535)
        splits = 65535;
    if (splits * C > (int64_t)WS_PART_ELEMS)
        splits = (int64_t)WS_PART_ELEMS / C;
    if (tiles > WS_TICKETS)
        splits = 1;
    if (splits < 1)
        splits = 1;
    const int64_t rps = (R + splits - 1) / splits;
    splits = (R + rps - 1) / rps;  // no empty split
    Workspace ws;
    if (splits > 1) {
        const int st = get_workspace(&ws);
        if (st != RED_OK)
            return st;
    }
    const dim3 grid((unsigned)tiles, (unsigned)splits);
    colprod_kernel<T, V><<<grid, CP_NT, 0, s>>>(x, R, C, rps, static_cast<T *>(ws.part), ws.tick, out);
    count_launches(1);
    return cuda_fail(cudaGetLastError(), "red_colprod launch");
}

template <typename T>
int launch_cp_t(const void *xv, int64_t R, int64_t C, void *outv, cudaStream_t s, const DeviceInfo &di)
{
    const T *x = static_cast<const T *>(xv);
    T *out = static_cast<T *>(outv);
    const uintptr_t a = (uintptr_t)x;
    if (C % 8 == 0 && a % 32 == 0)
        return launch_cp<T, 8>(x, R, C, out, s, di);
    if (C % 4 == 0 && a % 16 == 0)
        return launch_cp<T, 4>(x, R, C, out, s, di);
    return launch_cp<T, 1>(x, R, C, out, s, di);
}

}  // namespace

int launch_colprod(int dtype, const void *x, int64_t R, int64_t C, void *out, cudaStream_t s)
{
    DeviceInfo di;
    const int st = device_info(&di);
    if (st != RED_OK)
        return st;
    if (dtype == RED_F32)
        return launch_cp_t<float>(x, R, C, out, s, di);
    return launch_cp_t<uint32_t>(x, R, C, out, s, di);
}

}  // namespace red
