// red_stats.cu -- sum, max, min and sum |x| of one fp32 vector, or of every
// row of a row-major matrix, from a single read (separate calls read the
// data once per statistic).
//
// Same streaming structure as red_full's kernel: grid-stride 256-bit loads,
// 4 chunks of 8 in flight per thread, an unaligned head and the tail folded
// one at a time.  Each thread keeps the accumulators of Apache TVM docs,
// "reduction -> sm100_packed", "Algorithm" side by side: the 8-wide packed
// add.f32x2 sum (also for |x|) and the 4-wide max3 / min3 accumulators.  The
// CTA stage is the warp butterfly plus a shared-memory stage of the block
// reduce in the Triton vector-accumulation blog post, for each of the four
// statistics; the grid stage is last-block (partials in the workspace, the
// CTA that arrives last folds them; no CTA waits for another).
#include "red_internal.h"
#include "red_prims.cuh"
#include "red.h"

namespace red {
namespace {

constexpr int ST_NT = 512;
constexpr int ST_U = 4;
constexpr int ST_NW = ST_NT / 32;

struct Stats4 {
    Fold<OP_SUM> sum, asum;
    Fold<OP_MAX> mx;
    Fold<OP_MIN> mn;
    __device__ __forceinline__ void init()
    {
        sum.init();
        asum.init();
        mx.init();
        mn.init();
    }
    __device__ __forceinline__ void chunk(const float (&v)[8])
    {
        float a[8];
#pragma unroll
        for (int k = 0; k < 8; ++k)
            a[k] = fabsf(v[k]);
        sum.chunk(v);
        asum.chunk(a);
        mx.chunk(v);
        mn.chunk(v);
    }
    __device__ __forceinline__ void scalar(float v)
    {
        sum.scalar(v);
        asum.scalar(fabsf(v));
        mx.scalar(v);
        mn.scalar(v);
    }
    __device__ __forceinline__ void pair(float2 v)
    {
        sum.pair(v);
        asum.pair(make_float2(fabsf(v.x), fabsf(v.y)));
        mx.pair(v);
        mn.pair(v);
    }
    __device__ __forceinline__ void quad(float4 v)
    {
        sum.quad(v);
        asum.quad(make_float4(fabsf(v.x), fabsf(v.y), fabsf(v.z), fabsf(v.w)));
        mx.quad(v);
        mn.quad(v);
    }
};

// Reduce four values over the CTA; the results are valid in warp 0.
__device__ __forceinline__ void cta_reduce4(float &s, float &a, float &m, float &n, float (*sh)[ST_NW])
{
    s = group_tree<OP_SUM, 32>(s);
    a = group_tree<OP_SUM, 32>(a);
    m = group_tree<OP_MAX, 32>(m);
    n = group_tree<OP_MIN, 32>(n);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) {
        sh[0][warp] = s;
        sh[1][warp] = a;
        sh[2][warp] = m;
        sh[3][warp] = n;
    }
    __syncthreads();
    if (warp == 0) {
        const bool in = lane < ST_NW;
        s = group_tree<OP_SUM, pow2ceil(ST_NW)>(in ? sh[0][lane] : 0.0f);
        a = group_tree<OP_SUM, pow2ceil(ST_NW)>(in ? sh[1][lane] : 0.0f);
        m = group_tree<OP_MAX, pow2ceil(ST_NW)>(in ? sh[2][lane] : Op<OP_MAX>::identity());
        n = group_tree<OP_MIN, pow2ceil(ST_NW)>(in ? sh[3][lane] : Op<OP_MIN>::identity());
    }
}

// part: 4 * gridDim.x partials (sum, |x| sum, max, min per CTA); tick: one
// arrival counter; out: sum, max, min, sum |x|.
__global__ void __launch_bounds__(ST_NT, 2)
stats_kernel(const float *__restrict__ x, int64_t n, float *__restrict__ part, unsigned *__restrict__ tick,
             float *__restrict__ out)
{
    __shared__ float sh[4][ST_NW];
    pdl_enter();
    __shared__ int s_last;
    const int64_t h = head_to_32B(x, n);
    const int64_t nch = (n - h) >> 3;
    const int64_t t0 = h + (nch << 3);
    const int64_t tid = (int64_t)blockIdx.x * ST_NT + threadIdx.x;
    const int64_t nth = (int64_t)gridDim.x * ST_NT;
    const float *pa = x + h;

    Stats4 st;
    st.init();
    int64_t c = tid;
    for (; c + (ST_U - 1) * nth < nch; c += ST_U * nth) {
        float v[ST_U][8];
#pragma unroll
        for (int u = 0; u < ST_U; ++u)
            ld8(pa + 8 * (c + u * nth), v[u]);
#pragma unroll
        for (int u = 0; u < ST_U; ++u)
            st.chunk(v[u]);
    }
    for (; c < nch; c += nth) {
        float v[8];
        ld8(pa + 8 * c, v);
        st.chunk(v);
    }
    if (tid < h)
        st.scalar(ld1(x + tid));
    if (tid < n - t0)
        st.scalar(ld1(x + t0 + tid));

    float s = st.sum.finish(), a = st.asum.finish(), m = st.mx.finish(), mn = st.mn.finish();
    cta_reduce4(s, a, m, mn, sh);
    if (gridDim.x == 1) {
        if (threadIdx.x == 0) {
            out[0] = s;
            out[1] = m;
            out[2] = mn;
            out[3] = a;
        }
        return;
    }
    const unsigned G = gridDim.x;
    if (threadIdx.x == 0) {
        part[blockIdx.x] = s;
        part[G + blockIdx.x] = a;
        part[2 * G + blockIdx.x] = m;
        part[3 * G + blockIdx.x] = mn;
        __threadfence();
        s_last = (atomicAdd(tick, 1u) == G - 1);
    }
    __syncthreads();
    if (!s_last)
        return;
    __threadfence();
    float ws = 0.0f, wa = 0.0f, wm = Op<OP_MAX>::identity(), wn = Op<OP_MIN>::identity();
    for (unsigned i = threadIdx.x; i < G; i += ST_NT) {
        ws = Op<OP_SUM>::combine(ws, __ldcg(part + i));
        wa = Op<OP_SUM>::combine(wa, __ldcg(part + G + i));
        wm = fmaxf(wm, __ldcg(part + 2 * G + i));
        wn = fminf(wn, __ldcg(part + 3 * G + i));
    }
    cta_reduce4(ws, wa, wm, wn, sh);
    if (threadIdx.x == 0) {
        out[0] = ws;
        out[1] = wm;
        out[2] = wn;
        out[3] = wa;
        *tick = 0;
    }
}

// Per-row statistics: a group of G lanes per row, the row read as its
// 32-byte aligned interior in 256-bit blocks spread over the lanes (4 in
// flight per lane) plus its unaligned head and tail as naturally aligned
// 1-, 2- and 4-float pieces (lane 0 and the last lane), all four folds fed
// from the one read; out[4r .. 4r+4) = sum, max, min, sum |x|.
constexpr int SR_NT = 256;
constexpr int SR_U = 4;

template <int G>
__global__ void __launch_bounds__(SR_NT)
rows_stats_kernel(const float *__restrict__ x, int64_t rows, int64_t len, float *__restrict__ out)
{
    pdl_enter();
    constexpr int GPW = 32 / G;
    const int lane = threadIdx.x & 31, gl = lane & (G - 1), gw = lane / G;
    const int64_t warp = ((int64_t)blockIdx.x * SR_NT + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * SR_NT) >> 5;
    const int64_t x_mis = (int64_t)(((uintptr_t)x & 31u) >> 2);
    for (int64_t r0 = warp * GPW; r0 < rows; r0 += nwarps * GPW) {  // warp-uniform
        const int64_t r = r0 + gw;
        const bool live = r < rows;
        Stats4 st;
        st.init();
        if (live) {
            const int64_t b = r * len, e = b + len;
            const int64_t a = ((b + x_mis + 7) & ~int64_t(7)) - x_mis;
            const int64_t z = ((e + x_mis) & ~int64_t(7)) - x_mis;
            if (a <= z) {
                if (gl == 0) {
                    const int h = (int)(a - b);
                    const float *ph = x + b;
                    if (h & 1)
                        st.scalar(ld1(ph));
                    if (h & 2)
                        st.pair(ld2f(ph + (h & 1)));
                    if (h & 4)
                        st.quad(ld4f(ph + (h & 3)));
                }
                if (gl == G - 1) {
                    const int t = (int)(e - z);
                    const float *pt = x + z;
                    if (t & 4)
                        st.quad(ld4f(pt));
                    if (t & 2)
                        st.pair(ld2f(pt + (t & 4)));
                    if (t & 1)
                        st.scalar(ld1(pt + (t & 6)));
                }
                const int64_t nfull = (z - a) >> 3;
                const float *q = x + a;
                for (int64_t c0 = gl; c0 < nfull; c0 += (int64_t)SR_U * G) {
                    float v[SR_U][8];
#pragma unroll
                    for (int u = 0; u < SR_U; ++u)
                        if (c0 + u * G < nfull)
                            ld8(q + 8 * (c0 + u * G), v[u]);
#pragma unroll
                    for (int u = 0; u < SR_U; ++u)
                        if (c0 + u * G < nfull)
                            st.chunk(v[u]);
                }
            } else {
                // the row inside one 32-byte block (fewer than 8 floats):
                // every load of the lane out before any fold
                constexpr int KMAX = (7 + G - 1) / G;
                float t[KMAX];
#pragma unroll
                for (int k = 0; k < KMAX; ++k) {
                    const int64_t i = b + gl + (int64_t)k * G;
                    t[k] = i < e ? ld1(x + i) : 0.0f;
                }
#pragma unroll
                for (int k = 0; k < KMAX; ++k)
                    if (b + gl + (int64_t)k * G < e)
                        st.scalar(t[k]);
            }
        }
        const float s = group_tree<OP_SUM, G>(st.sum.finish());
        const float m = group_tree<OP_MAX, G>(st.mx.finish());
        const float n = group_tree<OP_MIN, G>(st.mn.finish());
        const float a = group_tree<OP_SUM, G>(st.asum.finish());
        if (live && gl == 0)
            *reinterpret_cast<float4 *>(out + 4 * r) = make_float4(s, m, n, a);
    }
}

// Rows of RB whole 32-byte blocks (RB = 2, 4 or 8: 16, 32 or 64 floats)
// from a 32-byte aligned base: the matrix read as one run of rows * RB
// blocks, grid-stride, SR_U blocks in flight per thread, consecutive lanes
// on consecutive blocks (every warp load 1 KB contiguous); a row's blocks
// sit in RB consecutive lanes (the warp's first block index is a multiple
// of 32), which meet in four butterflies; the row's first lane writes.
template <int RB>
__global__ void __launch_bounds__(SR_NT)
rows_stats_blocks_kernel(const float *__restrict__ x, int64_t rows, float *__restrict__ out)
{
    pdl_enter();
    static_assert(RB == 2 || RB == 4 || RB == 8, "blocks per row");
    const int lane = threadIdx.x & 31;
    const int64_t nblk = rows * RB;
    const int64_t tid = (int64_t)blockIdx.x * SR_NT + threadIdx.x;
    const int64_t nth = (int64_t)gridDim.x * SR_NT;
    for (int64_t c0 = tid; c0 - lane < nblk; c0 += (int64_t)SR_U * nth) {  // warp-uniform
        float v[SR_U][8];
#pragma unroll
        for (int u = 0; u < SR_U; ++u)
            if (c0 + u * nth < nblk)
                ld8(x + 8 * (c0 + u * nth), v[u]);
#pragma unroll
        for (int u = 0; u < SR_U; ++u) {
            const int64_t b = c0 + u * nth;
            Stats4 st;
            st.init();
            if (b < nblk)
                st.chunk(v[u]);
            const float s = group_tree<OP_SUM, RB>(st.sum.finish());
            const float m = group_tree<OP_MAX, RB>(st.mx.finish());
            const float n = group_tree<OP_MIN, RB>(st.mn.finish());
            const float a = group_tree<OP_SUM, RB>(st.asum.finish());
            if (b < nblk && (lane & (RB - 1)) == 0)
                *reinterpret_cast<float4 *>(out + 4 * (b / RB)) = make_float4(s, m, n, a);
        }
    }
}

template <int RB>
int launch_rows_stats_blocks(const float *x, int64_t rows, float *out, cudaStream_t s, int sms)
{
    static std::atomic<int> occ_cache{0};
    const int occ = cached_occupancy(occ_cache, (const void *)rows_stats_blocks_kernel<RB>, SR_NT);
    if (occ <= 0)
        return fail(RED_ECUDA, "red_rows_stats: kernel cannot be resident on this device");
    const int64_t need = (rows * RB + (int64_t)SR_NT * SR_U - 1) / ((int64_t)SR_NT * SR_U);
    int64_t ctas = (int64_t)sms * occ;
    if (need < ctas)
        ctas = need;
    if (ctas < 1)
        ctas = 1;
    const cudaError_t e = launch_pdl(rows_stats_blocks_kernel<RB>, dim3((unsigned)ctas), dim3(SR_NT), s, x, rows, out);
    count_launches(1);
    return cuda_fail(e != cudaSuccess ? e : cudaGetLastError(), "red_rows_stats launch");
}

template <int G>
int launch_rows_stats_g(const float *x, int64_t rows, int64_t len, float *out, cudaStream_t s, int sms)
{
    static std::atomic<int> occ_cache{0};
    const int occ = cached_occupancy(occ_cache, (const void *)rows_stats_kernel<G>, SR_NT);
    if (occ <= 0)
        return fail(RED_ECUDA, "red_rows_stats: kernel cannot be resident on this device");
    const int64_t rows_per_cta = (int64_t)(SR_NT / 32) * (32 / G);
    int64_t ctas = (rows + rows_per_cta - 1) / rows_per_cta;
    if (ctas > (int64_t)sms * occ)
        ctas = (int64_t)sms * occ;
    const cudaError_t e = launch_pdl(rows_stats_kernel<G>, dim3((unsigned)ctas), dim3(SR_NT), s, x, rows, len, out);
    count_launches(1);
    return cuda_fail(e != cudaSuccess ? e : cudaGetLastError(), "red_rows_stats launch");
}

}  // namespace

int launch_rows_stats(const float *x, int64_t rows, int64_t len, float *out, cudaStream_t s)
{
    DeviceInfo di;
    const int st = device_info(&di);
    if (st != RED_OK)
        return st;
    // rows of 16, 32 or 64 floats from a 32-byte aligned base: consecutive
    // lanes on consecutive blocks of the matrix
    if ((((uintptr_t)x) & 31u) == 0 && (len == 16 || len == 32 || len == 64)) {
        switch (len) {
        case 16: return launch_rows_stats_blocks<2>(x, rows, out, s, di.sms);
        case 32: return launch_rows_stats_blocks<4>(x, rows, out, s, di.sms);
        default: return launch_rows_stats_blocks<8>(x, rows, out, s, di.sms);
        }
    }
    int g = 1;  // about 32 floats per lane
    while (g < 32 && (int64_t)g * 64 <= len)
        g *= 2;
    switch (g) {
    case 1: return launch_rows_stats_g<1>(x, rows, len, out, s, di.sms);
    case 2: return launch_rows_stats_g<2>(x, rows, len, out, s, di.sms);
    case 4: return launch_rows_stats_g<4>(x, rows, len, out, s, di.sms);
    case 8: return launch_rows_stats_g<8>(x, rows, len, out, s, di.sms);
    case 16: return launch_rows_stats_g<16>(x, rows, len, out, s, di.sms);
    default: return launch_rows_stats_g<32>(x, rows, len, out, s, di.sms);
    }
}

int launch_full_stats(const float *x, int64_t n, float *out, cudaStream_t s)
{
    DeviceInfo di;
    int st = device_info(&di);
    if (st != RED_OK)
        return st;
    static std::atomic<int> occ_cache{0};
    const int occ = cached_occupancy(occ_cache, (const void *)stats_kernel, ST_NT);
    if (occ <= 0)
        return fail(RED_ECUDA, "red_full_stats: kernel cannot be resident on this device");
    const int64_t want = (n / 8 + 1 + (int64_t)ST_NT * ST_U - 1) / ((int64_t)ST_NT * ST_U);
    int64_t ctas = (int64_t)di.sms * occ;
    if (want < ctas)
        ctas = want;
    if (ctas < 1)
        ctas = 1;
    Workspace ws;
    if (ctas > 1) {
        st = get_workspace(&ws);
        if (st != RED_OK)
            return st;
    }
    const cudaError_t e =
        launch_pdl(stats_kernel, dim3((unsigned)ctas), dim3(ST_NT), s, x, n, static_cast<float *>(ws.part), ws.tick, out);
    count_launches(1);
    return cuda_fail(e != cudaSuccess ? e : cudaGetLastError(), "red_full_stats launch");
}

}  // namespace red
