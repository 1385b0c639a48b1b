// red_stats.cu -- sum, max, min and sum |x| of one fp32 vector from a single
// read (the three separate red_full calls read x three times).
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

}  // namespace

int launch_full_stats(const float *x, int64_t n, float *out, cudaStream_t s)
{
    DeviceInfo di;
    int st = device_info(&di);
    if (st != RED_OK)
        return st;
    static int occ = 0;
    if (occ == 0)
        occ = occupancy((const void *)stats_kernel, ST_NT);
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
    stats_kernel<<<(unsigned)ctas, ST_NT, 0, s>>>(x, n, static_cast<float *>(ws.part), ws.tick, out);
    count_launches(1);
    return cuda_fail(cudaGetLastError(), "red_full_stats launch");
}

}  // namespace red
