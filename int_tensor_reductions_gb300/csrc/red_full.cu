// red_full.cu -- the segmented full reduction: S CTAs cooperate on each of
// gridDim.y contiguous fp32 segments.  One segment is red_full (a vector to a
// scalar); many segments are the split-row path of red_rows for few, long
// rows.
//
// Per thread: 256-bit streaming loads of chunks of 8, U chunks in flight,
// folded by the 8-wide packed-add (sum) or 4-wide max3/min3 (max/min)
// accumulator of Apache TVM docs, "reduction -> sm100_packed", "Algorithm";
// an unaligned head and the ragged tail (each < 8 elements) are folded in
// scalar.  Per CTA: warp butterfly and shared-memory stage (the C block
// reduce of the Triton vector-accumulation blog post).  Per segment, the grid
// stage is one of:
//   two-pass    CTA partials to the workspace, then seg_finish_kernel;
//   last-block  CTA partials, fence, arrival counter; the CTA that arrives
//               last folds the partials (no CTA ever waits for another);
//   atomic      one atomic per CTA into the (identity-initialised) output,
//               the blog post's "one atomic per block" stage.
#include "red_internal.h"
#include "red_prims.cuh"
#include "red.h"

namespace red {
namespace {

constexpr int FULL_NT = 512;   // threads per CTA (2 resident per SM: 1024 threads)
constexpr int FULL_U = 4;      // 256-bit loads in flight per thread

enum : int { STAGE_TWO_PASS = 1, STAGE_LAST_BLOCK = 2, STAGE_ATOMIC = 3 };

// Order-preserving atomic max / min on an fp32 location: a non-negative
// value compares like its bit pattern as a signed int, a negative one like
// its bit pattern as an unsigned int in reverse.
template <int OP>
__device__ __forceinline__ void atomic_fold(float *addr, float v);

template <>
__device__ __forceinline__ void atomic_fold<OP_SUM>(float *addr, float v)
{
    atomicAdd(addr, v);
}

template <>
__device__ __forceinline__ void atomic_fold<OP_MAX>(float *addr, float v)
{
    if (!(__float_as_uint(v) & 0x80000000u))
        atomicMax(reinterpret_cast<int *>(addr), __float_as_int(v));
    else
        atomicMin(reinterpret_cast<unsigned *>(addr), __float_as_uint(v));
}

template <>
__device__ __forceinline__ void atomic_fold<OP_MIN>(float *addr, float v)
{
    if (!(__float_as_uint(v) & 0x80000000u))
        atomicMin(reinterpret_cast<int *>(addr), __float_as_int(v));
    else
        atomicMax(reinterpret_cast<unsigned *>(addr), __float_as_uint(v));
}

template <int OP>
__global__ void fill_identity_kernel(float *out, int64_t n)
{
    pdl_enter();
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n)
        out[i] = Op<OP>::identity();
}

// gridDim.x CTAs per segment, gridDim.y segments; segment y is
// x[y*len .. y*len+len).  part holds gridDim.x partials per segment, tick one
// arrival counter per segment.
template <int OP, int STAGE>
__global__ void __launch_bounds__(FULL_NT)
seg_kernel(const float *__restrict__ x, int64_t len, int accum, float *__restrict__ part,
           unsigned *__restrict__ tick, float *__restrict__ out)
{
    __shared__ float s_red[FULL_NT / 32];
    __shared__ int s_last;

    pdl_enter();
    const int64_t seg = blockIdx.y;
    const float *p = x + seg * len;
    const int64_t h = head_to_32B(p, len);
    const int64_t nch = (len - h) >> 3;
    const int64_t t0 = h + (nch << 3);
    const int64_t tid = (int64_t)blockIdx.x * FULL_NT + threadIdx.x;
    const int64_t nth = (int64_t)gridDim.x * FULL_NT;
    const float *pa = p + h;

    Fold<OP> f;
    f.init();
    int64_t c = tid;
    for (; c + (FULL_U - 1) * nth < nch; c += FULL_U * nth) {
        float v[FULL_U][8];
#pragma unroll
        for (int u = 0; u < FULL_U; ++u)
            ld8(pa + 8 * (c + u * nth), v[u]);
#pragma unroll
        for (int u = 0; u < FULL_U; ++u)
            f.chunk(v[u]);
    }
    for (; c < nch; c += nth) {
        float v[8];
        ld8(pa + 8 * c, v);
        f.chunk(v);
    }
    if (tid < h)
        f.scalar(ld1(p + tid));
    if (tid < len - t0)
        f.scalar(ld1(p + t0 + tid));

    float v = cta_reduce<OP, FULL_NT / 32>(f.finish(), s_red);

    if (STAGE == STAGE_ATOMIC) {
        if (threadIdx.x == 0)
            atomic_fold<OP>(out + seg, v);
        return;
    }
    if (gridDim.x == 1) {  // one CTA per segment: no grid stage
        if (threadIdx.x == 0)
            out[seg] = accum ? Op<OP>::combine(out[seg], v) : v;
        return;
    }
    if (threadIdx.x == 0)
        part[seg * gridDim.x + blockIdx.x] = v;
    if (STAGE == STAGE_TWO_PASS)
        return;

    // last-block stage: the CTA that arrives last folds the partials
    if (threadIdx.x == 0) {
        __threadfence();
        const unsigned t = atomicAdd(tick + seg, 1u);
        s_last = (t == gridDim.x - 1);
    }
    __syncthreads();
    if (!s_last)
        return;
    __threadfence();
    float w = Op<OP>::identity();
    for (int i = threadIdx.x; i < (int)gridDim.x; i += FULL_NT)
        w = Op<OP>::combine(w, __ldcg(part + seg * gridDim.x + i));
    w = cta_reduce<OP, FULL_NT / 32>(w, s_red);
    if (threadIdx.x == 0) {
        out[seg] = accum ? Op<OP>::combine(out[seg], w) : w;
        tick[seg] = 0;
    }
}

// Two-pass second stage: one CTA per segment folds its nparts partials.
template <int OP>
__global__ void __launch_bounds__(FULL_NT)
seg_finish_kernel(const float *__restrict__ part, int nparts, int accum, float *__restrict__ out)
{
    __shared__ float s_red[FULL_NT / 32];
    pdl_enter();
    const int64_t seg = blockIdx.x;
    float w = Op<OP>::identity();
    for (int i = threadIdx.x; i < nparts; i += FULL_NT)
        w = Op<OP>::combine(w, part[seg * nparts + i]);
    w = cta_reduce<OP, FULL_NT / 32>(w, s_red);
    if (threadIdx.x == 0)
        out[seg] = accum ? Op<OP>::combine(out[seg], w) : w;
}

template <int OP, int STAGE>
int seg_occupancy()
{
    static std::atomic<int> occ_cache{0};
    return cached_occupancy(occ_cache, (const void *)seg_kernel<OP, STAGE>, FULL_NT);
}

// Launch the segmented reduction with `splits` CTAs per segment.
template <int OP>
int launch_seg(int stage, const float *x, int64_t segs, int64_t len, int splits, int accum,
               float *out, const Workspace &ws, cudaStream_t s)
{
    const dim3 grid((unsigned)splits, (unsigned)segs);
    cudaError_t e = cudaSuccess;
    if (stage == STAGE_ATOMIC) {
        e = launch_pdl(fill_identity_kernel<OP>, dim3((unsigned)((segs + 255) / 256)), dim3(256), s, out, segs);
        if (e == cudaSuccess)
            e = launch_pdl(seg_kernel<OP, STAGE_ATOMIC>, grid, dim3(FULL_NT), s, x, len, 0, (float *)nullptr,
                           (unsigned *)nullptr, out);
        count_launches(2);
    } else if (stage == STAGE_TWO_PASS) {
        float *part = static_cast<float *>(ws.part);
        e = launch_pdl(seg_kernel<OP, STAGE_TWO_PASS>, grid, dim3(FULL_NT), s, x, len, accum, part,
                       (unsigned *)nullptr, out);
        count_launches(1);
        if (e == cudaSuccess && splits > 1) {
            e = launch_pdl(seg_finish_kernel<OP>, dim3((unsigned)segs), dim3(FULL_NT), s, (const float *)part, splits,
                           accum, out);
            count_launches(1);
        }
    } else {
        e = launch_pdl(seg_kernel<OP, STAGE_LAST_BLOCK>, grid, dim3(FULL_NT), s, x, len, accum,
                       static_cast<float *>(ws.part), ws.tick, out);
        count_launches(1);
    }
    return cuda_fail(e != cudaSuccess ? e : cudaGetLastError(), "segmented reduction launch");
}

int launch_seg_op(int op, int stage, const float *x, int64_t segs, int64_t len, int splits, int accum,
                  float *out, const Workspace &ws, cudaStream_t s)
{
    switch (op) {
    case OP_SUM: return launch_seg<OP_SUM>(stage, x, segs, len, splits, accum, out, ws, s);
    case OP_MAX: return launch_seg<OP_MAX>(stage, x, segs, len, splits, accum, out, ws, s);
    default: return launch_seg<OP_MIN>(stage, x, segs, len, splits, accum, out, ws, s);
    }
}

int ctas_per_sm(int op, int stage)
{
    const int k = knob(RED_KNOB_FULL_CTAS_PER_SM);
    if (k > 0)
        return k;
    switch (op * 4 + stage) {
    case OP_SUM * 4 + STAGE_TWO_PASS: return seg_occupancy<OP_SUM, STAGE_TWO_PASS>();
    case OP_SUM * 4 + STAGE_LAST_BLOCK: return seg_occupancy<OP_SUM, STAGE_LAST_BLOCK>();
    case OP_SUM * 4 + STAGE_ATOMIC: return seg_occupancy<OP_SUM, STAGE_ATOMIC>();
    case OP_MAX * 4 + STAGE_TWO_PASS: return seg_occupancy<OP_MAX, STAGE_TWO_PASS>();
    case OP_MAX * 4 + STAGE_LAST_BLOCK: return seg_occupancy<OP_MAX, STAGE_LAST_BLOCK>();
    case OP_MAX * 4 + STAGE_ATOMIC: return seg_occupancy<OP_MAX, STAGE_ATOMIC>();
    case OP_MIN * 4 + STAGE_TWO_PASS: return seg_occupancy<OP_MIN, STAGE_TWO_PASS>();
    case OP_MIN * 4 + STAGE_LAST_BLOCK: return seg_occupancy<OP_MIN, STAGE_LAST_BLOCK>();
    default: return seg_occupancy<OP_MIN, STAGE_ATOMIC>();
    }
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace

int launch_full(int op, const float *x, int64_t n, float *out, cudaStream_t s)
{
    DeviceInfo di;
    int st = device_info(&di);
    if (st != RED_OK)
        return st;
    int stage = full_stage(op);
    const int occ = ctas_per_sm(op, stage);
    if (occ <= 0)
        return fail(RED_ECUDA, "red_full: kernel cannot be resident on this device");
    // Enough CTAs to fill the machine once, but no more than the data needs
    // for every thread to have FULL_U chunks in its first round.
    const int64_t want = ceil_div(n / 8 + 1, (int64_t)FULL_NT * FULL_U);
    int64_t ctas = (int64_t)di.sms * occ;
    if (want < ctas)
        ctas = want;
    if (ctas < 1)
        ctas = 1;
    if (ctas == 1)
        stage = STAGE_LAST_BLOCK;  // one CTA writes the result itself: no grid stage, one launch
    Workspace ws;
    if (stage != STAGE_ATOMIC && ctas > 1) {
        st = get_workspace(&ws);
        if (st != RED_OK)
            return st;
    }
    return launch_seg_op(op, stage, x, 1, n, (int)ctas, 0, out, ws, s);
}

int launch_full_scratch(int op, const float *x, int64_t n, float *out, cudaStream_t s, float *part,
                        unsigned *tick, int64_t max_parts)
{
    DeviceInfo di;
    const int st = device_info(&di);
    if (st != RED_OK)
        return st;
    const int occ = ctas_per_sm(op, STAGE_LAST_BLOCK);
    if (occ <= 0)
        return fail(RED_ECUDA, "red_full_noalloc: kernel cannot be resident on this device");
    const int64_t want = ceil_div(n / 8 + 1, (int64_t)FULL_NT * FULL_U);
    int64_t ctas = (int64_t)di.sms * occ;
    if (want < ctas)
        ctas = want;
    if (ctas < 1)
        ctas = 1;
    if (ctas > max_parts)
        return fail(RED_EINVAL,
                    "red_full_noalloc: this launch needs %lld partial slots but the static scratch holds %lld "
                    "(lower RED_KNOB_FULL_CTAS_PER_SM)",
                    (long long)ctas, (long long)max_parts);
    Workspace ws;
    ws.part = part;
    ws.tick = tick;
    return launch_seg_op(op, STAGE_LAST_BLOCK, x, 1, n, (int)ctas, 0, out, ws, s);
}

int launch_rows_split(int op, const float *x, int64_t rows, int64_t len, int accum, float *out,
                      cudaStream_t s, const DeviceInfo &di)
{
    const int occ = ctas_per_sm(op, STAGE_LAST_BLOCK);
    if (occ <= 0)
        return fail(RED_ECUDA, "red_rows: kernel cannot be resident on this device");
    // rows * splits CTAs in one wave of resident CTAs (rounding the split
    // count up would leave a few CTAs to run alone after the wave)
    const int64_t target = (int64_t)di.sms * occ;
    int64_t splits = target / rows;
    const int64_t need = ceil_div(len / 8 + 1, (int64_t)FULL_NT * FULL_U);
    if (splits > need)
        splits = need;
    if (splits * rows > (int64_t)WS_PART_ELEMS)
        splits = (int64_t)WS_PART_ELEMS / rows;
    if (splits < 1)
        splits = 1;
    Workspace ws;
    if (splits > 1) {
        const int st = get_workspace(&ws);
        if (st != RED_OK)
            return st;
    }
    return launch_seg_op(op, STAGE_LAST_BLOCK, x, rows, len, (int)splits, accum, out, ws, s);
}

}  // namespace red
