// Log-sum-exp merge of the split partials (the "merge" half of split-KV,
// "I pushed Qwen3.8-27B to 124 tps on a single request on a RTX 3090",
// bullet "Split-KV attention kernel for the verify step").
//
// Split s of a row reports its normalised output o_s and lse_s = ln sum of
// exp(score) over its keys.  The row's result is
//     lse = ln sum_s exp(lse_s),   out = sum_s exp(lse_s - lse) * o_s,
// evaluated against the largest lse_s for range safety.  A split whose keys
// are all masked for the row has lse_s = -inf and weight 0.
//
// Grid: (split group, packed row), 256 threads.  Warp w accumulates the
// splits s = w, w + 8, ... over all D columns (each lane owns D/32 adjacent
// columns, so a warp reads one split's row as one coalesced segment), with
// the loads of up to eight of its splits in flight before any is used; the
// eight warps' sums are then added through shared memory.
#include <cuda_bf16.h>
#include <math.h>

#include "va_internal.h"

namespace va {
namespace {

constexpr int kThreads = 256;
constexpr int kSlices = kThreads / 32;

template <int D>
__global__ void __launch_bounds__(kThreads) combine_kernel(const CombineParams p) {
    constexpr int kCols = D / 32;   // columns per lane: 2, 4 or 8
    constexpr int kBatch = 8;       // splits per warp whose loads are in flight together
    __shared__ float red[kSlices][D];
    __shared__ float wsm[kSlices * kBatch];
    __shared__ float wred[kSlices];
    // programmatic dependent launch: the partials are the previous kernel's
    // output.  (No early trigger here: the next call's partial kernel would
    // take the SMs this grid still needs.)
    griddep_wait();
    const Group g = p.groups[blockIdx.x];
    const int r = blockIdx.y;
    const int rr = g.rg * p.rows_per_group + r;
    if (r >= p.rows_per_group || rr >= p.R) return;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n = g.n;
    const float *lse_col = p.lse_part + (size_t)g.first_part * p.rows_per_group + r;
    const size_t pstride = (size_t)p.rows_per_group * D;  // floats between splits
    const float *base = p.o_part + ((size_t)g.first_part * p.rows_per_group + r) * D + lane * kCols;

    // the first chunk's partial rows are requested before anything else, so
    // that their latency overlaps the lse maximum below
    float v[kBatch][kCols];
    auto load_chunk = [&](int c0) {
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int s = c0 + warp + kSlices * u;
            const float *src = base + (size_t)min(s, n - 1) * pstride;
#pragma unroll
            for (int c = 0; c < kCols; c += 2) {
                const float2 x = s < n ? *reinterpret_cast<const float2 *>(src + c) : make_float2(0.f, 0.f);
                v[u][c] = x.x;
                v[u][c + 1] = x.y;
            }
        }
    };
    load_chunk(0);

    // the row's maximum lse
    float m = -INFINITY;
    for (int s = tid; s < n; s += kThreads) m = fmaxf(m, lse_col[(size_t)s * p.rows_per_group]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) wred[warp] = m;
    __syncthreads();
    m = wred[0];
#pragma unroll
    for (int i = 1; i < kSlices; ++i) m = fmaxf(m, wred[i]);

    // by chunks of kSlices * kBatch splits: warp w takes splits c0 + w + kSlices * u
    float acc[kCols];
#pragma unroll
    for (int c = 0; c < kCols; ++c) acc[c] = 0.f;
    float zl = 0.f;  // this thread's share of sum exp(lse_s - m)
    for (int c0 = 0; c0 < n; c0 += kSlices * kBatch) {
        if (c0 > 0) load_chunk(c0);
        __syncthreads();  // wsm free
        if (tid < kSlices * kBatch) {
            const int s = c0 + (tid % kSlices) + kSlices * (tid / kSlices);
            float e = 0.f;
            if (s < n) {
                const float l = lse_col[(size_t)s * p.rows_per_group];
                e = (m == -INFINITY || l == -INFINITY) ? 0.f : expf(l - m);
            }
            wsm[tid] = e;
            zl += e;
        }
        __syncthreads();
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const float ws = wsm[warp + kSlices * u];
#pragma unroll
            for (int c = 0; c < kCols; ++c) acc[c] = fmaf(ws, v[u][c], acc[c]);
        }
    }
#pragma unroll
    for (int c = 0; c < kCols; ++c) red[warp][lane * kCols + c] = acc[c];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) zl += __shfl_xor_sync(0xffffffffu, zl, o);
    __syncthreads();
    if (lane == 0) wred[warp] = zl;
    __syncthreads();
    float z = 0.f;
#pragma unroll
    for (int i = 0; i < kSlices; ++i) z += wred[i];
    const float inv = z > 0.f ? 1.f / z : 0.f;

    const int t = rr / p.G, h = g.kvh * p.G + rr % p.G;
    const size_t orow = (size_t)(g.b * p.T + t) * p.Hq + h;
    for (int d = 2 * tid; d < D; d += 2 * kThreads) {
        float a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int i = 0; i < kSlices; ++i) {
            a0 += red[i][d];
            a1 += red[i][d + 1];
        }
        *reinterpret_cast<__nv_bfloat162 *>(p.out + orow * D + d) = __floats2bfloat162_rn(a0 * inv, a1 * inv);
    }
    if (tid == 0 && p.lse) p.lse[orow] = z > 0.f ? m + logf(z) : -INFINITY;
}

template <int D>
cudaError_t launch_d(const CombineParams &p, int num_groups, int max_splits, cudaStream_t s) {
    (void)max_splits;
    dim3 grid(num_groups, p.rows_per_group);
    return launch_pdl(combine_kernel<D>, grid, dim3(kThreads), 0, s, p);
}

}  // namespace

cudaError_t launch_combine(const CombineParams &p, int num_groups, int max_splits, cudaStream_t s) {
    if (num_groups <= 0) return cudaSuccess;
    switch (p.D) {
    case 64: return launch_d<64>(p, num_groups, max_splits, s);
    case 128: return launch_d<128>(p, num_groups, max_splits, s);
    default: return launch_d<256>(p, num_groups, max_splits, s);
    }
}

}  // namespace va
