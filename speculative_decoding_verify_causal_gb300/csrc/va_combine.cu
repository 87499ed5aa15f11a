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
// Grid: (split group, packed row); each thread owns head_dim columns
// d = tid, tid + 128, ... and reads the group's partials coalesced.
#include <cuda_bf16.h>
#include <math.h>

#include "va_internal.h"

namespace va {
namespace {

constexpr int kThreads = 128;

__global__ void __launch_bounds__(kThreads) combine_kernel(const CombineParams p) {
    extern __shared__ float w[];  // [n] weights exp(lse_s - lse)
    const Group g = p.groups[blockIdx.x];
    const int r = blockIdx.y;
    const int rr = g.rg * p.rows_per_group + r;
    if (r >= p.rows_per_group || rr >= p.R) return;
    const int tid = threadIdx.x;
    const int n = g.n;

    float m = -INFINITY;
    for (int s = tid; s < n; s += kThreads)
        m = fmaxf(m, p.lse_part[(size_t)(g.first_part + s) * p.rows_per_group + r]);
    __shared__ float red[kThreads / 32];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((tid & 31) == 0) red[tid >> 5] = m;
    __syncthreads();
    m = red[0];
#pragma unroll
    for (int i = 1; i < kThreads / 32; ++i) m = fmaxf(m, red[i]);
    __syncthreads();

    float z = 0.f;
    for (int s = tid; s < n; s += kThreads) {
        const float l = p.lse_part[(size_t)(g.first_part + s) * p.rows_per_group + r];
        const float e = (m == -INFINITY || l == -INFINITY) ? 0.f : expf(l - m);
        w[s] = e;
        z += e;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
    if ((tid & 31) == 0) red[tid >> 5] = z;
    __syncthreads();
    z = 0.f;
#pragma unroll
    for (int i = 0; i < kThreads / 32; ++i) z += red[i];
    const float inv = z > 0.f ? 1.f / z : 0.f;

    const int t = rr / p.G, h = g.kvh * p.G + rr % p.G;
    const size_t orow = (size_t)(g.b * p.T + t) * p.Hq + h;
    __syncthreads();  // w[] complete
    // Thread owns two adjacent columns; eight splits are loaded before any is
    // accumulated so that the loads overlap.
    const size_t pstride = (size_t)p.rows_per_group * p.D;  // floats between splits
    const float *base = p.o_part + ((size_t)g.first_part * p.rows_per_group + r) * p.D;
    for (int d = 2 * tid; d < p.D; d += 2 * kThreads) {
        float2 acc = make_float2(0.f, 0.f);
        int s = 0;
        for (; s + 8 <= n; s += 8) {
            float2 v[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) v[k] = *reinterpret_cast<const float2 *>(base + (s + k) * pstride + d);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                acc.x = fmaf(w[s + k], v[k].x, acc.x);
                acc.y = fmaf(w[s + k], v[k].y, acc.y);
            }
        }
        for (; s < n; ++s) {
            const float2 v = *reinterpret_cast<const float2 *>(base + s * pstride + d);
            acc.x = fmaf(w[s], v.x, acc.x);
            acc.y = fmaf(w[s], v.y, acc.y);
        }
        __nv_bfloat162 o = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
        *reinterpret_cast<__nv_bfloat162 *>(p.out + orow * p.D + d) = o;
    }
    if (tid == 0 && p.lse) p.lse[orow] = z > 0.f ? m + logf(z) : -INFINITY;
}

}  // namespace

cudaError_t launch_combine(const CombineParams &p, int num_groups, int max_splits, cudaStream_t s) {
    if (num_groups <= 0) return cudaSuccess;
    const size_t smem = sizeof(float) * (size_t)max_splits;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(combine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
    }
    dim3 grid(num_groups, p.rows_per_group);
    combine_kernel<<<grid, kThreads, smem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace va
