// CUDA-core partial-attention kernel (the small-row path).
//
// Used when the packed rows of a kv head (G query heads x T verify tokens)
// are too few to fill a tensor-core tile, e.g. T = 1 decode with a small
// group, and as the always-available fallback.  Dot products run on the
// FP32 pipes with warp-shuffle reductions for the softmax statistics.
//
// One CTA = one work item: up to 16 packed rows of one kv head of one
// sequence over one key range (one split of "split-KV", from "I pushed
// Qwen3.8-27B to 124 tps on a single request on a RTX 3090", bullet
// "Split-KV attention kernel for the verify step").  Per 32-key tile:
//   1. the 32 K and V rows are gathered through the block table (16-byte
//      loads; 8 / 4 bytes for the 4-bit / 2-bit caches), dequantised
//      (fp8-e4m3 / int8 / int4 / int2 times the per-token scale, or bf16) and
//      staged in shared memory as fp32;
//   2. lane j of each warp scores key j against the warp's rows, applies the
//      bottom-right causal mask (verify token t sees keys j <= L - T + t) and
//      updates the row's running max / sum with shuffles (online softmax in
//      base 2: the scale log2(e)/sqrt(D) is folded into q);
//   3. every thread owns a slice of head_dim for all rows and accumulates
//      P x V after rescaling by exp2(m_old - m_new).
// The item then writes either the final bf16 output and natural-log LSE (an
// unsplit sequence) or its normalised fp32 partial and LSE for the combine.
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <math.h>

#include "va_internal.h"

namespace va {
namespace {

constexpr int kThreads = 128;

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

__device__ __forceinline__ uint16_t float_to_bf16_bits(float f) {
    __nv_bfloat16 h = __float2bfloat16_rn(f);
    return *reinterpret_cast<uint16_t *>(&h);
}

// Decode the 16 bytes of `raw` (one aligned chunk of a cache row) into floats.
template <int DT>
__device__ __forceinline__ void decode16(const uint4 &raw, float *dst, float scale);

template <>
__device__ __forceinline__ void decode16<VA_BF16>(const uint4 &raw, float *dst, float) {
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        dst[2 * i] = __uint_as_float(w[i] << 16);
        dst[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

template <>
__device__ __forceinline__ void decode16<VA_FP8_E4M3>(const uint4 &raw, float *dst, float scale) {
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int hlf = 0; hlf < 2; ++hlf) {
            __nv_fp8x2_storage_t pair = static_cast<__nv_fp8x2_storage_t>(w[i] >> (16 * hlf));
            __half2_raw h2 = __nv_cvt_fp8x2_to_halfraw2(pair, __NV_E4M3);
            float2 f = __half22float2(*reinterpret_cast<__half2 *>(&h2));
            dst[4 * i + 2 * hlf] = f.x * scale;
            dst[4 * i + 2 * hlf + 1] = f.y * scale;
        }
    }
}

template <>
__device__ __forceinline__ void decode16<VA_INT8>(const uint4 &raw, float *dst, float scale) {
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int k = 0; k < 4; ++k)
            dst[4 * i + k] = static_cast<float>(static_cast<int8_t>(w[i] >> (8 * k))) * scale;
}

// 4-bit / 2-bit caches: 16 codes in 8 / 4 bytes (raw.x, raw.y), code k of a
// word in bits [k bits, (k + 1) bits), sign-extended by an arithmetic shift.
template <>
__device__ __forceinline__ void decode16<VA_INT4>(const uint4 &raw, float *dst, float scale) {
    const uint32_t w[2] = {raw.x, raw.y};
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int k = 0; k < 8; ++k)
            dst[8 * i + k] = static_cast<float>(static_cast<int32_t>(w[i] << (28 - 4 * k)) >> 28) * scale;
}

template <>
__device__ __forceinline__ void decode16<VA_INT2>(const uint4 &raw, float *dst, float scale) {
#pragma unroll
    for (int k = 0; k < 16; ++k)
        dst[k] = static_cast<float>(static_cast<int32_t>(raw.x << (30 - 2 * k)) >> 30) * scale;
}

// Bits per cached element, and the raw bytes holding one decode16 chunk.
template <int DT>
__host__ __device__ constexpr int elem_bits() {
    return DT == VA_BF16 ? 16 : DT == VA_INT4 ? 4 : DT == VA_INT2 ? 2 : 8;
}

// One chunk of a cache row as 16 / 8 / 4 aligned bytes (unused words zero).
template <int BYTES>
__device__ __forceinline__ uint4 load_chunk(const uint8_t *src) {
    if constexpr (BYTES == 16) {
        return *reinterpret_cast<const uint4 *>(src);
    } else if constexpr (BYTES == 8) {
        const uint2 v = *reinterpret_cast<const uint2 *>(src);
        return make_uint4(v.x, v.y, 0u, 0u);
    } else {
        return make_uint4(*reinterpret_cast<const uint32_t *>(src), 0u, 0u, 0u);
    }
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

template <int D>
constexpr int smem_floats() {
    return kWarpRows * D + kWarpTile * (D + 1) + kWarpTile * D + kWarpRows * kWarpTile +
           3 * kWarpRows + kWarpTile;
}

template <int D, int DT>
__global__ void __launch_bounds__(kThreads) warp_partial_kernel(const PartialParams p) {
    constexpr int RB = kWarpRows;
    constexpr int TK = kWarpTile;
    constexpr int EPC = DT == VA_BF16 ? 8 : 16;     // elements per decoded chunk
    constexpr int CB = EPC * elem_bits<DT>() / 8;   // raw bytes per chunk (16, 8 or 4)
    constexpr int RB_BYTES = D * elem_bits<DT>() / 8;  // bytes per cache row
    constexpr int CPR = D / EPC;                    // chunks per cache row
    constexpr int DPT = (D + kThreads - 1) / kThreads;  // head_dim slice per thread
    // programmatic dependent launch: nothing of the caller's is touched before this
    griddep_wait();

    extern __shared__ float smem[];
    float *Qs = smem;                 // [RB][D]   q * log2(e)/sqrt(D)
    float *Ks = Qs + RB * D;          // [TK][D+1] dequantised keys (padded rows)
    float *Vs = Ks + TK * (D + 1);    // [TK][D]   dequantised values
    float *Ps = Vs + TK * D;          // [RB][TK]  probabilities of the tile
    float *As = Ps + RB * TK;         // [RB]      rescale factor of the tile
    float *Ms = As + RB;              // [RB]      final running max (log2 units)
    float *Ls = Ms + RB;              // [RB]      final running sum
    int *Valid = reinterpret_cast<int *>(Ls + RB);  // [TK] key passed bound checks

    const Item it = p.items[blockIdx.x];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = p.G, T = p.T;
    const int row0 = it.rg * p.rows_per_group;
    const int nrows = min(p.rows_per_group, p.R - row0);
    const int Hkv = p.Hkv;

    if (tid == 0 && p.seq_lens[it.b] != it.L) atomicOr(p.flags, kFlagSeqLenMismatch);

    for (int i = tid; i < RB * D; i += kThreads) {
        const int r = i / D, d = i % D;
        float v = 0.f;
        if (r < nrows) {
            const int rr = row0 + r;
            const int t = rr / G, h = it.kvh * G + rr % G;
            v = bf16_bits_to_float(p.q[((size_t)(it.b * T + t) * p.Hq + h) * D + d]) * p.sm_scale_log2;
        }
        Qs[i] = v;
    }

    float m_run[RB / 4], l_run[RB / 4];
#pragma unroll
    for (int i = 0; i < RB / 4; ++i) {
        m_run[i] = -INFINITY;
        l_run[i] = 0.f;
    }
    float acc[RB][DPT];
#pragma unroll
    for (int r = 0; r < RB; ++r)
#pragma unroll
        for (int k = 0; k < DPT; ++k) acc[r][k] = 0.f;

    const uint8_t *kbase = static_cast<const uint8_t *>(p.k_pages);
    const uint8_t *vbase = static_cast<const uint8_t *>(p.v_pages);
    const int32_t *bt = p.block_table + (size_t)it.b * p.bt_stride;

    for (int k0 = it.k_begin; k0 < it.k_end; k0 += TK) {
        __syncthreads();  // previous tile fully consumed
        if (tid < TK) {
            const int key = k0 + tid;
            int ok = key < it.k_end;
            if (ok && p.num_pages > 0) {
                const int page = bt[key / VA_PAGE_SIZE];
                if (page < 0 || page >= p.num_pages) {
                    atomicOr(p.flags, kFlagBadPage);
                    ok = 0;
                }
            }
            Valid[tid] = ok;
        }
        __syncthreads();
        for (int c = tid; c < TK * CPR; c += kThreads) {
            const int j = c / CPR, part = c % CPR;
            const int key = k0 + j;
            float kf[EPC], vf[EPC];
            if (Valid[j]) {
                const int page = bt[key / VA_PAGE_SIZE];
                const size_t row = ((size_t)page * VA_PAGE_SIZE + key % VA_PAGE_SIZE) * Hkv + it.kvh;
                const uint4 kr = load_chunk<CB>(kbase + row * RB_BYTES + part * CB);
                const uint4 vr = load_chunk<CB>(vbase + row * RB_BYTES + part * CB);
                const float ks = DT == VA_BF16 ? 1.f : p.k_scale[row];
                const float vs = DT == VA_BF16 ? 1.f : p.v_scale[row];
                decode16<DT>(kr, kf, ks);
                decode16<DT>(vr, vf, vs);
            } else {
#pragma unroll
                for (int e = 0; e < EPC; ++e) kf[e] = vf[e] = 0.f;
            }
#pragma unroll
            for (int e = 0; e < EPC; ++e) {
                Ks[j * (D + 1) + part * EPC + e] = kf[e];
                Vs[j * D + part * EPC + e] = vf[e];
            }
        }
        __syncthreads();

        // scores + online softmax statistics: warp w owns rows w, w+4, ...
#pragma unroll
        for (int i = 0; i < RB / 4; ++i) {
            const int r = warp + 4 * i;
            if (r >= nrows) break;
            const int t = (row0 + r) / G;
            const int key = k0 + lane;
            const bool vis = Valid[lane] && key <= it.L - T + t;
            float dot = 0.f;
#pragma unroll 8
            for (int d = 0; d < D; ++d) dot = fmaf(Qs[r * D + d], Ks[lane * (D + 1) + d], dot);
            const float s = vis ? dot : -INFINITY;
            const float m_new = fmaxf(m_run[i], warp_max(s));
            float alpha = 1.f, pr = 0.f;
            if (m_new != -INFINITY) {
                alpha = m_run[i] == -INFINITY ? 0.f : exp2f(m_run[i] - m_new);
                pr = vis ? exp2f(s - m_new) : 0.f;
            }
            l_run[i] = l_run[i] * alpha + warp_sum(pr);
            m_run[i] = m_new;
            Ps[r * TK + lane] = pr;
            if (lane == 0) As[r] = alpha;
        }
        __syncthreads();

        // P x V: thread owns columns d = tid + 128*k of every row
#pragma unroll
        for (int r = 0; r < RB; ++r) {
            if (r < nrows) {
                const float a = As[r];
#pragma unroll
                for (int k = 0; k < DPT; ++k) acc[r][k] *= a;
            }
        }
        for (int j = 0; j < TK; ++j) {
            float v[DPT];
#pragma unroll
            for (int k = 0; k < DPT; ++k) {
                const int d = tid + k * kThreads;
                v[k] = d < D ? Vs[j * D + d] : 0.f;
            }
#pragma unroll
            for (int r = 0; r < RB; ++r) {
                const float pr = Ps[r * TK + j];
#pragma unroll
                for (int k = 0; k < DPT; ++k) acc[r][k] = fmaf(pr, v[k], acc[r][k]);
            }
        }
    }

#pragma unroll
    for (int i = 0; i < RB / 4; ++i) {
        const int r = warp + 4 * i;
        if (r < nrows && lane == 0) {
            Ms[r] = m_run[i];
            Ls[r] = l_run[i];
        }
    }
    __syncthreads();

#pragma unroll
    for (int r = 0; r < RB; ++r) {
        if (r >= nrows) break;
        const float l = Ls[r];
        const float inv = l > 0.f ? 1.f / l : 0.f;
        const float lse_nat = l > 0.f ? (Ms[r] + log2f(l)) * 0.69314718055994531f : -INFINITY;
        const int rr = row0 + r;
        const int t = rr / G, h = it.kvh * G + rr % G;
        if (it.part < 0) {
            const size_t orow = ((size_t)(it.b * T + t) * p.Hq + h);
#pragma unroll
            for (int k = 0; k < DPT; ++k) {
                const int d = tid + k * kThreads;
                if (d < D) p.out[orow * D + d] = float_to_bf16_bits(acc[r][k] * inv);
            }
            if (tid == 0 && p.lse) p.lse[orow] = lse_nat;
        } else {
            const size_t prow = (size_t)it.part * p.rows_per_group + r;
#pragma unroll
            for (int k = 0; k < DPT; ++k) {
                const int d = tid + k * kThreads;
                if (d < D) p.o_part[prow * D + d] = acc[r][k] * inv;
            }
            if (tid == 0) p.lse_part[prow] = lse_nat;
        }
    }
}

template <int D, int DT>
cudaError_t launch_one(const PartialParams &p, int n, cudaStream_t s) {
    const size_t smem = sizeof(float) * smem_floats<D>();
    auto k = warp_partial_kernel<D, DT>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(k, dim3(n), dim3(kThreads), smem, s, p);
}

template <int D>
cudaError_t launch_d(const PartialParams &p, int dtype, int n, cudaStream_t s) {
    switch (dtype) {
    case VA_BF16: return launch_one<D, VA_BF16>(p, n, s);
    case VA_FP8_E4M3: return launch_one<D, VA_FP8_E4M3>(p, n, s);
    case VA_INT8: return launch_one<D, VA_INT8>(p, n, s);
    case VA_INT4: return launch_one<D, VA_INT4>(p, n, s);
    default: return launch_one<D, VA_INT2>(p, n, s);
    }
}

}  // namespace

cudaError_t launch_warp_partial(const PartialParams &p, int head_dim, int kv_dtype, int n,
                                cudaStream_t s) {
    if (n <= 0) return cudaSuccess;
    switch (head_dim) {
    case 64: return launch_d<64>(p, kv_dtype, n, s);
    case 128: return launch_d<128>(p, kv_dtype, n, s);
    default: return launch_d<256>(p, kv_dtype, n, s);
    }
}

}  // namespace va
