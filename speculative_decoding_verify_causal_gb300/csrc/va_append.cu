// KV append with quantise-on-write: the T verify tokens' K and V rows go into
// the paged cache, quantised per (token, kv head) with an absmax fp32 scale
// ("I pushed Qwen3.8-27B to 381 tps for a single request on a RTX 3090",
// "DFlash2 past 64k": int8 cache in 16-token pages, and "KVarN 4/2-bit KV
// cache", read as the int8 rule with 4 / 2 bits; "I pushed Qwen3.8-27B to
// 124 tps on a single request on a RTX 3090", "What we had": fp8 cache).
//
// One warp per (k or v, sequence, token, kv head) row; lane l holds elements
// [l E, l E + E) of the D-long row (E = D / 32).  The absmax is a warp
// max-reduction (exact); the scale and the quotients are IEEE fp32 divisions
// (__fdiv_rn), the e4m3 code is the hardware's round-to-nearest-even
// saturating conversion and the integer codes a round-half-even conversion, so
// every byte is the one the definition in verify_attn.h fixes.  HBM-bound:
// 2 B read and bits / 8 B (+ 4 B per row) written per element.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "va_internal.h"

namespace va {
namespace {

constexpr int kThreads = 256;
constexpr int kRowsPerBlock = kThreads / 32;

struct AppendParams {
    const uint16_t *k_new, *v_new;  // bf16 [B, T, Hkv, D]
    void *k_pages, *v_pages;
    float *k_scale, *v_scale;
    const int32_t *block_table;
    const int32_t *seq_lens;
    int *flags;
    int B, T, Hkv, bt_stride, num_pages, rows;  // rows = 2 * B * T * Hkv
};

template <int E>
struct Vec;  // the E bf16 values of a lane as one load
template <>
struct Vec<2> {
    using In = uint32_t;
};
template <>
struct Vec<4> {
    using In = uint2;
};
template <>
struct Vec<8> {
    using In = uint4;
};

template <int D, int DT>
__global__ void __launch_bounds__(kThreads) append_kernel(const AppendParams p) {
    constexpr int E = D / 32;
    using In = typename Vec<E>::In;
    griddep_wait();  // the new rows may come from the previous kernel on the stream
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row = blockIdx.x * kRowsPerBlock + warp;
    if (row >= p.rows) return;
    const int per_kv = p.B * p.T * p.Hkv;
    const int kv = row / per_kv, rem = row % per_kv;  // rem = (b T + t) Hkv + g
    const int g = rem % p.Hkv, bt_row = rem / p.Hkv;
    const int b = bt_row / p.T, t = bt_row % p.T;
    const int pos = p.seq_lens[b] - p.T + t;
    int page = -1;
    if (pos >= 0) page = p.block_table[(size_t)b * p.bt_stride + pos / VA_PAGE_SIZE];
    if (pos < 0 || (p.num_pages > 0 && (page < 0 || page >= p.num_pages))) {
        if (lane == 0 && p.flags) atomicOr(p.flags, 1);
        return;
    }
    const size_t dst_row = ((size_t)page * VA_PAGE_SIZE + pos % VA_PAGE_SIZE) * p.Hkv + g;
    const uint16_t *src = (kv == 0 ? p.k_new : p.v_new) + (size_t)rem * D + lane * E;
    const In raw = *reinterpret_cast<const In *>(src);
    const uint16_t *h = reinterpret_cast<const uint16_t *>(&raw);

    if constexpr (DT == VA_BF16) {
        unsigned char *dst = static_cast<unsigned char *>(kv == 0 ? p.k_pages : p.v_pages);
        *reinterpret_cast<In *>(dst + (dst_row * D + lane * E) * 2) = raw;
    } else if constexpr (DT == VA_INT4 || DT == VA_INT2) {
        // 4-bit / 2-bit codes: the int8 rule with qmax 7 / 1, each lane's E
        // codes packed into an F-bit field (element e at bit e * bits), then
        // the fields of 32 / F neighbouring lanes ORed into one 32-bit word
        // (lane order = element order, so the word is the row's little-endian
        // bit stream) that the first of them stores.
        constexpr int kBits = DT == VA_INT4 ? 4 : 2;
        constexpr int qm = (1 << (kBits - 1)) - 1;
        constexpr int F = E * kBits;          // 4 .. 32 bits per lane
        constexpr int kLanesPerWord = 32 / F;
        float x[E];
        float a = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            x[e] = __uint_as_float((uint32_t)h[e] << 16);
            a = fmaxf(a, fabsf(x[e]));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
        const float s = a > 0.f ? __fdiv_rn(a, (float)qm) : 1.f;
        uint32_t field = 0;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const int c = max(-qm, min(qm, __float2int_rn(__fdiv_rn(x[e], s))));
            field |= ((uint32_t)c & ((1u << kBits) - 1)) << (e * kBits);
        }
        uint32_t word = field;
#pragma unroll
        for (int k = 1; k < kLanesPerWord; ++k) {
            const uint32_t nb = __shfl_down_sync(0xffffffffu, field, k);
            if (lane + k < 32) word |= nb << (k * F);
        }
        unsigned char *dst = static_cast<unsigned char *>(kv == 0 ? p.k_pages : p.v_pages) +
                             dst_row * (D * kBits / 8);
        if (lane % kLanesPerWord == 0) *reinterpret_cast<uint32_t *>(dst + lane * F / 8) = word;
        if (lane == 0) (kv == 0 ? p.k_scale : p.v_scale)[dst_row] = s;
    } else {
        float x[E];
        float a = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            x[e] = __uint_as_float((uint32_t)h[e] << 16);
            a = fmaxf(a, fabsf(x[e]));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
        const float qmax = DT == VA_FP8_E4M3 ? 448.f : 127.f;
        const float s = a > 0.f ? __fdiv_rn(a, qmax) : 1.f;
        // codes of elements e, e + 1 as one 16-bit pair, element e in the low byte
        uint32_t pair[E / 2];
#pragma unroll
        for (int e = 0; e < E; e += 2) {
            float y0 = __fdiv_rn(x[e], s), y1 = __fdiv_rn(x[e + 1], s);
            if constexpr (DT == VA_FP8_E4M3) {
                y0 = fminf(fmaxf(y0, -448.f), 448.f);
                y1 = fminf(fmaxf(y1, -448.f), 448.f);
                pair[e / 2] = (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(y0, y1), __NV_SATFINITE, __NV_E4M3);
            } else {
                const uint32_t c0 = (uint32_t)(max(-127, min(127, __float2int_rn(y0))) & 0xFF);
                const uint32_t c1 = (uint32_t)(max(-127, min(127, __float2int_rn(y1))) & 0xFF);
                pair[e / 2] = c0 | (c1 << 8);
            }
        }
        unsigned char *dst = static_cast<unsigned char *>(kv == 0 ? p.k_pages : p.v_pages) + dst_row * D + lane * E;
        if constexpr (E == 2) {
            *reinterpret_cast<uint16_t *>(dst) = (uint16_t)pair[0];
        } else if constexpr (E == 4) {
            *reinterpret_cast<uint32_t *>(dst) = pair[0] | (pair[1] << 16);
        } else {
            *reinterpret_cast<uint2 *>(dst) = make_uint2(pair[0] | (pair[1] << 16), pair[2] | (pair[3] << 16));
        }
        if (lane == 0) (kv == 0 ? p.k_scale : p.v_scale)[dst_row] = s;
    }
}

template <int D>
cudaError_t launch_d(const AppendParams &p, int dtype, cudaStream_t s) {
    const dim3 grid((p.rows + kRowsPerBlock - 1) / kRowsPerBlock);
    switch (dtype) {
    case VA_BF16: return launch_pdl(append_kernel<D, VA_BF16>, grid, dim3(kThreads), 0, s, p);
    case VA_FP8_E4M3: return launch_pdl(append_kernel<D, VA_FP8_E4M3>, grid, dim3(kThreads), 0, s, p);
    case VA_INT8: return launch_pdl(append_kernel<D, VA_INT8>, grid, dim3(kThreads), 0, s, p);
    case VA_INT4: return launch_pdl(append_kernel<D, VA_INT4>, grid, dim3(kThreads), 0, s, p);
    default: return launch_pdl(append_kernel<D, VA_INT2>, grid, dim3(kThreads), 0, s, p);
    }
}

}  // namespace
}  // namespace va

extern "C" int verify_attn_kv_append(const void *k_new, const void *v_new, int num_seqs, int T,
                                     int num_kv_heads, int head_dim, va_kv_dtype kv_dtype, void *k_pages,
                                     void *v_pages, float *k_scale, float *v_scale,
                                     const int32_t *block_table, int block_table_stride,
                                     const int32_t *seq_lens, int num_pages, int *flags, void *stream) {
    if (!k_new || !v_new || !k_pages || !v_pages || !block_table || !seq_lens) return VA_ERR_INVALID_ARGUMENT;
    if (num_seqs < 1 || T < 1 || num_kv_heads < 1 || block_table_stride < 1 || num_pages < 0)
        return VA_ERR_INVALID_ARGUMENT;
    if (head_dim != 64 && head_dim != 128 && head_dim != 256) return VA_ERR_UNSUPPORTED;
    if (kv_dtype < VA_BF16 || kv_dtype > VA_INT2) return VA_ERR_UNSUPPORTED;
    if (kv_dtype != VA_BF16 && (!k_scale || !v_scale)) return VA_ERR_INVALID_ARGUMENT;
    auto misaligned = [](const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) != 0; };
    if (misaligned(k_new) || misaligned(v_new) || misaligned(k_pages) || misaligned(v_pages))
        return VA_ERR_INVALID_ARGUMENT;  // rows move as 16-byte (bf16 in) / 8-byte (codes out) units
    const long long rows = 2LL * num_seqs * T * num_kv_heads;
    if (rows > (1LL << 30)) return VA_ERR_INVALID_ARGUMENT;
    va::AppendParams p{};
    p.k_new = static_cast<const uint16_t *>(k_new);
    p.v_new = static_cast<const uint16_t *>(v_new);
    p.k_pages = k_pages;
    p.v_pages = v_pages;
    p.k_scale = k_scale;
    p.v_scale = v_scale;
    p.block_table = block_table;
    p.seq_lens = seq_lens;
    p.flags = flags;
    p.B = num_seqs;
    p.T = T;
    p.Hkv = num_kv_heads;
    p.bt_stride = block_table_stride;
    p.num_pages = num_pages;
    p.rows = (int)rows;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    switch (head_dim) {
    case 64: e = va::launch_d<64>(p, kv_dtype, s); break;
    case 128: e = va::launch_d<128>(p, kv_dtype, s); break;
    default: e = va::launch_d<256>(p, kv_dtype, s); break;
    }
    if (e != cudaSuccess) {
        va::note_cuda_error(e);
        return VA_ERR_CUDA;
    }
    return VA_OK;
}
