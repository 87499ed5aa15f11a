// CUDA-core partial-attention kernel: the few-rows path.
//
// For a kv head whose packed rows (G query heads x T verify tokens) are too
// few to fill a tensor-core tile -- T = 1 decode with a small group -- the
// dot products run on the FP32 pipes ("I pushed Qwen3.8-27B to 124 tps on a
// single request on a RTX 3090", bullet "Split-KV attention kernel for the
// verify step": split the cache so that a handful of queries still fills the
// chip).  Each CTA takes one work item: up to 4 packed rows of one kv head of
// one sequence over one key range.  Nothing is staged in shared memory on the
// way: every warp streams its own batches of keys straight into registers and
// keeps its own online-softmax state, and the CTA's four warps merge their
// states once at the end.
//
// Per batch of KG keys (a 16-token page holds one or two batches):
//   * lane l owns elements [l D/32, (l+1) D/32) of every cache row, so the
//     32 lanes read a row as one contiguous, coalesced run of D * bits / 8
//     bytes (16 to 512), for the KG key rows and the KG value rows at once;
//   * the codes become fp32 exactly on the FP32 pipe (integers through the
//     2^23 magic number, bf16 by a shift; fp8-e4m3 through the hardware's
//     exact conversion to fp16); the per-token scales multiply the scores and
//     the probabilities, not the elements;
//   * each lane's partial dot products of the batch (one per key and row) are
//     summed across the warp by a transpose-reduction: at each of log2(KG)
//     exchange steps a lane keeps half of its values and adds the partner's
//     copy of them, so that after the plain steps that remain, lane l holds
//     the full score of key key_of(l) -- about one shuffle per key and row;
//   * base-2 online softmax with the running max moved (and the accumulator
//     rescaled) only when a batch's max exceeds it by more than 2^8; the
//     probabilities times the v scale are broadcast back by shuffles and
//     accumulated into each lane's slice of O.
// Rows past the item's count and keys past its end or the causal bound
// (verify token t sees keys j <= L - T + t) weigh zero.  The item writes the
// final bf16 output and natural-log LSE (an unsplit sequence) or its
// normalised fp32 partial and LSE for the combine.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <math.h>

#include "va_internal.h"

namespace va {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr float kRescaleLog2 = 8.0f;

__host__ __device__ constexpr int elem_bits(int dt) {
    return dt == VA_BF16 ? 16 : dt == VA_INT4 ? 4 : dt == VA_INT2 ? 2 : 8;
}

// A lane's slice of one cache row: LB = (D / 32) * bits bits, loaded as the
// narrowest aligned unit that holds it.  Slices of 4 bits (2-bit codes at
// D = 64) share a byte between two lanes.
template <int LB>
struct Slice {
    static constexpr int kWords = LB >= 32 ? LB / 32 : 1;
    uint32_t w[kWords];
    __device__ __forceinline__ void load(const uint8_t *row, int lane) {
        if constexpr (LB == 128) {
            const uint4 v = __ldg(reinterpret_cast<const uint4 *>(row) + lane);
            w[0] = v.x, w[1] = v.y, w[2] = v.z, w[3] = v.w;
        } else if constexpr (LB == 64) {
            const uint2 v = __ldg(reinterpret_cast<const uint2 *>(row) + lane);
            w[0] = v.x, w[1] = v.y;
        } else if constexpr (LB == 32) {
            w[0] = __ldg(reinterpret_cast<const uint32_t *>(row) + lane);
        } else if constexpr (LB == 16) {
            w[0] = __ldg(reinterpret_cast<const uint16_t *>(row) + lane);
        } else if constexpr (LB == 8) {
            w[0] = __ldg(row + lane);
        } else {
            static_assert(LB == 4, "slice width");
            w[0] = (uint32_t)__ldg(row + (lane >> 1)) >> (4 * (lane & 1));
        }
    }
    __device__ __forceinline__ void zero() {
#pragma unroll
        for (int i = 0; i < kWords; ++i) w[i] = 0u;
    }
};

// Packed fp32 pairs (sm_100+): each half of fma/add/mul.f32x2 is one
// IEEE-rounded fp32 operation, the same result as the scalar instruction, at
// half the issue cost.
__device__ __forceinline__ uint64_t pk2(uint32_t lo, uint32_t hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
    return r;
}
__device__ __forceinline__ uint64_t pk2f(float lo, float hi) { return pk2(__float_as_uint(lo), __float_as_uint(hi)); }
__device__ __forceinline__ float2 upk2(uint64_t r) {
    uint32_t lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=r"(lo), "=r"(hi) : "l"(r));
    return make_float2(__uint_as_float(lo), __uint_as_float(hi));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// The slice's EL codes as EL / 2 exact fp32 pairs (elements 2i, 2i + 1), the
// codes themselves, not yet scaled.  Integers: a code c with offset
// u = c + 2^(b-1) in [0, 2^b) is placed in the low mantissa bits of 2^23 (u
// XOR-ed into 0x4B000000 | 2^(b-1) flips the sign bit of the two's-complement
// field into that offset), and 2^23 plus the offset is subtracted with one
// paired add: both steps are exact.  bf16 is a shift; fp8-e4m3 goes through
// the hardware's exact conversion to fp16.
template <int DT, int EL>
__device__ __forceinline__ void decode2(const uint32_t *w, uint64_t *f) {
    if constexpr (DT == VA_BF16) {
#pragma unroll
        for (int i = 0; i < EL / 2; ++i) f[i] = pk2(w[i] << 16, w[i] & 0xFFFF0000u);
    } else if constexpr (DT == VA_INT8) {
        const uint64_t off = pk2f(-8388736.0f, -8388736.0f);
#pragma unroll
        for (int i = 0; i < EL / 2; ++i) {
            const uint32_t x = w[i / 2] ^ 0x80808080u;
            const int k = 2 * (i % 2);
            f[i] = add2(pk2(__byte_perm(x, 0x4B000000u, 0x7440 + k), __byte_perm(x, 0x4B000000u, 0x7441 + k)), off);
        }
    } else if constexpr (DT == VA_INT4) {
        const uint64_t off = pk2f(-8388616.0f, -8388616.0f);
#pragma unroll
        for (int i = 0; i < EL / 2; ++i) {
            const uint32_t x = w[i / 4] >> (8 * (i % 4));
            f[i] = add2(pk2((x & 0xFu) ^ 0x4B000008u, ((x >> 4) & 0xFu) ^ 0x4B000008u), off);
        }
    } else if constexpr (DT == VA_INT2) {
        const uint64_t off = pk2f(-8388610.0f, -8388610.0f);
#pragma unroll
        for (int i = 0; i < EL / 2; ++i) {
            const uint32_t x = w[i / 8] >> (4 * (i % 8));
            f[i] = add2(pk2((x & 0x3u) ^ 0x4B000002u, ((x >> 2) & 0x3u) ^ 0x4B000002u), off);
        }
    } else {  // fp8-e4m3
#pragma unroll
        for (int i = 0; i < EL / 2; ++i) {
            const uint32_t x = w[i / 2] >> (16 * (i % 2));
            __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(x & 0xFFFFu), __NV_E4M3);
            const float2 v = __half22float2(*reinterpret_cast<__half2 *>(&h));
            f[i] = pk2f(v.x, v.y);
        }
    }
}

// The same codes as plain fp32 values, one subtract per element: the form the
// one-row kernel uses (it is bound by memory, and the pair form's extra
// combining add per key costs it more than the paired arithmetic saves).
template <int DT, int EL>
__device__ __forceinline__ void decode(const uint32_t *w, float *f) {
    if constexpr (DT == VA_BF16) {
#pragma unroll
        for (int e = 0; e < EL; ++e) {
            const uint32_t x = w[e / 2];
            f[e] = __uint_as_float((e & 1) ? (x & 0xFFFF0000u) : (x << 16));
        }
    } else if constexpr (DT == VA_INT8) {
#pragma unroll
        for (int i = 0; i < (EL + 3) / 4; ++i) {
            const uint32_t x = w[i] ^ 0x80808080u;
#pragma unroll
            for (int k = 0; k < 4; ++k)
                if (4 * i + k < EL)
                    f[4 * i + k] = __uint_as_float(__byte_perm(x, 0x4B000000u, 0x7440 + k)) - 8388736.0f;
        }
    } else if constexpr (DT == VA_INT4) {
#pragma unroll
        for (int e = 0; e < EL; ++e)
            f[e] = __uint_as_float(((w[e / 8] >> (4 * (e % 8))) & 0xFu) ^ 0x4B000008u) - 8388616.0f;
    } else if constexpr (DT == VA_INT2) {
#pragma unroll
        for (int e = 0; e < EL; ++e)
            f[e] = __uint_as_float(((w[e / 16] >> (2 * (e % 16))) & 0x3u) ^ 0x4B000002u) - 8388610.0f;
    } else {  // fp8-e4m3
#pragma unroll
        for (int i = 0; i < (EL + 1) / 2; ++i) {
            const uint32_t x = w[i / 2] >> (16 * (i % 2));
            __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(x & 0xFFFFu), __NV_E4M3);
            const float2 v = __half22float2(*reinterpret_cast<__half2 *>(&h));
            f[2 * i] = v.x;
            if (2 * i + 1 < EL) f[2 * i + 1] = v.y;
        }
    }
}

// One-row kernel: the codes as scalars, with the offsets removed by paired
// adds for the packed caches (measured -3 % there) and by scalar subtracts
// otherwise (int8 +2.5 % with pairs).
template <int DT, int EL>
__device__ __forceinline__ void decode_one_row(const uint32_t *w, float *f) {
    if constexpr (DT == VA_INT4 || DT == VA_INT2) {
        uint64_t f2[EL / 2];
        decode2<DT, EL>(w, f2);
#pragma unroll
        for (int i = 0; i < EL / 2; ++i) {
            const float2 v = upk2(f2[i]);
            f[2 * i] = v.x;
            f[2 * i + 1] = v.y;
        }
    } else {
        decode<DT, EL>(w, f);
    }
}

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint16_t float_to_bf16_bits(float f) {
    __nv_bfloat16 h = __float2bfloat16_rn(f);
    return *reinterpret_cast<uint16_t *>(&h);
}

template <int KG>
struct KeyBits {
    static constexpr int value = KG == 16 ? 4 : KG == 8 ? 3 : KG == 4 ? 2 : 1;
};

// Transpose-reduction of KG values per lane over the warp: afterwards every
// lane's v[0] is the warp-wide sum of value key_of_lane(lane), whose bits are
// lane bits 4, 3, ... (most significant first, log2(KG) of them).
template <int KG>
__device__ __forceinline__ void transpose_reduce(float (&v)[KG], int lane) {
    constexpr int kB = KeyBits<KG>::value;
#pragma unroll
    for (int step = 0; step < 5; ++step) {
        const int o = 16 >> step;
        if (step < kB) {
            const int half = KG >> (step + 1);
            const bool upper = (lane & o) != 0;
#pragma unroll
            for (int i = 0; i < KG / 2; ++i) {
                if (i < half) {
                    const float send = upper ? v[i] : v[i + half];
                    const float keep = upper ? v[i + half] : v[i];
                    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
                }
            }
        } else {
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
        }
    }
}

template <int KG>
__device__ __forceinline__ int key_of_lane(int lane) {
    return (lane >> (5 - KeyBits<KG>::value)) & (KG - 1);
}

template <int KG>
__device__ __forceinline__ int lane_of_key(int k) {
    return k << (5 - KeyBits<KG>::value);
}

// Maximum over the batch's keys (the lanes of one key hold the same value).
template <int KG>
__device__ __forceinline__ float key_max(float v) {
#pragma unroll
    for (int i = 0; i < KeyBits<KG>::value; ++i) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16 >> i));
    return v;
}

template <int D, int DT, int RPI>
struct Geometry {
    static constexpr int EL = D / 32;                   // elements of a row per lane
    static constexpr int LB = EL * elem_bits(DT);       // bits of a row per lane
    static constexpr int ROWB = D * elem_bits(DT) / 8;  // bytes per cache row
    // keys per batch: 16 (more bytes in flight per warp) where the registers
    // allow it without spills -- one row, and two rows of fp8 or packed codes
    // (measured at two rows: fp8 -8 %, int4 -4 %; int8 and bf16 spill, +5-7 %)
    static constexpr int KG =
        (RPI == 1 || (RPI == 2 && (DT == VA_FP8_E4M3 || DT == VA_INT4 || DT == VA_INT2))) ? 16 : 8;
};

template <int D, int DT, int RPI>
__global__ void __launch_bounds__(kThreads, warp_ctas_per_sm(DT, RPI)) warp_partial_kernel(const PartialParams p) {
    using Gm = Geometry<D, DT, RPI>;
    constexpr int EL = Gm::EL, KG = Gm::KG;
    constexpr bool kQuant = DT != VA_BF16;
    static_assert(VA_PAGE_SIZE % KG == 0 && kWarpTile % KG == 0, "a batch lies inside one page");
    __shared__ float sm_m[kWarps][RPI], sm_l[kWarps][RPI];
    __shared__ float sm_o[kWarps][RPI][D];

    // programmatic dependent launch: nothing of the caller's is touched before this
    griddep_wait();
    const Item it = p.items[blockIdx.x];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = p.G, T = p.T, Hkv = p.Hkv;
    const int row0 = it.rg * p.rows_per_group;
    const int nrows = min(p.rows_per_group, p.R - row0);
    if (tid == 0 && p.seq_lens[it.b] != it.L) atomicOr(p.flags, kFlagSeqLenMismatch);

    // this lane's slice of the item's q rows, times log2(e) / sqrt(D)
    float q[RPI][EL];
    int last_visible[RPI];
#pragma unroll
    for (int r = 0; r < RPI; ++r) {
        last_visible[r] = -1;  // padding rows see nothing
#pragma unroll
        for (int e = 0; e < EL; ++e) q[r][e] = 0.f;
        if (r < nrows) {
            const int rr = row0 + r;
            const int t = rr / G, h = it.kvh * G + rr % G;
            const uint16_t *qrow = p.q + ((size_t)(it.b * T + t) * p.Hq + h) * D + lane * EL;
#pragma unroll
            for (int e = 0; e < EL; ++e) q[r][e] = __uint_as_float((uint32_t)__ldg(qrow + e) << 16) * p.sm_scale_log2;
            last_visible[r] = it.L - T + t;
        }
    }

    uint64_t q2[RPI][EL / 2];  // q as fp32 pairs
    float m_run[RPI], l_run[RPI];
    uint64_t acc[RPI][EL / 2];  // this lane's slice of O as fp32 pairs
#pragma unroll
    for (int r = 0; r < RPI; ++r) {
        m_run[r] = -INFINITY;
        l_run[r] = 0.f;
#pragma unroll
        for (int i = 0; i < EL / 2; ++i) {
            q2[r][i] = pk2f(q[r][2 * i], q[r][2 * i + 1]);
            acc[r][i] = 0ull;  // (+0.0f, +0.0f)
        }
    }

    const uint8_t *kbase = static_cast<const uint8_t *>(p.k_pages);
    const uint8_t *vbase = static_cast<const uint8_t *>(p.v_pages);
    const int32_t *bt = p.block_table + (size_t)it.b * p.bt_stride;
    const int my_key = key_of_lane<KG>(lane);
    const bool key_owner = (lane & ((32 / KG) - 1)) == 0;  // one lane per key adds to l
    const int nbatch = (it.k_end - it.k_begin + KG - 1) / KG;

    // Batches are dealt to the warps round-robin; every batch lies inside one
    // 16-token page (items start at multiples of the 32-key split tile).
    for (int bi = warp; bi < nbatch; bi += kWarps) {
        const int j0 = it.k_begin + bi * KG;
        int page = __ldg(bt + j0 / VA_PAGE_SIZE);
        bool page_ok = true;
        if (p.num_pages > 0 && (page < 0 || page >= p.num_pages)) {
            if (lane == 0) atomicOr(p.flags, kFlagBadPage);
            page_ok = false;
            page = 0;  // not read: the batch's keys are all masked below
        }
        const size_t row_first = ((size_t)page * VA_PAGE_SIZE + j0 % VA_PAGE_SIZE) * Hkv + it.kvh;
        const int nvalid = page_ok ? min(KG, it.k_end - j0) : 0;

        // every load of the batch first: KG key slices, KG value slices, the
        // scales of this lane's key
        Slice<Gm::LB> k_raw[KG], v_raw[KG];
#pragma unroll
        for (int k = 0; k < KG; ++k) {
            if (k < nvalid) {
                const size_t row = row_first + (size_t)k * Hkv;
                k_raw[k].load(kbase + row * Gm::ROWB, lane);
                v_raw[k].load(vbase + row * Gm::ROWB, lane);
            } else {
                k_raw[k].zero();
                v_raw[k].zero();
            }
        }
        float kscale = 1.f, vscale = 1.f;
        if (kQuant && my_key < nvalid) {
            const size_t row = row_first + (size_t)my_key * Hkv;
            kscale = __ldg(p.k_scale + row);
            vscale = __ldg(p.v_scale + row);
        }

        // scores: this lane's partial dot products, then the transpose-reduction
        float s[RPI];
        {
            float part[RPI][KG];
#pragma unroll
            for (int k = 0; k < KG; ++k) {
                if constexpr (RPI == 1) {
                    float f[EL];
                    decode_one_row<DT, EL>(k_raw[k].w, f);
                    float a = 0.f;
#pragma unroll
                    for (int e = 0; e < EL; ++e) a = fmaf(q[0][e], f[e], a);
                    part[0][k] = a;
                } else {
                    uint64_t f[EL / 2];
                    decode2<DT, EL>(k_raw[k].w, f);
#pragma unroll
                    for (int r = 0; r < RPI; ++r) {
                        uint64_t a = 0ull;
#pragma unroll
                        for (int i = 0; i < EL / 2; ++i) a = fma2(q2[r][i], f[i], a);
                        const float2 h = upk2(a);
                        part[r][k] = h.x + h.y;
                    }
                }
            }
#pragma unroll
            for (int r = 0; r < RPI; ++r) {
                transpose_reduce<KG>(part[r], lane);
                const bool vis = my_key < nvalid && j0 + my_key <= last_visible[r];
                s[r] = vis ? part[r][0] * kscale : -INFINITY;
            }
        }

        // online softmax per row, then P x V into this lane's slice of O
        float pv[RPI];
#pragma unroll
        for (int r = 0; r < RPI; ++r) {
            const float bmax = key_max<KG>(s[r]);
            if (bmax > m_run[r] + kRescaleLog2) {  // uniform across the warp
                const float alpha = m_run[r] == -INFINITY ? 0.f : ex2_approx(m_run[r] - bmax);
                m_run[r] = bmax;
                l_run[r] *= alpha;
                const uint64_t a2 = pk2f(alpha, alpha);
#pragma unroll
                for (int i = 0; i < EL / 2; ++i) acc[r][i] = mul2(acc[r][i], a2);
            }
            const float pr = s[r] == -INFINITY ? 0.f : ex2_approx(s[r] - m_run[r]);
            if (key_owner) l_run[r] += pr;
            pv[r] = pr * vscale;
        }
#pragma unroll
        for (int k = 0; k < KG; ++k) {
            if constexpr (RPI == 1) {
                float f[EL];
                decode_one_row<DT, EL>(v_raw[k].w, f);
                const float w = __shfl_sync(0xffffffffu, pv[0], lane_of_key<KG>(k));
#pragma unroll
                for (int i = 0; i < EL / 2; ++i) {
                    const float2 o = upk2(acc[0][i]);
                    acc[0][i] = pk2f(fmaf(w, f[2 * i], o.x), fmaf(w, f[2 * i + 1], o.y));
                }
            } else {
                uint64_t f[EL / 2];
                decode2<DT, EL>(v_raw[k].w, f);
#pragma unroll
                for (int r = 0; r < RPI; ++r) {
                    const float w = __shfl_sync(0xffffffffu, pv[r], lane_of_key<KG>(k));
                    const uint64_t w2 = pk2f(w, w);
#pragma unroll
                    for (int i = 0; i < EL / 2; ++i) acc[r][i] = fma2(w2, f[i], acc[r][i]);
                }
            }
        }
    }

    // merge the four warps' states: O = sum_w 2^(m_w - M) O_w / sum_w 2^(m_w - M) l_w
#pragma unroll
    for (int r = 0; r < RPI; ++r) {
        float l = l_run[r];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
        if (lane == 0) {
            sm_m[warp][r] = m_run[r];
            sm_l[warp][r] = l;
        }
#pragma unroll
        for (int i = 0; i < EL / 2; ++i) {
            const float2 o = upk2(acc[r][i]);
            sm_o[warp][r][lane * EL + 2 * i] = o.x;
            sm_o[warp][r][lane * EL + 2 * i + 1] = o.y;
        }
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < RPI; ++r) {
        if (r >= nrows) break;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm_m[w][r]);
        float wgt[kWarps], L = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            wgt[w] = sm_m[w][r] == -INFINITY ? 0.f : exp2f(sm_m[w][r] - M);
            L += wgt[w] * sm_l[w][r];
        }
        const float inv = L > 0.f ? 1.f / L : 0.f;
        const float lse_nat = L > 0.f ? (M + log2f(L)) * 0.69314718055994531f : -INFINITY;
        const int rr = row0 + r;
        const int t = rr / G, h = it.kvh * G + rr % G;
        const size_t orow = (size_t)(it.b * T + t) * p.Hq + h;
        const size_t prow = (size_t)it.part * p.rows_per_group + r;
        for (int d = tid; d < D; d += kThreads) {
            float o = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) o = fmaf(wgt[w], sm_o[w][r][d], o);
            o *= inv;
            if (it.part < 0)
                p.out[orow * D + d] = float_to_bf16_bits(o);
            else
                p.o_part[prow * D + d] = o;
        }
        if (tid == 0) {
            if (it.part < 0) {
                if (p.lse) p.lse[orow] = lse_nat;
            } else {
                p.lse_part[prow] = lse_nat;
            }
        }
    }
}

template <int D, int DT, int RPI>
cudaError_t launch_one(const PartialParams &p, int n, cudaStream_t s) {
    return launch_pdl(warp_partial_kernel<D, DT, RPI>, dim3(n), dim3(kThreads), 0, s, p);
}

template <int D, int DT>
cudaError_t launch_rows(const PartialParams &p, int n, cudaStream_t s) {
    switch (warp_rows_variant(p.rows_per_group)) {
    case 1: return launch_one<D, DT, 1>(p, n, s);
    case 2: return launch_one<D, DT, 2>(p, n, s);
    default: return launch_one<D, DT, 4>(p, n, s);
    }
}

template <int D>
cudaError_t launch_d(const PartialParams &p, int dtype, int n, cudaStream_t s) {
    switch (dtype) {
    case VA_BF16: return launch_rows<D, VA_BF16>(p, n, s);
    case VA_FP8_E4M3: return launch_rows<D, VA_FP8_E4M3>(p, n, s);
    case VA_INT8: return launch_rows<D, VA_INT8>(p, n, s);
    case VA_INT4: return launch_rows<D, VA_INT4>(p, n, s);
    default: return launch_rows<D, VA_INT2>(p, n, s);
    }
}

}  // namespace

cudaError_t launch_warp_partial(const PartialParams &p, int head_dim, int kv_dtype, int n,
                                cudaStream_t s) {
    if (n <= 0) return cudaSuccess;
    if (p.rows_per_group > kWarpRows) return cudaErrorInvalidValue;
    switch (head_dim) {
    case 64: return launch_d<64>(p, kv_dtype, n, s);
    case 128: return launch_d<128>(p, kv_dtype, n, s);
    default: return launch_d<256>(p, kv_dtype, n, s);
    }
}

}  // namespace va
