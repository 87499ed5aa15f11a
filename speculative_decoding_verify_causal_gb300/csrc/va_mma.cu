// Tensor-core partial-attention kernel for sm_103a (tcgen05 + TMEM + TMA).
//
// One CTA = one work item: the G*T packed query rows of one kv head of one
// sequence (padded to the 128-row MMA tile) against one split of the paged
// KV cache ("I pushed Qwen3.8-27B to 124 tps on a single request on a RTX
// 3090", bullet "Split-KV attention kernel for the verify step").  Packing
// all rows that share a kv head into the M dimension is the GB300 form of the
// idea in "Four Tesla V100s from 2017 matched my RTX 5090 on single-request
// Qwen 3.8 decode", section "What I actually built" (lay the verify rows onto
// the tensor instruction's row tile so the extra drafted tokens ride along
// almost for free); the same section's advice to leave the data compressed
// until the step before the tensor core is followed here: the cache stays 8-,
// 4- or 2-bit from HBM into shared memory and is expanded right before the
// MMA.
//
// Per 64-key tile (4 pages):
//   producer warp    stages the item's page ids, then TMA-gathers the pages
//                    named by the block table (4-D tensor map over [page,
//                    slot, kv head, d], one box per page) into a ring of raw
//                    stages, K then V of every tile (the first stage of each
//                    slot already during set-up);
//   dequant warps    (fp8-e4m3 / int8 / int4 / int2) two groups of four, one
//                    taking the K tile and one the V tile of every tile: a raw
//                    stage goes to registers and back to the producer, then
//                    fp16 -- every conversion is exact -- into the 128-byte-swizzled
//                    layout the MMA reads; the K group also carries each
//                    key's k and v scale (loaded two tiles ahead) into a ring
//                    the softmax reads (bf16 caches are TMA'd straight into
//                    the MMA layout);
//   MMA warp         one thread issues S = Q K^T (A = Q in TMEM, B = K tile in
//                    shared memory, D = S in TMEM, M=128 N=64 K=16 x D/16) and
//                    O += P V (A = P in TMEM, B = V tile, N = D);
//   softmax warps    two per TMEM lane quarter (one thread per packed row and
//                    half of the tile's keys): read S from TMEM, apply the
//                    per-key k scale and the bottom-right causal mask, keep the
//                    running max / sum (base 2; the max is only moved, and O
//                    rescaled, when it grows by more than 2^8), write
//                    P * v_scale * 2^beta (fp16) back over S in TMEM, and at
//                    the end write O / (l 2^beta) and the log-sum-exp (split
//                    partials leave by TMA box stores).  2^beta is a power of
//                    two chosen from each tile's largest v scale (kept while it
//                    still fits), so that P * v_scale stays in fp16's normal
//                    range for value rows of any magnitude; it is folded into
//                    the exponent, so it costs no multiply.
// Scales are constant along head_dim, so dequantisation is an exact cast
// and the scales are folded into the scores (k) and into P (v).
//
// Every wait on an mbarrier gives up after 2 s, records kFlagTimeout and
// unwinds; nothing spins forever.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <math.h>

#include <cstring>
#include <mutex>

#include "va_internal.h"
#include "va_sm100.cuh"

namespace va {
namespace {

using namespace sm100;

constexpr int kTile = kMmaTile;     // keys per S tile (MMA N)
constexpr int kMaxRawStages = 6;    // raw (as cached) stages: one 64-key K or V tile each
constexpr int kMinRawStages = 3;
constexpr int kBfStages = 3;        // bf16: 64-key stages TMA'd straight into MMA layout
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr float kRescaleLog2 = 8.0f;
constexpr int kScaleRing = 4;       // per-tile k/v scales handed to the softmax warps
constexpr int kRingFloats = 2 * kTile + 4;  // one ring slot: k[64], v[64], largest v scale of each half, pad
constexpr int kMaxItemPages = kMmaMaxItemTokens / VA_PAGE_SIZE;  // page ids staged in smem
constexpr int kSetupBar = 10;       // named barrier: set-up done (producer arrives, the rest wait)

enum : int { kFlagTimeout = 4 };

struct MmaParams {
    CUtensorMap tm_k;  // 64-byte aligned members first
    CUtensorMap tm_v;
    CUtensorMap tm_o;  // split partials o_part as [num_parts * rows_per_group, D] fp32 (unused if none)
    PartialParams p;
    int raw_stages;    // quantised caches: stages of the raw ring (fits the smem budget)
};

template <int D, int DT>
struct Cfg {
    static constexpr bool kQuant = DT != VA_BF16;
    static constexpr int kNumBuf = kQuant ? 2 : (D == 256 ? 2 : kBfStages);  // 64 KB bf16 stages at D = 256
    static constexpr int kConvBytes = kTile * D * 2;   // K or V tile, 16-bit, SW128 chunks of 64 d
    static constexpr int kChunkBytes = kTile * 128;    // one 64-d chunk of a tile
    static constexpr int kBits = DT == VA_BF16 ? 16 : DT == VA_INT4 ? 4 : DT == VA_INT2 ? 2 : 8;
    static constexpr int kRowBytes = D * kBits / 8;    // one cached row (token, kv head)
    static constexpr int kRawTileBytes = kTile * kRowBytes;  // one K or V tile as cached
    // warps 0-7 softmax (two per TMEM lane quarter), 8-15 dequant (quantised
    // caches only: 8-11 K, 12-15 V), then the producer and the MMA issuer
    static constexpr int kSoftmaxWarps = 8;
    static constexpr int kDequantWarps = kQuant ? 8 : 0;
    static constexpr int kProducerWarp = kSoftmaxWarps + kDequantWarps;
    static constexpr int kMmaWarp = kProducerWarp + 1;
    static constexpr int kWarps = kMmaWarp + 1;
    static constexpr int kThreads = kWarps * 32;
    static constexpr uint32_t kQCol = 0;
    static constexpr uint32_t kOCol = D / 2;
    static constexpr uint32_t kSCol = D / 2 + D;
    static constexpr uint32_t kTmemCols = 512;
};

// Shared memory carve-up (byte offsets from a 1024-aligned base).  The raw
// ring (quantised caches) holds one pass per stage, in the order the dequant
// warps consume them: K of tile 0, V of tile 0, K of tile 1, ...
template <int D, int DT>
struct Smem {
    using C = Cfg<D, DT>;
    uint32_t conv_k, conv_v;         // kNumBuf buffers each
    uint32_t raw, raw_stride;        // raw stages
    uint32_t pids;                   // the item's page ids (kMaxItemPages ints)
    uint32_t scale_ring;             // kScaleRing slots of kRingFloats
    uint32_t xchg;                   // softmax pair exchange: [2][2][128] maxima + [2][128] sums
    uint32_t bars;                   // mbarriers
    uint32_t total;
    __host__ __device__ Smem(int Hkv, int nst) {
        conv_k = 0;
        conv_v = conv_k + C::kNumBuf * C::kConvBytes;
        raw = conv_v + C::kNumBuf * C::kConvBytes;
        (void)Hkv;
        raw_stride = C::kQuant ? C::kRawTileBytes : 0;
        pids = raw + (C::kQuant ? nst * raw_stride : 0);
        scale_ring = pids + kMaxItemPages * 4;
        xchg = scale_ring + (C::kQuant ? kScaleRing * kRingFloats * 4 : 0);
        bars = xchg + 6 * 128 * 4;
        total = bars + 64 * 8 + 16;
    }
};

// Barrier slots (8 bytes each) inside Smem::bars.
enum Bar : int {
    kRawFull = 0,                          // kMaxRawStages
    kRawEmpty = kRawFull + kMaxRawStages,  // kMaxRawStages
    kKFull = kRawEmpty + kMaxRawStages,    // kNumBuf (<= 3)
    kKEmpty = kKFull + 3,
    kVFull = kKEmpty + 3,
    kVEmpty = kVFull + 3,
    kSFull = kVEmpty + 3,               // 2
    kPFull = kSFull + 2,                // 2
    kPEmpty = kPFull + 2,               // 2
    kODone = kPEmpty + 2,
    kOFinal = kODone + 1,
    kQReady = kOFinal + 1,
    kRingFree = kQReady + 1,            // kScaleRing: the softmax has read a tile's scales
    kNumBars = kRingFree + kScaleRing,
};

static_assert(kNumBars <= 64, "the barrier block holds 64 mbarriers");

__device__ __forceinline__ float bf16_bits_to_float(uint32_t b) { return __uint_as_float(b << 16); }

// 2^x with the hardware approximation (relative error ~2^-22; -inf -> +0).
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Packed fp32 pairs (sm_100+): each lane of a pair is one IEEE-rounded fp32
// multiply / fused multiply-add / add, the same result as the scalar
// instruction, at half the issue cost.
__device__ __forceinline__ uint64_t f2_pack(uint32_t lo, uint32_t hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
    return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t r, uint32_t &lo, uint32_t &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=r"(lo), "=r"(hi) : "l"(r));
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
// max of three (one instruction on sm_100+)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ uint32_t pack_bf162(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

// int8 -> fp16, exact: bias each byte to u = b + 128, place it in the low
// mantissa bits of 1024.0 (0x6400 | u = 1024 + u) and subtract 1152.  This is
// the published "magic number" integer-to-float conversion (e.g. Kim et al.,
// "Who Says Elephants Can't Run", 2022); here it is written out for 4 bytes.
__device__ __forceinline__ void int8x4_to_half2x2(uint32_t w, uint32_t &lo, uint32_t &hi) {
    const uint32_t x = w ^ 0x80808080u;
    uint32_t a, b;
    asm("prmt.b32 %0, %1, %2, 0x4140;" : "=r"(a) : "r"(x), "r"(0x64646464u));
    asm("prmt.b32 %0, %1, %2, 0x4342;" : "=r"(b) : "r"(x), "r"(0x64646464u));
    const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));  // 1152
    __half2 ha = __hsub2(*reinterpret_cast<__half2 *>(&a), bias);
    __half2 hb = __hsub2(*reinterpret_cast<__half2 *>(&b), bias);
    lo = *reinterpret_cast<uint32_t *>(&ha);
    hi = *reinterpret_cast<uint32_t *>(&hb);
}

__device__ __forceinline__ void e4m3x4_to_half2x2(uint32_t w, uint32_t &lo, uint32_t &hi) {
    __half2_raw a = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w & 0xFFFFu), __NV_E4M3);
    __half2_raw b = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w >> 16), __NV_E4M3);
    lo = *reinterpret_cast<uint32_t *>(&a);
    hi = *reinterpret_cast<uint32_t *>(&b);
}

// 4-bit codes -> fp16, exact, the same magic-number idea: code k of w sits in
// bits [4k, 4k + 4); a nibble n of a two's-complement code c has n ^ 8 = c + 8
// in [0, 16), so (n ^ 8) | 0x6400 is the fp16 1024 + c + 8 and subtracting
// 1032 leaves c.  One mask-and-xor makes the pairs (c_s, c_s+4); byte
// permutes put them in element order.  h[j] = (c_2j, c_2j+1).
__device__ __forceinline__ void int4x8_to_half2x4(uint32_t w, uint32_t (&h)[4]) {
    uint32_t a[4];
#pragma unroll
    for (int s = 0; s < 4; ++s) a[s] = ((w >> (4 * s)) & 0x000F000Fu) ^ 0x64086408u;
    asm("prmt.b32 %0, %1, %2, 0x5410;" : "=r"(h[0]) : "r"(a[0]), "r"(a[1]));
    asm("prmt.b32 %0, %1, %2, 0x5410;" : "=r"(h[1]) : "r"(a[2]), "r"(a[3]));
    asm("prmt.b32 %0, %1, %2, 0x7632;" : "=r"(h[2]) : "r"(a[0]), "r"(a[1]));
    asm("prmt.b32 %0, %1, %2, 0x7632;" : "=r"(h[3]) : "r"(a[2]), "r"(a[3]));
    const __half2 bias = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));  // 1032
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        __half2 v = __hsub2(*reinterpret_cast<__half2 *>(&h[j]), bias);
        h[j] = *reinterpret_cast<uint32_t *>(&v);
    }
}

// 2-bit codes -> fp16, exact: code k of w in bits [2k, 2k + 2), (n ^ 2) = c + 2
// in [0, 4), bias 1026; pairs (c_s, c_s+8) permuted into element order.
__device__ __forceinline__ void int2x16_to_half2x8(uint32_t w, uint32_t (&h)[8]) {
    uint32_t a[8];
#pragma unroll
    for (int s = 0; s < 8; ++s) a[s] = ((w >> (2 * s)) & 0x00030003u) ^ 0x64026402u;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        asm("prmt.b32 %0, %1, %2, 0x5410;" : "=r"(h[j]) : "r"(a[2 * j]), "r"(a[2 * j + 1]));
        asm("prmt.b32 %0, %1, %2, 0x7632;" : "=r"(h[4 + j]) : "r"(a[2 * j]), "r"(a[2 * j + 1]));
    }
    const __half2 bias = __halves2half2(__ushort_as_half(0x6402), __ushort_as_half(0x6402));  // 1026
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        __half2 v = __hsub2(*reinterpret_cast<__half2 *>(&h[j]), bias);
        h[j] = *reinterpret_cast<uint32_t *>(&v);
    }
}

// The 16 elements of one raw piece of a quantised cache row -> 8 fp16 pairs
// in element order.  A piece is 16 / 8 / 4 bytes (8-bit / 4-bit / 2-bit).
template <int DT>
struct RawPiece {
    static constexpr int kWords = DT == VA_INT4 ? 2 : DT == VA_INT2 ? 1 : 4;
    uint32_t w[kWords];
    __device__ __forceinline__ void load(uint32_t a) {
        if constexpr (kWords == 4) {
            const uint4 v = lds_u4(a);
            w[0] = v.x, w[1] = v.y, w[2] = v.z, w[3] = v.w;
        } else if constexpr (kWords == 2) {
            const uint2 v = lds_u2(a);
            w[0] = v.x, w[1] = v.y;
        } else {
            w[0] = lds_u32(a);
        }
    }
    __device__ __forceinline__ void to_half(uint32_t (&hw)[8]) const {
        if constexpr (DT == VA_INT2) {
            int2x16_to_half2x8(w[0], hw);
        } else if constexpr (DT == VA_INT4) {
            uint32_t a[4], b[4];
            int4x8_to_half2x4(w[0], a);
            int4x8_to_half2x4(w[1], b);
#pragma unroll
            for (int j = 0; j < 4; ++j) hw[j] = a[j], hw[4 + j] = b[j];
        } else {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                if constexpr (DT == VA_INT8)
                    int8x4_to_half2x2(w[k], hw[2 * k], hw[2 * k + 1]);
                else
                    e4m3x4_to_half2x2(w[k], hw[2 * k], hw[2 * k + 1]);
            }
        }
    }
};

// Byte offset of 16-byte unit u (0..7) of tile row `row` inside a 64-d chunk
// of a 128-byte-swizzled tile (rows of 128 bytes, 8-row / 1024-byte atoms).
__device__ __forceinline__ uint32_t sw128(int row, int u) { return row * 128 + ((u ^ (row & 7)) << 4); }

template <int D, int DT>
__global__ void __launch_bounds__(Cfg<D, DT>::kThreads, 1)
mma_partial_kernel(const __grid_constant__ MmaParams mp) {
    using C = Cfg<D, DT>;
    static_assert(2 * C::kNumBuf * C::kConvBytes >= (D / 32) * kMmaRows * 128, "fp32 staging fits the tile buffers");
    const PartialParams &p = mp.p;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int nst = C::kQuant ? mp.raw_stages : 1;  // raw stages (quantised caches only)
    const Smem<D, DT> L(p.Hkv, nst);
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + L.bars;
    auto bar = [&](int i) { return bar0 + 8u * i; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L.bars + kNumBars * 8);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // Programmatic dependent launch: the launch may overlap the previous
    // kernel's tail; wait for it (it may have written the inputs or the work
    // list) before any load.  No early trigger for the next kernel: the
    // combine would only take SMs from this grid's tail (measured slower).
    griddep_wait();
    const Item it = p.items[blockIdx.x];
    const int G = p.G, T = p.T, Hkv = p.Hkv;
    const int row0 = it.rg * p.rows_per_group;
    const int nrows = min(p.rows_per_group, p.R - row0);
    const int nkeys = it.k_end - it.k_begin;
    const int ntiles = (nkeys + kTile - 1) / kTile;
    const int32_t *bt = p.block_table + (size_t)it.b * p.bt_stride;

    const int lp0 = it.k_begin / VA_PAGE_SIZE;                               // first logical page
    const int npages_item = (it.k_end + VA_PAGE_SIZE - 1) / VA_PAGE_SIZE - lp0;
    // producer: lane pg < 4 issues the TMA box of page pg of a tile (page ids
    // from shared memory, 0 past the end); one raw stage per K or V pass
    auto tile_page = [&](int i) -> int {
        const int k = i * (kTile / VA_PAGE_SIZE) + lane;
        return (lane < kTile / VA_PAGE_SIZE && k < npages_item) ? (int)lds_u32(sbase + L.pids + 4u * k) : 0;
    };
    auto tile_npg = [&](int i) { return min(kTile / VA_PAGE_SIZE, npages_item - i * (kTile / VA_PAGE_SIZE)); };
    auto issue_raw = [&](int ps) {
        const int slot = ps % nst, i = ps >> 1, kv = ps & 1;
        const int npg = tile_npg(i);
        const int page = tile_page(i);
        const uint32_t page_bytes = VA_PAGE_SIZE * C::kRowBytes;  // one page, one head, as cached
        if (lane == 0) mbar_arrive_expect_tx(bar(kRawFull + slot), npg * page_bytes);
        __syncwarp();
        if (lane < npg)
            tma_load_4d(sbase + L.raw + slot * L.raw_stride + lane * page_bytes, kv == 0 ? &mp.tm_k : &mp.tm_v, 0,
                        it.kvh, 0, page, bar(kRawFull + slot));
        __syncwarp();
    };
    int pre_issued = 0;  // raw stages the producer issued during set-up
    if (warp == C::kProducerWarp) {
        // Set-up by the producer warp, which then arrives at the set-up
        // barrier without waiting for the others: its first copies go out
        // while the other warps load Q and allocate TMEM.  The first page
        // ids are requested before anything else.
        int pg_first[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int k = 32 * j + lane;
            pg_first[j] = k < npages_item ? __ldg(bt + lp0 + k) : 0;
        }
        if (lane == 0) {
            prefetch_tensormap(&mp.tm_k);
            prefetch_tensormap(&mp.tm_v);
            for (int i = 0; i < kMaxRawStages; ++i) {
                mbar_init(bar(kRawFull + i), 1);
                mbar_init(bar(kRawEmpty + i), C::kQuant ? C::kDequantWarps / 2 : 1);  // one dequant group
            }
            for (int i = 0; i < 3; ++i) {
                mbar_init(bar(kKFull + i), C::kQuant ? C::kDequantWarps / 2 : 1);
                mbar_init(bar(kVFull + i), C::kQuant ? C::kDequantWarps / 2 : 1);
                mbar_init(bar(kKEmpty + i), 1);
                mbar_init(bar(kVEmpty + i), 1);
            }
            for (int i = 0; i < 2; ++i) {
                mbar_init(bar(kSFull + i), 1);                    // QK^T committed
                mbar_init(bar(kPFull + i), C::kSoftmaxWarps);     // softmax has written P
                mbar_init(bar(kPEmpty + i), 1);                   // P x V done: S/P buffer free
            }
            mbar_init(bar(kODone), 1);
            mbar_init(bar(kOFinal), 1);
            mbar_init(bar(kQReady), C::kSoftmaxWarps + C::kDequantWarps);
            for (int i = 0; i < kScaleRing; ++i) mbar_init(bar(kRingFree + i), C::kSoftmaxWarps);
            fence_barrier_init();
        }
        // the item's page ids -> smem (bad entries replaced by page 0 and
        // flagged); four loads per lane in flight at a time
        for (int k0 = 0; k0 < npages_item; k0 += 128) {
            int pg[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int k = k0 + 32 * j + lane;
                pg[j] = k0 == 0 ? pg_first[j] : (k < npages_item ? __ldg(bt + lp0 + k) : 0);
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int k = k0 + 32 * j + lane;
                if (k >= npages_item) continue;
                if (p.num_pages > 0 && (pg[j] < 0 || pg[j] >= p.num_pages)) {
                    atomicOr(p.flags, kFlagBadPage);
                    pg[j] = 0;
                }
                sts_u32(sbase + L.pids + 4u * k, (uint32_t)pg[j]);
            }
        }
        __syncwarp();
        named_bar_arrive(kSetupBar, C::kThreads);
        // the first stages (each slot's first use needs no wait) go out now,
        // while the other warps load Q
        if constexpr (C::kQuant) {
            pre_issued = min(nst, 2 * ntiles);
            for (int ps = 0; ps < pre_issued; ++ps) issue_raw(ps);
        }
    } else if (warp == C::kMmaWarp) {
        tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
        tmem_relinquish();
    }
    // Q rows are written to TMEM by the warps of each lane quarter: the two
    // softmax warps and (quantised caches) the two dequant warps of quarter
    // q = warp % 4 each take one part of the row's d range.  The loads are
    // issued now, one round trip overlapping the set-up.
    constexpr int kQParts = C::kQuant ? 4 : 2;
    constexpr int kQv = D / 8 / kQParts;  // 16-byte loads per part
    const bool q_warp = warp < C::kSoftmaxWarps + C::kDequantWarps;
    const int q_part = warp < C::kSoftmaxWarps ? (warp >> 2) : 2 + ((warp - C::kSoftmaxWarps) >> 2);
    uint4 qv[kQv];
    int t_r = 0;
    if (q_warp) {
        const int r = (warp & 3) * 32 + lane;
        if (r < nrows) {
            const int rr = row0 + r;
            t_r = rr / G;
            const int h = it.kvh * G + rr % G;
            const uint4 *qrow = reinterpret_cast<const uint4 *>(p.q + ((size_t)(it.b * T + t_r) * p.Hq + h) * D) +
                                q_part * kQv;
#pragma unroll
            for (int k = 0; k < kQv; ++k) qv[k] = __ldg(qrow + k);
        } else {
#pragma unroll
            for (int k = 0; k < kQv; ++k) qv[k] = make_uint4(0, 0, 0, 0);
        }
    }
    if (warp != C::kProducerWarp) {
        tc_fence_before();
        named_bar_sync(kSetupBar, C::kThreads);
        tc_fence_after();
    }
    const uint32_t tmem = warp == C::kProducerWarp ? 0u : *tmem_slot;
    bool ok = true;
    float q_prescale = 1.f;  // power of two folded into fp16 q (quantised caches)
    if (q_warp) {
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;
        const uint32_t lane_tm = tmem + ((uint32_t)(quarter * 32) << 16);
        const uint32_t xq = sbase + L.xchg;  // [part][128] row maxima
        if (C::kQuant) {
            float amax = 0.f;
#pragma unroll
            for (int k = 0; k < kQv; ++k) {
                const uint32_t w[4] = {qv[k].x, qv[k].y, qv[k].z, qv[k].w};
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    amax = fmaxf(amax, fmaxf(fabsf(bf16_bits_to_float(w[e] & 0xFFFFu)),
                                             fabsf(__uint_as_float(w[e] & 0xFFFF0000u))));
            }
            sts_f32(xq + 4u * (q_part * 128 + r), amax);
            named_bar_sync(5 + quarter, 32 * kQParts);
#pragma unroll
            for (int o = 0; o < kQParts; ++o) amax = fmaxf(amax, lds_f32(xq + 4u * (o * 128 + r)));
            named_bar_sync(5 + quarter, 32 * kQParts);  // the slots are reused by the softmax
            if (amax > 0.f) {
                int e;
                frexpf(amax, &e);                     // amax in [2^(e-1), 2^e)
                q_prescale = exp2f((float)(15 - e));  // amax * prescale in [2^14, 2^15): exact fp16
            }
        }
        // two bf16 -> one TMEM column; this part is columns [q_part * 4 kQv, +4 kQv)
        constexpr int kCols = 4 * kQv < 32 ? 4 * kQv : 32;
        const uint32_t qcol = lane_tm + C::kQCol + q_part * 4 * kQv;
#pragma unroll
        for (int c0 = 0; c0 < 4 * kQv; c0 += kCols) {
            uint32_t v[kCols];
#pragma unroll
            for (int k = 0; k < kCols / 4; ++k) {
                const uint4 x = qv[c0 / 4 + k];
                const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if (C::kQuant)
                        v[4 * k + e] = pack_half2(bf16_bits_to_float(w[e] & 0xFFFFu) * q_prescale,
                                                  __uint_as_float(w[e] & 0xFFFF0000u) * q_prescale);
                    else
                        v[4 * k + e] = w[e];
                }
            }
            if constexpr (kCols == 8)
                tmem_st8(qcol + c0, *reinterpret_cast<uint32_t(*)[8]>(&v[0]));
            else if constexpr (kCols == 16)
                tmem_st16(qcol + c0, *reinterpret_cast<uint32_t(*)[16]>(&v[0]));
            else
                tmem_st32(qcol + c0, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kQReady));
    }

    if (warp == C::kProducerWarp) {
        // ------------------------------------------------------------ producer
        // The whole warp walks the stages (K and V of every tile) after the
        // ones issued during set-up, each once the dequant group has handed
        // its slot back.
        if constexpr (C::kQuant) {
            const int npass = 2 * ntiles;
            int issued = pre_issued;
            for (int ps = pre_issued; ps < npass; ++ps) {
                const int slot = ps % nst, use = ps / nst;  // use >= 1 here
                ok = __shfl_sync(0xffffffffu, (int)mbar_wait(bar(kRawEmpty + slot), (use & 1) ^ 1, kWaitNs), 0);
                if (!ok) break;
                issue_raw(ps);
                issued = ps + 1;
            }
            // drain: every issued copy must land before the CTA may exit
            if (lane == 0) {
                const int first = issued > nst ? issued - nst : 0;
                for (int ps = first; ps < issued; ++ps)
                    if (!mbar_wait(bar(kRawFull + ps % nst), (ps / nst) & 1, kWaitNs)) ok = false;
            }
        } else {
            const uint32_t box_bytes = VA_PAGE_SIZE * 128;  // 16 rows x 64 bf16
            int issued = 0;
            for (int i = 0; i < ntiles; ++i) {
                const int buf = i % C::kNumBuf, use = i / C::kNumBuf;
                ok = __shfl_sync(0xffffffffu,
                                 (int)(mbar_wait(bar(kKEmpty + buf), (use & 1) ^ 1, kWaitNs) &&
                                       mbar_wait(bar(kVEmpty + buf), (use & 1) ^ 1, kWaitNs)),
                                 0);
                if (!ok) break;
                const int npg = tile_npg(i);
                const int page = tile_page(i);
                const uint32_t kb = sbase + L.conv_k + buf * C::kConvBytes;
                const uint32_t vb = sbase + L.conv_v + buf * C::kConvBytes;
                if (lane == 0) {
                    mbar_arrive_expect_tx(bar(kKFull + buf), npg * (D / 64) * box_bytes);
                    mbar_arrive_expect_tx(bar(kVFull + buf), npg * (D / 64) * box_bytes);
                }
                __syncwarp();
                if (lane < npg) {
#pragma unroll
                    for (int c = 0; c < D / 64; ++c) {
                        tma_load_4d(kb + c * C::kChunkBytes + lane * box_bytes, &mp.tm_k, c * 64, it.kvh, 0, page,
                                    bar(kKFull + buf));
                        tma_load_4d(vb + c * C::kChunkBytes + lane * box_bytes, &mp.tm_v, c * 64, it.kvh, 0, page,
                                    bar(kVFull + buf));
                    }
                }
                __syncwarp();
                issued = i + 1;
            }
            if (lane == 0) {
                const int first = issued > C::kNumBuf ? issued - C::kNumBuf : 0;
                for (int i = first; i < issued; ++i) {
                    if (!mbar_wait(bar(kKFull + i % C::kNumBuf), (i / C::kNumBuf) & 1, kWaitNs)) ok = false;
                    if (!mbar_wait(bar(kVFull + i % C::kNumBuf), (i / C::kNumBuf) & 1, kWaitNs)) ok = false;
                }
            }
        }
    } else if (warp == C::kMmaWarp) {
        // ------------------------------------------------------------ MMA issue
        if (lane == 0) {
            constexpr int kAB = C::kQuant ? 0 : 1;  // fp16 (quantised caches) or bf16
            constexpr uint32_t idS = idesc_f16(128, kTile, kAB, 0, 0);
            constexpr uint32_t idO = idesc_f16(128, D, kAB, 0, 1);  // A = P (TMEM), B = V (MN-major)
            const uint32_t s_tm = tmem + C::kSCol, o_tm = tmem + C::kOCol, q_tm = tmem + C::kQCol;
            // K tile: K-major (d contiguous) SW128, 8-row groups 1024 B apart.
            // V tile: MN-major (d contiguous) SW128, 64-d chunks kChunkBytes apart.
            const uint64_t kdesc0 = smem_desc(sbase + L.conv_k, 16, 1024, 2);
            const uint64_t vdesc0 = smem_desc(sbase + L.conv_v, C::kChunkBytes, 1024, 2);
            constexpr uint32_t kBufStep = C::kConvBytes >> 4;
            ok = mbar_wait(bar(kQReady), 0, kWaitNs);
            auto issue_pv = [&](int j) -> bool {
                const int b = j & 1, buf = j % C::kNumBuf, use = j / C::kNumBuf;
                if (!mbar_wait(bar(kPFull + b), (j >> 1) & 1, kWaitNs)) return false;
                if (!mbar_wait(bar(kVFull + buf), use & 1, kWaitNs)) return false;
                tc_fence_after();
                const uint64_t vd = vdesc0 + (uint64_t)(buf * kBufStep);
                // P of tile j: fp16 pairs in the first kTile / 2 columns of S buffer b
#pragma unroll
                for (int kk = 0; kk < kTile / 16; ++kk)
                    mma_ts(o_tm, s_tm + b * kTile + kk * 8, vd + (uint64_t)(kk * (16 * 128 >> 4)), idO,
                           (j > 0 || kk > 0) ? 1u : 0u);
                mma_commit(bar(kVEmpty + buf));
                mma_commit(bar(kPEmpty + b));
                mma_commit(bar(kODone));
                return true;
            };
            for (int i = 0; i < ntiles && ok; ++i) {
                const int b = i & 1, buf = i % C::kNumBuf, use = i / C::kNumBuf;
                // S buffer b holds P of tile i - 2 until that P x V has completed
                if (!mbar_wait(bar(kKFull + buf), use & 1, kWaitNs) ||
                    !mbar_wait(bar(kPEmpty + b), ((i >> 1) & 1) ^ 1, kWaitNs)) { ok = false; break; }
                tc_fence_after();
                const uint64_t kd = kdesc0 + (uint64_t)(buf * kBufStep);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_ts(s_tm + b * kTile, q_tm + kk * 8,
                           kd + (uint64_t)((kk / 4) * (C::kChunkBytes >> 4) + (kk % 4) * 2), idS, kk > 0 ? 1u : 0u);
                mma_commit(bar(kSFull + b));
                mma_commit(bar(kKEmpty + buf));
                if (i > 0 && !issue_pv(i - 1)) { ok = false; break; }
            }
            if (ok && ntiles > 0) ok = issue_pv(ntiles - 1);
            mma_commit(bar(kOFinal));
            if (p.seq_lens[it.b] != it.L) atomicOr(p.flags, kFlagSeqLenMismatch);  // off the critical path
            if (!mbar_wait(bar(kOFinal), 0, kWaitNs)) ok = false;
        }
    } else if (warp < C::kSoftmaxWarps) {
        // ------------------------------------------------------------ softmax
        // Warps w and w+4 share TMEM lane quarter w % 4 (rows 32q..32q+31):
        // half h = w / 4 owns S columns [32h, 32h + 32) of every tile, O
        // columns [h D/2, (h+1) D/2) and the row's d range [h D/2, (h+1) D/2)
        // of Q.  The pair exchanges per-row maxima through shared memory.
        const int quarter = warp & 3, half = warp >> 2;
        const int r = quarter * 32 + lane;
        const bool row_ok = r < nrows;
        const bool warp_active = quarter * 32 < nrows;  // same for both warps of a pair
        const uint32_t lane_tm = tmem + ((uint32_t)(quarter * 32) << 16);
        const int pair_bar = 1 + quarter;
        const uint32_t xmax = sbase + L.xchg;                 // [parity][half][128]
        const uint32_t xsum = xmax + 2 * 2 * 128 * 4;          // [half][128]
        const float c_r = p.sm_scale_log2 / q_prescale;  // score scale in log2 units
        float m_run = -INFINITY, l_run = 0.f;
        int beta = 0;  // value normaliser of the tiles so far (quantised caches): 2^beta
        const int last_visible = it.L - T + t_r;  // bottom-right causal mask
        const uint32_t ring = sbase + L.scale_ring;  // shared address of the scale ring
        for (int i = 0; i < ntiles; ++i) {
            const int b = i & 1;
            if (!mbar_wait(bar(kSFull + b), (i >> 1) & 1, kWaitNs)) { ok = false; break; }
            tc_fence_after();
            if (!warp_active) {  // all rows of this quarter are padding: only release the scales
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(kRingFree + i % kScaleRing));
            } else {
                const int key0 = it.k_begin + i * kTile + half * 32;  // first key of this half
                uint32_t s[32];
                tmem_ld32(lane_tm + C::kSCol + b * kTile + half * 32, s);
                tmem_wait_ld();
                const uint32_t slot = ring + (i % kScaleRing) * kRingFloats * 4;
                const uint32_t ks = slot + half * 32 * 4;
                const uint32_t vs = ks + kTile * 4;
                // pages outside the pool (only checked when the pool size is
                // known) were replaced by page 0 when loading: mask their keys
                uint32_t bad_pages = 0;
                if (p.num_pages > 0) {
#pragma unroll
                    for (int pg = 0; pg < 2; ++pg) {
                        const int key = key0 + pg * VA_PAGE_SIZE;
                        if (key < it.k_end) {
                            const int page = bt[key / VA_PAGE_SIZE];
                            if (page < 0 || page >= p.num_pages) bad_pages |= 1u << pg;
                        }
                    }
                }
                const bool full = row_ok && key0 + 32 <= it.k_end && key0 + 31 <= last_visible && bad_pages == 0;
                // x = raw score * k_scale (masked keys -inf); 8 independent max chains
                float mx[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) mx[k] = -INFINITY;
                if (__all_sync(0xffffffffu, full)) {
#pragma unroll
                    for (int j4 = 0; j4 < 8; ++j4) {
                        if (C::kQuant) {  // k scales: two packed multiplies per four keys
                            const uint4 sc = lds_u4(ks + 16 * j4);
                            f2_unpack(f2_mul(f2_pack(s[4 * j4], s[4 * j4 + 1]), f2_pack(sc.x, sc.y)), s[4 * j4],
                                      s[4 * j4 + 1]);
                            f2_unpack(f2_mul(f2_pack(s[4 * j4 + 2], s[4 * j4 + 3]), f2_pack(sc.z, sc.w)),
                                      s[4 * j4 + 2], s[4 * j4 + 3]);
                        }
                        const int c = j4 & 3;  // four chains of three-input maxima
                        mx[c] = fmax3(mx[c], __uint_as_float(s[4 * j4]), __uint_as_float(s[4 * j4 + 1]));
                        mx[c] = fmax3(mx[c], __uint_as_float(s[4 * j4 + 2]), __uint_as_float(s[4 * j4 + 3]));
                    }
                } else {
#pragma unroll
                    for (int j4 = 0; j4 < 8; ++j4) {
                        float4 sc = make_float4(1.f, 1.f, 1.f, 1.f);
                        if (C::kQuant) sc = lds_f4(ks + 16 * j4);
                        const float scv[4] = {sc.x, sc.y, sc.z, sc.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int j = 4 * j4 + e;
                            const int key = key0 + j;
                            const bool vis = row_ok && key < it.k_end && key <= last_visible &&
                                             !((bad_pages >> (j / VA_PAGE_SIZE)) & 1u);
                            const float v = vis ? __uint_as_float(s[j]) * scv[e] : -INFINITY;
                            s[j] = __float_as_uint(v);
                            mx[j & 7] = fmaxf(mx[j & 7], v);
                        }
                    }
                }
                float mt = fmaxf(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], fmaxf(mx[5], fmaxf(mx[6], mx[7]))));
                // exchange with the other half (double-buffered by tile parity)
                sts_f32(xmax + 4u * ((b * 2 + half) * 128 + r), mt);
                named_bar_sync(pair_bar, 64);
                mt = fmaxf(mt, lds_f32(xmax + 4u * ((b * 2 + 1 - half) * 128 + r)));
                const float m_tile = mt * c_r;  // -inf stays -inf (c_r > 0)
                const bool grow = m_tile > m_run + kRescaleLog2;
                const bool rescale = grow && m_run != -INFINITY;
                float alpha = 1.f;
                if (grow) {
                    if (rescale) alpha = ex2_approx(m_run - m_tile);
                    m_run = m_tile;
                    l_run *= alpha;
                }
                // Value normaliser (quantised caches): P carries p * v_scale * 2^beta
                // with 2^beta bringing the tile's largest v scale into [1, 2); beta
                // is kept while that product stays in [2^-6, 4), so that P stays in
                // fp16's normal range whatever the values' magnitude.  Every thread
                // takes the same decision from the same two maxima; O, which holds
                // the earlier tiles at the previous beta, follows a change.
                int dbeta = 0;
                if (C::kQuant) {
                    const float mv = fmaxf(lds_f32(slot + 4u * (2 * kTile)), lds_f32(slot + 4u * (2 * kTile + 1)));
                    if (mv > 0.f) {
                        const float rr = mv * __uint_as_float((uint32_t)(127 + beta) << 23);
                        if (i == 0 || !(rr >= 0x1p-6f && rr < 4.f)) {
                            // mv in [2^(E-127), 2^(E-126)): beta = 127 - E, capped at 118
                            // so that p 2^beta (p <= 2^8) stays finite in fp32
                            const int E = max(9, min(253, (int)((__float_as_uint(mv) >> 23) & 0xFFu)));
                            dbeta = i == 0 ? 0 : (127 - E) - beta;
                            beta = 127 - E;
                        }
                    }
                }
                // powers of two: exact
                const float fo =
                    dbeta == 0 ? alpha : alpha * __uint_as_float((uint32_t)(127 + max(-126, min(127, dbeta))) << 23);
                if (__any_sync(0xffffffffu, fo != 1.f) && i > 0) {
                    // O holds the earlier tiles: wait until PV(i-1) has landed
                    // (its commit completes the ((i-1)/2)-th phase of P buffer (i-1)%2)
                    if (!mbar_wait(bar(kPEmpty + ((i - 1) & 1)), ((i - 1) >> 1) & 1, kWaitNs)) { ok = false; }
                    tc_fence_after();
#pragma unroll 1
                    for (int c0 = half * (D / 2); c0 < (half + 1) * (D / 2); c0 += 32) {
                        uint32_t o[32];
                        tmem_ld32(lane_tm + C::kOCol + c0, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * fo);
                        tmem_st32(lane_tm + C::kOCol + c0, o);
                    }
                    tmem_wait_st();
                }
                // p = 2^(x*c - m); masked keys give 2^-inf = 0 and carry a zero
                // v scale, so no select is needed
                const float neg_m = (m_run == -INFINITY ? 0.f : -m_run) + (float)beta;
                const uint64_t c2 = f2_pack(__float_as_uint(c_r), __float_as_uint(c_r));
                const uint64_t nm2 = f2_pack(__float_as_uint(neg_m), __float_as_uint(neg_m));
                uint32_t pk[16];
                uint64_t ls[2] = {0ull, 0ull};  // packed partial sums (+0.0f pairs)
#pragma unroll
                for (int j4 = 0; j4 < 8; ++j4) {
                    uint32_t a[4];
                    f2_unpack(f2_fma(f2_pack(s[4 * j4], s[4 * j4 + 1]), c2, nm2), a[0], a[1]);
                    f2_unpack(f2_fma(f2_pack(s[4 * j4 + 2], s[4 * j4 + 3]), c2, nm2), a[2], a[3]);
                    uint32_t pb[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) pb[e] = __float_as_uint(ex2_approx(__uint_as_float(a[e])));
                    const uint64_t p01 = f2_pack(pb[0], pb[1]), p23 = f2_pack(pb[2], pb[3]);
                    ls[j4 & 1] = f2_add(ls[j4 & 1], f2_add(p01, p23));
                    if (C::kQuant) {
                        const uint4 sc = lds_u4(vs + 16 * j4);
                        uint32_t w[4];
                        f2_unpack(f2_mul(p01, f2_pack(sc.x, sc.y)), w[0], w[1]);
                        f2_unpack(f2_mul(p23, f2_pack(sc.z, sc.w)), w[2], w[3]);
                        pk[2 * j4] = pack_half2(__uint_as_float(w[0]), __uint_as_float(w[1]));
                        pk[2 * j4 + 1] = pack_half2(__uint_as_float(w[2]), __uint_as_float(w[3]));
                    } else {
                        pk[2 * j4] = pack_bf162(__uint_as_float(pb[0]), __uint_as_float(pb[1]));
                        pk[2 * j4 + 1] = pack_bf162(__uint_as_float(pb[2]), __uint_as_float(pb[3]));
                    }
                }
                uint32_t l0, l1;
                f2_unpack(f2_add(ls[0], ls[1]), l0, l1);
                l_run += (__uint_as_float(l0) + __uint_as_float(l1)) * __uint_as_float((uint32_t)(127 - beta) << 23);
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(kRingFree + i % kScaleRing));  // scale slot read
                // P row r, keys [32 half, 32 half + 32) -> columns [16 half, 16 half + 16)
                // of S buffer b (the pair has read both halves of S: they met at
                // the max exchange above)
                tmem_st16(lane_tm + C::kSCol + b * kTile + half * 16, pk);
                tmem_wait_st();
            }
            if (!C::kQuant && it.k_begin + i * kTile + kTile > it.k_end) {
                // last tile of the item: rows past the split end hold whatever
                // the cache has there; zero them so that 0 * V stays 0 in P x V
                const int key0 = it.k_begin + i * kTile;
                const int buf = i % C::kNumBuf;
                if (!mbar_wait(bar(kVFull + buf), (i / C::kNumBuf) & 1, kWaitNs)) ok = false;
                const int valid = it.k_end - key0;
                const uint32_t vb = sbase + L.conv_v + buf * C::kConvBytes;
                const int qt = warp * 32 + lane;  // 0..255 over the softmax warps
                for (int e = qt; e < (kTile - valid) * (D / 8); e += C::kSoftmaxWarps * 32) {
                    const int row = valid + e / (D / 8), u16 = e % (D / 8);
                    sts_u4(vb + (u16 / 8) * C::kChunkBytes + sw128(row, u16 % 8), make_uint4(0, 0, 0, 0));
                }
                fence_proxy_async_smem();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kPFull + b));
        }
        // epilogue: O / l and the log-sum-exp (the pair adds its partial sums).
        // An unsplit item's rows go to out as bf16: staged in the tile buffers
        // (free once the last P x V has completed), 16-byte units XOR-swizzled
        // by row, then copied out with consecutive 16-byte stores.  A split's
        // fp32 partials are staged as the boxes of the partials' tensor map
        // and leave by TMA, one 32-column chunk at a time, each store starting
        // as soon as the four warps of its half have staged it.
        if (!mbar_wait(bar(kOFinal), 0, kWaitNs)) ok = false;
        tc_fence_after();
        const bool final_out = it.part < 0;
        const int cb = D / 8;  // 16-byte units per staged bf16 row
        const uint32_t stage = sbase + L.conv_k;
        // fp32 chunk stride (rows padded to 8 keep every box 1024-byte aligned)
        const uint32_t cstride = (uint32_t)((p.rows_per_group + 7) / 8 * 8) * 128u;
        auto unit = [](int row, int c) { return (uint32_t)(((c & ~7) | ((c ^ row) & 7)) << 4); };
        float inv = 0.f;
        if (warp_active) {
            sts_f32(xsum + 4u * (half * 128 + r), l_run);
            named_bar_sync(pair_bar, 64);
            const float l_tot = l_run + lds_f32(xsum + 4u * ((1 - half) * 128 + r));
            inv = l_tot > 0.f ? (1.f / l_tot) * __uint_as_float((uint32_t)(127 - beta) << 23) : 0.f;
            const float lse_nat = l_tot > 0.f ? (m_run + log2f(l_tot)) * 0.69314718055994531f : -INFINITY;
            if (row_ok && half == 0 && ok) {  // the row's log-sum-exp
                const int rr = row0 + r;
                const size_t orow = (size_t)(it.b * T + t_r) * p.Hq + it.kvh * G + rr % G;
                if (final_out) {
                    if (p.lse) p.lse[orow] = lse_nat;
                } else {
                    p.lse_part[(size_t)it.part * p.rows_per_group + r] = lse_nat;
                }
            }
        }
        if (final_out) {
            if (warp_active) {
                const uint32_t srow = stage + (uint32_t)(r * cb * 16);
#pragma unroll 1
                for (int c0 = half * (D / 2); c0 < (half + 1) * (D / 2); c0 += 32) {
                    uint32_t o[32];
                    tmem_ld32(lane_tm + C::kOCol + c0, o);
                    tmem_wait_ld();
                    if (!row_ok) continue;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        uint4 w;
                        w.x = pack_bf162(__uint_as_float(o[8 * k + 0]) * inv, __uint_as_float(o[8 * k + 1]) * inv);
                        w.y = pack_bf162(__uint_as_float(o[8 * k + 2]) * inv, __uint_as_float(o[8 * k + 3]) * inv);
                        w.z = pack_bf162(__uint_as_float(o[8 * k + 4]) * inv, __uint_as_float(o[8 * k + 5]) * inv);
                        w.w = pack_bf162(__uint_as_float(o[8 * k + 6]) * inv, __uint_as_float(o[8 * k + 7]) * inv);
                        sts_u4(srow + unit(r, c0 / 8 + k), w);
                    }
                }
            }
            named_bar_sync(9, C::kSoftmaxWarps * 32);  // all rows staged
            if (ok) {
                const int st = warp * 32 + lane;  // 0 .. 255
                for (int e = st; e < nrows * cb; e += C::kSoftmaxWarps * 32) {
                    const int row = e / cb, c = e % cb;
                    const uint4 v = lds_u4(stage + (uint32_t)(row * cb * 16) + unit(row, c));
                    const int rr = row0 + row;
                    const size_t orow = (size_t)(it.b * T + rr / G) * p.Hq + it.kvh * G + rr % G;
                    *reinterpret_cast<uint4 *>(reinterpret_cast<unsigned char *>(p.out) + orow * D * 2 + c * 16) = v;
                }
            }
        } else {
            // rows past nrows in a box are padding that nothing reads
            const bool issuer = ok && quarter == 0 && lane == 0;
#pragma unroll 1
            for (int c0 = half * (D / 2); c0 < (half + 1) * (D / 2); c0 += 32) {
                const uint32_t chunk = stage + (uint32_t)(c0 / 32) * cstride;
                if (warp_active) {
                    uint32_t o[32];
                    tmem_ld32(lane_tm + C::kOCol + c0, o);
                    tmem_wait_ld();
                    if (row_ok) {
                        // row r of the chunk, 16-byte units XOR-swizzled by r % 8 (the
                        // tensor map's 128-byte swizzle; also conflict-free here)
                        const uint32_t crow = chunk + (uint32_t)r * 128u;
#pragma unroll
                        for (int k = 0; k < 8; ++k)
                            sts_u4(crow + ((k ^ (r & 7)) << 4),
                                   make_uint4(__float_as_uint(__uint_as_float(o[4 * k]) * inv),
                                              __float_as_uint(__uint_as_float(o[4 * k + 1]) * inv),
                                              __float_as_uint(__uint_as_float(o[4 * k + 2]) * inv),
                                              __float_as_uint(__uint_as_float(o[4 * k + 3]) * inv)));
                    }
                    fence_proxy_async_smem();  // staged rows -> the TMA store
                }
                named_bar_sync(11 + half, 128);  // the half's four warps have staged this chunk
                if (issuer) {
                    tma_store_2d(&mp.tm_o, c0, it.part * p.rows_per_group, chunk);
                    bulk_commit_group();
                }
            }
            if (issuer) bulk_wait_group_read0();  // shared memory stays valid until the stores have read it
        }
    } else if constexpr (C::kQuant) {
        // ------------------------------------------------------------ dequant
        // Two groups of four warps, one per lane quarter each: warps 8-11 take
        // the K tile of every tile (plus this head's k and v scales, which the
        // softmax of the tile needs), warps 12-15 the V tile, so that the K
        // pass of tile i+1 runs beside the V pass of tile i.  int8 / e4m3 /
        // int4 / int2 -> fp16 (exact) into the MMA layout; each thread takes
        // pieces of 16 consecutive elements, whatever their width in bytes.
        constexpr int kGT = C::kDequantWarps * 16;             // threads per group
        const int dq = tid - C::kSoftmaxWarps * 32;            // 0 .. 2 kGT - 1
        const int kv = dq / kGT;                               // 0: K group, 1: V group
        const int dt = dq % kGT;
        const uint32_t ring = sbase + L.scale_ring;
        constexpr int kChunks = kTile * D / 16;                // 16-element raw pieces per tile
        constexpr int kPer = kChunks / kGT;                    // per thread (2, 4 or 8)
        constexpr int kPieceBytes = 16 * C::kBits / 8;          // 16, 8 or 4
        constexpr int kRowStep = kGT * 16 / D;                 // tile rows between a thread's chunks
        static_assert(kPer * kGT == kChunks && kRowStep % 8 == 0, "chunks must divide evenly");
        // this thread's chunks sit kGT * 16 raw bytes (kRowStep rows, a
        // multiple of the swizzle period) apart; destinations of the first
        // chunk's two 16-byte fp16 units (store order alternates between 64-d
        // chunks so that a quarter-warp never hits a bank twice)
        const int n0 = dt * 16 / D, d0 = (dt * 16) % D;
        const uint32_t woff_lo = (d0 / 64) * C::kChunkBytes + sw128(n0, (d0 % 64) / 8);
        const uint32_t woff_hi = (d0 / 64) * C::kChunkBytes + sw128(n0, (d0 % 64) / 8 + 1);
        const bool odd_chunk = (d0 / 64) & 1;
        // K group: thread dt carries one scale of a tile, k (dt < 64) or v of
        // key dt % 64, loaded from global two tiles before it is needed
        static_assert(kGT == 2 * kTile, "one scale per K-group thread");
        const float *scale_src = dt < kTile ? p.k_scale : p.v_scale;
        auto load_scale = [&](int i) -> float {
            const int n = dt % kTile;
            const int key = it.k_begin + i * kTile + n;
            if (i >= ntiles || key >= it.k_end) return 0.f;
            const int page = (int)lds_u32(sbase + L.pids + 4u * (i * (kTile / VA_PAGE_SIZE) + n / VA_PAGE_SIZE));
            return __ldg(scale_src + ((size_t)page * VA_PAGE_SIZE + n % VA_PAGE_SIZE) * Hkv + it.kvh);
        };
        // two tiles of scales in flight: a global load under load takes about as
        // long as a tile
        float scale_cur = 0.f, scale_nxt = 0.f;
        if (kv == 0) {
            scale_cur = load_scale(0);
            scale_nxt = load_scale(1);
        }
        for (int i = 0; i < ntiles && ok; ++i) {
            const int ps = 2 * i + kv;  // raw passes: K of tile 0, V of tile 0, K of tile 1, ...
            const int buf = i % C::kNumBuf, use = i / C::kNumBuf;
            const int nvalid = min(kTile, it.k_end - (it.k_begin + i * kTile));
            const int slot = ps % nst;
            // the raw bytes go to registers and the stage is handed back to
            // the producer at once, before waiting for the fp16 buffer
            if (!mbar_wait(bar(kRawFull + slot), (ps / nst) & 1, kWaitNs)) {
                ok = false;
                break;
            }
            const uint32_t st = sbase + L.raw + slot * L.raw_stride + dt * kPieceBytes;
            const uint32_t dst = sbase + (kv == 0 ? L.conv_k : L.conv_v) + buf * C::kConvBytes;
            RawPiece<DT> raw[kPer];
#pragma unroll
            for (int jj = 0; jj < kPer; ++jj) raw[jj].load(st + jj * kGT * kPieceBytes);
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kRawEmpty + slot));
            // the tile's scales move up the pipeline and the load two tiles
            // ahead is issued now, before this pass's stores fill the
            // shared-memory queue
            float scale_out = 0.f;
            if (kv == 0) {
                scale_out = scale_cur;
                scale_cur = scale_nxt;
                scale_nxt = load_scale(i + 2);
            }
            if (!mbar_wait(bar((kv == 0 ? kKEmpty : kVEmpty) + buf), (use & 1) ^ 1, kWaitNs)) {
                ok = false;
                break;
            }
#pragma unroll
            for (int jj = 0; jj < kPer; ++jj) {
                uint32_t hw[8];
                raw[jj].to_half(hw);
                uint4 lo = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                uint4 hi = make_uint4(hw[4], hw[5], hw[6], hw[7]);
                if (n0 + jj * kRowStep >= nvalid) lo = hi = make_uint4(0, 0, 0, 0);  // past the split end
                const uint32_t row_off = jj * kRowStep * 128;
                if (odd_chunk) {
                    sts_u4(dst + woff_hi + row_off, hi);
                    sts_u4(dst + woff_lo + row_off, lo);
                } else {
                    sts_u4(dst + woff_lo + row_off, lo);
                    sts_u4(dst + woff_hi + row_off, hi);
                }
            }
            if (kv == 0) {  // the tile's k and v scales (zero past the end) -> ring
                // slot i % kScaleRing held tile i - kScaleRing, whose softmax has to have read it
                if (!mbar_wait(bar(kRingFree + i % kScaleRing), ((i / kScaleRing) & 1) ^ 1, kWaitNs)) ok = false;
                const uint32_t slot = ring + (i % kScaleRing) * kRingFloats * 4;
                sts_f32(slot + 4u * dt, scale_out);
                if (dt >= kTile) {  // the largest v scale of this warp's 32 keys (scales are >= 0:
                                    // their bits order like unsigned integers)
                    const uint32_t mv = __reduce_max_sync(0xffffffffu, __float_as_uint(scale_out));
                    if (lane == 0) sts_u32(slot + 4u * (2 * kTile + (dt - kTile) / 32), mv);
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar((kv == 0 ? kKFull : kVFull) + buf));
        }
    }

    if (!ok) atomicOr(p.flags, kFlagTimeout);
    tc_fence_before();
    __syncthreads();
    if (warp == C::kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
        else
            cudaGetLastError();
    });
    return fn;
}

// The split partials [num_parts * rows_per_group, D] fp32 as boxes of 32
// columns x rows_per_group rows, 128-byte swizzled in shared memory.
bool make_part_map(CUtensorMap *m, float *o_part, int D, int rows_per_group, int num_parts) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)num_parts * rows_per_group};
    cuuint64_t strides[1] = {(cuuint64_t)D * 4};
    cuuint32_t box[2] = {32u, (cuuint32_t)rows_per_group};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, o_part, dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 4-D view of a page pool [pages, 16, Hkv, row]: dims innermost first.  A
// bf16 row is D elements (boxes of 64, swizzled into the MMA layout); a
// quantised row is its D * bits / 8 bytes (one box per page and head: 16, 32,
// 64, 128 or 256 bytes wide, always a multiple of 16).
bool make_map(CUtensorMap *m, const void *base, int D, int bits, int Hkv, int num_pages) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const bool bf16 = bits == 16;
    const cuuint64_t eb = bf16 ? 2 : 1;
    const cuuint64_t row = bf16 ? (cuuint64_t)D : (cuuint64_t)D * bits / 8;  // elements of the map's type
    const cuuint64_t pages = num_pages > 0 ? (cuuint64_t)num_pages : (cuuint64_t)1 << 30;
    cuuint64_t dims[4] = {row, (cuuint64_t)Hkv, (cuuint64_t)VA_PAGE_SIZE, pages};
    cuuint64_t strides[3] = {row * eb, (cuuint64_t)Hkv * row * eb, (cuuint64_t)VA_PAGE_SIZE * Hkv * row * eb};
    cuuint32_t box[4] = {bf16 ? 64u : (cuuint32_t)row, 1u, (cuuint32_t)VA_PAGE_SIZE, 1u};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 4,
                     const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     bf16 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int D, int DT>
cudaError_t launch_one(const PartialParams &p, int n, cudaStream_t s) {
    MmaParams mp;
    mp.p = p;
    if (!make_map(&mp.tm_k, p.k_pages, D, Cfg<D, DT>::kBits, p.Hkv, p.num_pages) ||
        !make_map(&mp.tm_v, p.v_pages, D, Cfg<D, DT>::kBits, p.Hkv, p.num_pages))
        return cudaErrorInvalidValue;
    memset(&mp.tm_o, 0, sizeof(mp.tm_o));
    if (p.num_parts > 0 && !make_part_map(&mp.tm_o, p.o_part, D, p.rows_per_group, p.num_parts))
        return cudaErrorInvalidValue;
    int nst = 0;
    if (Cfg<D, DT>::kQuant) {
        nst = kMaxRawStages;
        while (nst > kMinRawStages && Smem<D, DT>(p.Hkv, nst).total + 1024 > kMaxSmemPerBlock) --nst;
    }
    mp.raw_stages = nst;
    const Smem<D, DT> L(p.Hkv, nst);
    const size_t smem = L.total + 1024;  // + alignment slack
    if (smem > kMaxSmemPerBlock) return cudaErrorInvalidConfiguration;
    auto k = mma_partial_kernel<D, DT>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(k, dim3(n), dim3(Cfg<D, DT>::kThreads), smem, s, mp);
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

// Shared memory of the tensor-core kernel with the fewest raw stages it runs
// with (the planner falls back to the CUDA-core kernel when this exceeds the
// per-block limit).
size_t mma_smem_bytes(int head_dim, int kv_dtype, int Hkv) {
    const bool bf = kv_dtype == VA_BF16;
    switch (head_dim) {
    case 64: return (bf ? Smem<64, VA_BF16>(Hkv, 0).total : Smem<64, VA_INT8>(Hkv, kMinRawStages).total) + 1024;
    case 128: return (bf ? Smem<128, VA_BF16>(Hkv, 0).total : Smem<128, VA_INT8>(Hkv, kMinRawStages).total) + 1024;
    default: return (bf ? Smem<256, VA_BF16>(Hkv, 0).total : Smem<256, VA_INT8>(Hkv, kMinRawStages).total) + 1024;
    }
}

cudaError_t launch_mma_partial(const PartialParams &p, int head_dim, int kv_dtype, int n, cudaStream_t s) {
    if (n <= 0) return cudaSuccess;
    switch (head_dim) {
    case 64: return launch_d<64>(p, kv_dtype, n, s);
    case 128: return launch_d<128>(p, kv_dtype, n, s);
    default: return launch_d<256>(p, kv_dtype, n, s);
    }
}

}  // namespace va
