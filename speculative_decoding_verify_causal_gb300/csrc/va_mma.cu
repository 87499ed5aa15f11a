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
// almost for free); keeping the cache 1 byte per element until the last step
// before the tensor core is the same section's "keep it compressed while it is
// read from HBM".
//
// Per 64-key tile (4 pages):
//   producer warp    TMA-gathers the pages named by the block table (4-D
//                    tensor map over [page, slot, kv head, d]) plus the
//                    pages' scale blocks (1-D bulk copies);
//   dequant warps    (fp8-e4m3 / int8) convert the raw bytes to fp16 -- both
//                    conversions are exact -- into the 128-byte-swizzled
//                    layout the MMA reads (bf16 caches are TMA'd straight
//                    into that layout);
//   MMA warp         one thread issues S = Q K^T (A = Q in TMEM, B = K tile in
//                    shared memory, D = S in TMEM, M=128 N=64 K=16 x D/16) and
//                    O += P V (A = P in TMEM, B = V tile, N = D);
//   softmax warps    one thread per packed row: reads its S row from TMEM,
//                    applies the per-key k scale and the bottom-right causal
//                    mask, keeps the running max / sum (base 2; the max is
//                    only moved, and O rescaled, when it grows by more than
//                    2^8), writes P * v_scale (fp16) back over S in TMEM,
//                    and at the end writes O / l and the log-sum-exp.
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

#include <mutex>

#include "va_internal.h"
#include "va_sm100.cuh"

namespace va {
namespace {

using namespace sm100;

constexpr int kTile = kMmaTile;     // keys per S tile (MMA N)
constexpr int kRawKeys = 32;        // keys per raw (8-bit) stage: 2 pages
constexpr int kRawStages = 4;
constexpr int kBfStages = 3;        // bf16: 64-key stages TMA'd straight into MMA layout
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr float kRescaleLog2 = 8.0f;
constexpr int kScaleRing = 4;       // per-tile k/v scales handed to the softmax warps

enum : int { kFlagTimeout = 4 };

struct MmaParams {
    CUtensorMap tm_k;  // 64-byte aligned members first
    CUtensorMap tm_v;
    PartialParams p;
};

template <int D, int DT>
struct Cfg {
    static constexpr bool kQuant = DT != VA_BF16;
    static constexpr int kNumBuf = kQuant ? 2 : kBfStages;
    static constexpr int kConvBytes = kTile * D * 2;   // K or V tile, 16-bit, SW128 chunks of 64 d
    static constexpr int kChunkBytes = kTile * 128;    // one 64-d chunk of a tile
    static constexpr int kRawBytes = kRawKeys * D;     // K or V half tile, 8-bit
    static constexpr int kWarps = kQuant ? 10 : 6;
    static constexpr int kThreads = kWarps * 32;
    static constexpr uint32_t kQCol = 0;
    static constexpr uint32_t kOCol = D / 2;
    static constexpr uint32_t kSCol = D / 2 + D;
    static constexpr uint32_t kTmemCols = 512;
};

// Shared memory carve-up (byte offsets from a 1024-aligned base).
template <int D, int DT>
struct Smem {
    using C = Cfg<D, DT>;
    uint32_t conv_k, conv_v;       // kNumBuf buffers each
    uint32_t raw, raw_stride;      // kRawStages stages (quantised only)
    uint32_t raw_v, raw_ks, raw_vs;  // offsets inside a raw stage
    uint32_t scale_ring;           // kScaleRing x (64 k + 64 v) floats
    uint32_t bars;                 // mbarriers
    uint32_t total;
    __host__ __device__ explicit Smem(int Hkv) {
        conv_k = 0;
        conv_v = conv_k + C::kNumBuf * C::kConvBytes;
        raw = conv_v + C::kNumBuf * C::kConvBytes;
        const uint32_t sc = 2u * VA_PAGE_SIZE * Hkv * 4;  // one stage's scale blocks (2 pages)
        raw_v = C::kRawBytes;
        raw_ks = 2 * C::kRawBytes;
        raw_vs = raw_ks + sc;
        raw_stride = C::kQuant ? ((raw_vs + sc + 127) / 128 * 128) : 0;
        scale_ring = raw + (C::kQuant ? kRawStages * raw_stride : 0);
        bars = scale_ring + (C::kQuant ? kScaleRing * 2 * kTile * 4 : 0);
        total = bars + 64 * 8 + 16;
    }
};

// Barrier slots (8 bytes each) inside Smem::bars.
enum Bar : int {
    kRawFull = 0,                       // kRawStages
    kRawEmpty = kRawFull + kRawStages,  // kRawStages
    kKFull = kRawEmpty + kRawStages,    // kNumBuf (<= 3)
    kKEmpty = kKFull + 3,
    kVFull = kKEmpty + 3,
    kVEmpty = kVFull + 3,
    kSFull = kVEmpty + 3,               // 2
    kSFree = kSFull + 2,                // 2
    kPFull = kSFree + 2,                // 2
    kODone = kPFull + 2,
    kOFinal = kODone + 1,
    kQReady = kOFinal + 1,
    kNumBars = kQReady + 1,
};

__device__ __forceinline__ float bf16_bits_to_float(uint32_t b) { return __uint_as_float(b << 16); }

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

// Byte offset of 16-byte unit u (0..7) of tile row `row` inside a 64-d chunk
// of a 128-byte-swizzled tile (rows of 128 bytes, 8-row / 1024-byte atoms).
__device__ __forceinline__ uint32_t sw128(int row, int u) { return row * 128 + ((u ^ (row & 7)) << 4); }

template <int D, int DT>
__global__ void __launch_bounds__(Cfg<D, DT>::kThreads, 1)
mma_partial_kernel(const __grid_constant__ MmaParams mp) {
    using C = Cfg<D, DT>;
    const PartialParams &p = mp.p;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const Smem<D, DT> L(p.Hkv);
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + L.bars;
    auto bar = [&](int i) { return bar0 + 8u * i; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L.bars + kNumBars * 8);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const Item it = p.items[blockIdx.x];
    const int G = p.G, T = p.T, Hkv = p.Hkv;
    const int row0 = it.rg * p.rows_per_group;
    const int nrows = min(p.rows_per_group, p.R - row0);
    const int nkeys = it.k_end - it.k_begin;
    const int ntiles = (nkeys + kTile - 1) / kTile;
    const int32_t *bt = p.block_table + (size_t)it.b * p.bt_stride;

    if (tid == 0) {
        for (int i = 0; i < kRawStages; ++i) {
            mbar_init(bar(kRawFull + i), 1);
            mbar_init(bar(kRawEmpty + i), 4);
        }
        for (int i = 0; i < 3; ++i) {
            mbar_init(bar(kKFull + i), C::kQuant ? 4 : 1);
            mbar_init(bar(kVFull + i), C::kQuant ? 4 : 1);
            mbar_init(bar(kKEmpty + i), 1);
            mbar_init(bar(kVEmpty + i), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(kSFull + i), 1);
            mbar_init(bar(kSFree + i), 1);
            mbar_init(bar(kPFull + i), 4);
        }
        mbar_init(bar(kODone), 1);
        mbar_init(bar(kOFinal), 1);
        mbar_init(bar(kQReady), 4);
        fence_barrier_init();
        if (p.seq_lens[it.b] != it.L) atomicOr(p.flags, kFlagSeqLenMismatch);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    bool ok = true;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            prefetch_tensormap(&mp.tm_k);
            prefetch_tensormap(&mp.tm_v);
            if (C::kQuant) {
                const int nraw = (nkeys + kRawKeys - 1) / kRawKeys;
                const uint32_t page_bytes = VA_PAGE_SIZE * D;          // one page, one head, 8-bit
                const uint32_t scale_bytes = VA_PAGE_SIZE * Hkv * 4;   // one page's scale block
                int issued = 0;
                for (int rs = 0; rs < nraw && ok; ++rs) {
                    const int slot = rs % kRawStages, use = rs / kRawStages;
                    if (!mbar_wait(bar(kRawEmpty + slot), (use & 1) ^ 1, kWaitNs)) { ok = false; break; }
                    const int key0 = it.k_begin + rs * kRawKeys;
                    const int npg = min(2, (it.k_end - key0 + VA_PAGE_SIZE - 1) / VA_PAGE_SIZE);
                    const uint32_t st = sbase + L.raw + slot * L.raw_stride;
                    mbar_arrive_expect_tx(bar(kRawFull + slot), npg * 2 * (page_bytes + scale_bytes));
                    for (int pg = 0; pg < npg; ++pg) {
                        int page = bt[key0 / VA_PAGE_SIZE + pg];
                        if (p.num_pages > 0 && (page < 0 || page >= p.num_pages)) {
                            atomicOr(p.flags, kFlagBadPage);
                            page = 0;  // load a real page; the dequant masks these keys out
                        }
                        tma_load_4d(st + pg * page_bytes, &mp.tm_k, 0, it.kvh, 0, page, bar(kRawFull + slot));
                        tma_load_4d(st + L.raw_v + pg * page_bytes, &mp.tm_v, 0, it.kvh, 0, page,
                                    bar(kRawFull + slot));
                        bulk_load(st + L.raw_ks + pg * scale_bytes, p.k_scale + (size_t)page * VA_PAGE_SIZE * Hkv,
                                  scale_bytes, bar(kRawFull + slot));
                        bulk_load(st + L.raw_vs + pg * scale_bytes, p.v_scale + (size_t)page * VA_PAGE_SIZE * Hkv,
                                  scale_bytes, bar(kRawFull + slot));
                    }
                    issued = rs + 1;
                }
                // drain: every issued copy must land before the CTA may exit
                const int first = issued > kRawStages ? issued - kRawStages : 0;
                for (int rs = first; rs < issued; ++rs)
                    if (!mbar_wait(bar(kRawFull + rs % kRawStages), (rs / kRawStages) & 1, kWaitNs)) ok = false;
            } else {
                const uint32_t box_bytes = VA_PAGE_SIZE * 128;  // 16 rows x 64 bf16
                int issued = 0;
                for (int i = 0; i < ntiles && ok; ++i) {
                    const int buf = i % C::kNumBuf, use = i / C::kNumBuf;
                    if (!mbar_wait(bar(kKEmpty + buf), (use & 1) ^ 1, kWaitNs) ||
                        !mbar_wait(bar(kVEmpty + buf), (use & 1) ^ 1, kWaitNs)) { ok = false; break; }
                    const int key0 = it.k_begin + i * kTile;
                    const int npg = min(kTile / VA_PAGE_SIZE, (it.k_end - key0 + VA_PAGE_SIZE - 1) / VA_PAGE_SIZE);
                    const uint32_t kb = sbase + L.conv_k + buf * C::kConvBytes;
                    const uint32_t vb = sbase + L.conv_v + buf * C::kConvBytes;
                    mbar_arrive_expect_tx(bar(kKFull + buf), npg * (D / 64) * box_bytes);
                    mbar_arrive_expect_tx(bar(kVFull + buf), npg * (D / 64) * box_bytes);
                    for (int pg = 0; pg < npg; ++pg) {
                        int page = bt[key0 / VA_PAGE_SIZE + pg];
                        if (p.num_pages > 0 && (page < 0 || page >= p.num_pages)) {
                            atomicOr(p.flags, kFlagBadPage);
                            page = 0;
                        }
#pragma unroll
                        for (int c = 0; c < D / 64; ++c) {
                            tma_load_4d(kb + c * C::kChunkBytes + pg * box_bytes, &mp.tm_k, c * 64, it.kvh, 0, page,
                                        bar(kKFull + buf));
                            tma_load_4d(vb + c * C::kChunkBytes + pg * box_bytes, &mp.tm_v, c * 64, it.kvh, 0, page,
                                        bar(kVFull + buf));
                        }
                    }
                    issued = i + 1;
                }
                const int first = issued > C::kNumBuf ? issued - C::kNumBuf : 0;
                for (int i = first; i < issued; ++i) {
                    if (!mbar_wait(bar(kKFull + i % C::kNumBuf), (i / C::kNumBuf) & 1, kWaitNs)) ok = false;
                    if (!mbar_wait(bar(kVFull + i % C::kNumBuf), (i / C::kNumBuf) & 1, kWaitNs)) ok = false;
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issue
        if (lane == 0) {
            constexpr int kAB = C::kQuant ? 0 : 1;  // fp16 (quantised caches) or bf16
            constexpr uint32_t idS = idesc_f16(128, kTile, kAB, 0, 0);
            constexpr uint32_t idO = idesc_f16(128, D, kAB, 0, 1);
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
#pragma unroll
                for (int kk = 0; kk < kTile / 16; ++kk)
                    mma_ts(o_tm, s_tm + b * kTile + kk * 8, vd + (uint64_t)(kk * (16 * 128 >> 4)), idO,
                           (j > 0 || kk > 0) ? 1u : 0u);
                mma_commit(bar(kVEmpty + buf));
                mma_commit(bar(kSFree + b));
                mma_commit(bar(kODone));
                return true;
            };
            for (int i = 0; i < ntiles && ok; ++i) {
                const int b = i & 1, buf = i % C::kNumBuf, use = i / C::kNumBuf;
                if (!mbar_wait(bar(kKFull + buf), use & 1, kWaitNs) ||
                    !mbar_wait(bar(kSFree + b), ((i >> 1) & 1) ^ 1, kWaitNs)) { ok = false; break; }
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
            if (!mbar_wait(bar(kOFinal), 0, kWaitNs)) ok = false;
        }
    } else if (warp < 6) {
        // ------------------------------------------------------------ softmax
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;
        const bool row_ok = r < nrows;
        const bool warp_active = quarter * 32 < nrows;
        const uint32_t lane_tm = tmem + ((uint32_t)(quarter * 32) << 16);
        int t_r = 0;
        float c_r = p.sm_scale_log2;  // score scale in log2 units (divided by q's power-of-two prescale)
        // Q row -> TMEM (fp16 with an exact power-of-two prescale for
        // quantised caches; bf16 as is)
        {
            const uint4 *qrow = nullptr;
            if (row_ok) {
                const int rr = row0 + r;
                t_r = rr / G;
                const int h = it.kvh * G + rr % G;
                qrow = reinterpret_cast<const uint4 *>(p.q + ((size_t)(it.b * T + t_r) * p.Hq + h) * D);
            }
            float qscale = 1.f;
            if (C::kQuant && row_ok) {
                float amax = 0.f;
                for (int i = 0; i < D / 8; ++i) {
                    const uint4 v = qrow[i];
                    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        amax = fmaxf(amax, fmaxf(fabsf(bf16_bits_to_float(w[k] & 0xFFFFu)),
                                                 fabsf(__uint_as_float(w[k] & 0xFFFF0000u))));
                }
                if (amax > 0.f) {
                    int e;
                    frexpf(amax, &e);  // amax in [2^(e-1), 2^e)
                    qscale = exp2f((float)(15 - e));  // amax * qscale in [2^14, 2^15)
                    c_r = p.sm_scale_log2 / qscale;
                }
            }
#pragma unroll 1
            for (int c0 = 0; c0 < D / 2; c0 += 32) {
                uint32_t v[32];
                if (row_ok) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const uint4 x = qrow[c0 / 4 + i];
                        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            if (C::kQuant)
                                v[4 * i + k] = pack_half2(bf16_bits_to_float(w[k] & 0xFFFFu) * qscale,
                                                          __uint_as_float(w[k] & 0xFFFF0000u) * qscale);
                            else
                                v[4 * i + k] = w[k];
                        }
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = 0u;
                }
                tmem_st32(lane_tm + C::kQCol + c0, v);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kQReady));
        }
        float m_run = -INFINITY, l_run = 0.f;
        const int last_visible = it.L - T + t_r;  // bottom-right causal mask
        const float *ring = reinterpret_cast<const float *>(smem + L.scale_ring);
        for (int i = 0; i < ntiles; ++i) {
            const int b = i & 1;
            if (!mbar_wait(bar(kSFull + b), (i >> 1) & 1, kWaitNs)) { ok = false; break; }
            tc_fence_after();
            if (warp_active) {
                const int key0 = it.k_begin + i * kTile;
                uint32_t s[64];
                tmem_ld32(lane_tm + C::kSCol + b * kTile, *reinterpret_cast<uint32_t(*)[32]>(&s[0]));
                tmem_ld32(lane_tm + C::kSCol + b * kTile + 32, *reinterpret_cast<uint32_t(*)[32]>(&s[32]));
                tmem_wait_ld();
                const float *ks = ring + (i % kScaleRing) * 2 * kTile;
                const float *vs = ks + kTile;
                // pages outside the pool (only checked when the pool size is
                // known) were replaced by page 0 when loading: mask their keys
                uint32_t bad_pages = 0;
                if (p.num_pages > 0) {
#pragma unroll
                    for (int pg = 0; pg < kTile / VA_PAGE_SIZE; ++pg) {
                        const int key = key0 + pg * VA_PAGE_SIZE;
                        if (key < it.k_end) {
                            const int page = bt[key / VA_PAGE_SIZE];
                            if (page < 0 || page >= p.num_pages) bad_pages |= 1u << pg;
                        }
                    }
                }
                const bool full = key0 + kTile <= it.k_end && key0 + kTile - 1 <= last_visible && row_ok &&
                                  bad_pages == 0;
                float x[64];
                float mt = -INFINITY;
#pragma unroll
                for (int j = 0; j < 64; ++j) {
                    float v = __uint_as_float(s[j]);
                    if (C::kQuant) v *= ks[j];
                    if (!full) {
                        const int key = key0 + j;
                        const bool vis = row_ok && key < it.k_end && key <= last_visible &&
                                         !((bad_pages >> (j / VA_PAGE_SIZE)) & 1u);
                        v = vis ? v : -INFINITY;
                    }
                    x[j] = v;
                    mt = fmaxf(mt, v);
                }
                const float m_tile = mt * c_r;  // -inf stays -inf (c_r > 0)
                const bool grow = m_tile > m_run + kRescaleLog2;
                const bool rescale = grow && m_run != -INFINITY;
                float alpha = 1.f;
                if (grow) {
                    if (rescale) alpha = exp2f(m_run - m_tile);
                    m_run = m_tile;
                    l_run *= alpha;
                }
                if (__any_sync(0xffffffffu, rescale) && i > 0) {
                    // O holds the earlier tiles: wait until PV(i-1) has landed
                    if (!mbar_wait(bar(kODone), (i - 1) & 1, kWaitNs)) { ok = false; }
                    tc_fence_after();
#pragma unroll 1
                    for (int c0 = 0; c0 < D; c0 += 32) {
                        uint32_t o[32];
                        tmem_ld32(lane_tm + C::kOCol + c0, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
                        tmem_st32(lane_tm + C::kOCol + c0, o);
                    }
                    tmem_wait_st();
                }
                const float neg_m = m_run == -INFINITY ? 0.f : -m_run;
                uint32_t pk[32];
                float lsum = 0.f;
#pragma unroll
                for (int j = 0; j < 64; j += 2) {
                    float p0 = 0.f, p1 = 0.f;
                    if (x[j] != -INFINITY) p0 = exp2f(fmaf(x[j], c_r, neg_m));
                    if (x[j + 1] != -INFINITY) p1 = exp2f(fmaf(x[j + 1], c_r, neg_m));
                    lsum += p0 + p1;
                    if (C::kQuant) {
                        const float w0 = x[j] != -INFINITY ? p0 * vs[j] : 0.f;
                        const float w1 = x[j + 1] != -INFINITY ? p1 * vs[j + 1] : 0.f;
                        pk[j / 2] = pack_half2(w0, w1);
                    } else {
                        pk[j / 2] = pack_bf162(p0, p1);
                    }
                }
                l_run += lsum;
                tmem_st32(lane_tm + C::kSCol + b * kTile, pk);
                tmem_wait_st();
            }
            if (!C::kQuant && it.k_begin + i * kTile + kTile > it.k_end) {
                // last tile of the item: rows past the split end hold whatever
                // the cache has there; zero them so that 0 * V stays 0 in P x V
                const int key0 = it.k_begin + i * kTile;
                const int buf = i % C::kNumBuf;
                if (!mbar_wait(bar(kVFull + buf), (i / C::kNumBuf) & 1, kWaitNs)) ok = false;
                const int valid = it.k_end - key0;
                unsigned char *vb = smem + L.conv_v + buf * C::kConvBytes;
                const int qt = (warp - 2) * 32 + lane;  // 0..127 over the 4 softmax warps
                for (int e = qt; e < (kTile - valid) * (D / 8); e += 128) {
                    const int row = valid + e / (D / 8), u16 = e % (D / 8);
                    *reinterpret_cast<uint4 *>(vb + (u16 / 8) * C::kChunkBytes + sw128(row, u16 % 8)) =
                        make_uint4(0, 0, 0, 0);
                }
                fence_proxy_async_smem();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kPFull + b));
        }
        // epilogue: O / l and the log-sum-exp
        if (!mbar_wait(bar(kOFinal), 0, kWaitNs)) ok = false;
        tc_fence_after();
        if (warp_active && ok) {
            const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
            const float lse_nat = l_run > 0.f ? (m_run + log2f(l_run)) * 0.69314718055994531f : -INFINITY;
            const int rr = row0 + r;
            const int h = it.kvh * G + rr % G;
            const size_t orow = (size_t)(it.b * T + t_r) * p.Hq + h;
            const size_t prow = (size_t)it.part * p.rows_per_group + r;
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t o[32];
                tmem_ld32(lane_tm + C::kOCol + c0, o);
                tmem_wait_ld();
                if (!row_ok) continue;
                if (it.part < 0) {
                    uint4 *dst = reinterpret_cast<uint4 *>(p.out + orow * D + c0);
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        uint4 w;
                        w.x = pack_bf162(__uint_as_float(o[8 * k + 0]) * inv, __uint_as_float(o[8 * k + 1]) * inv);
                        w.y = pack_bf162(__uint_as_float(o[8 * k + 2]) * inv, __uint_as_float(o[8 * k + 3]) * inv);
                        w.z = pack_bf162(__uint_as_float(o[8 * k + 4]) * inv, __uint_as_float(o[8 * k + 5]) * inv);
                        w.w = pack_bf162(__uint_as_float(o[8 * k + 6]) * inv, __uint_as_float(o[8 * k + 7]) * inv);
                        dst[k] = w;
                    }
                } else {
                    float4 *dst = reinterpret_cast<float4 *>(p.o_part + prow * D + c0);
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        dst[k] = make_float4(__uint_as_float(o[4 * k]) * inv, __uint_as_float(o[4 * k + 1]) * inv,
                                             __uint_as_float(o[4 * k + 2]) * inv,
                                             __uint_as_float(o[4 * k + 3]) * inv);
                }
            }
            if (row_ok) {
                if (it.part < 0) {
                    if (p.lse) p.lse[orow] = lse_nat;
                } else {
                    p.lse_part[prow] = lse_nat;
                }
            }
        }
    } else if (C::kQuant) {
        // ------------------------------------------------------------ dequant
        const int dt = tid - 6 * 32;  // 0..127
        const int dwarp = warp - 6;
        float *ring = reinterpret_cast<float *>(smem + L.scale_ring);
        constexpr int kChunks = kRawKeys * D / 16;  // 16-byte raw chunks per half tile
        for (int i = 0; i < ntiles && ok; ++i) {
            const int buf = i % C::kNumBuf, use = i / C::kNumBuf;
            const int key0 = it.k_begin + i * kTile;
            float *ks_out = ring + (i % kScaleRing) * 2 * kTile;
            float *vs_out = ks_out + kTile;
#pragma unroll 1
            for (int kv = 0; kv < 2 && ok; ++kv) {
                const int empty_bar = kv == 0 ? kKEmpty : kVEmpty;
                if (!mbar_wait(bar(empty_bar + buf), (use & 1) ^ 1, kWaitNs)) { ok = false; break; }
                unsigned char *dst = smem + (kv == 0 ? L.conv_k : L.conv_v) + buf * C::kConvBytes;
#pragma unroll 1
                for (int h = 0; h < 2; ++h) {
                    const int rs = 2 * i + h;
                    const int hkey0 = key0 + h * kRawKeys;
                    const bool have = hkey0 < it.k_end;
                    const int slot = rs % kRawStages;
                    if (have && !mbar_wait(bar(kRawFull + slot), (rs / kRawStages) & 1, kWaitNs)) {
                        ok = false;
                        break;
                    }
                    const unsigned char *st = smem + L.raw + slot * L.raw_stride;
                    const unsigned char *src = st + (kv == 0 ? 0 : L.raw_v);
#pragma unroll 2
                    for (int q = dt; q < kChunks; q += 128) {
                        const int n = q * 16 / D;            // key within the half tile
                        const int d0 = (q * 16) % D;
                        const int row = h * kRawKeys + n;    // key within the 64-key tile
                        const int key = hkey0 + n;
                        uint4 w = make_uint4(0, 0, 0, 0);
                        if (have && key < it.k_end) {
                            const uint4 raw = *reinterpret_cast<const uint4 *>(src + n * D + d0);
                            const uint32_t rw[4] = {raw.x, raw.y, raw.z, raw.w};
                            uint32_t hw[8];
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                if (DT == VA_INT8)
                                    int8x4_to_half2x2(rw[k], hw[2 * k], hw[2 * k + 1]);
                                else
                                    e4m3x4_to_half2x2(rw[k], hw[2 * k], hw[2 * k + 1]);
                            }
                            const int c = d0 / 64, u0 = (d0 % 64) / 8;
                            const uint4 lo = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                            const uint4 hi = make_uint4(hw[4], hw[5], hw[6], hw[7]);
                            unsigned char *cb = dst + c * C::kChunkBytes;
                            if (c & 1) {  // alternate the store order between chunks: no bank conflicts
                                *reinterpret_cast<uint4 *>(cb + sw128(row, u0 + 1)) = hi;
                                *reinterpret_cast<uint4 *>(cb + sw128(row, u0)) = lo;
                            } else {
                                *reinterpret_cast<uint4 *>(cb + sw128(row, u0)) = lo;
                                *reinterpret_cast<uint4 *>(cb + sw128(row, u0 + 1)) = hi;
                            }
                        } else {
                            const int c = d0 / 64, u0 = (d0 % 64) / 8;
                            unsigned char *cb = dst + c * C::kChunkBytes;
                            *reinterpret_cast<uint4 *>(cb + sw128(row, u0)) = w;
                            *reinterpret_cast<uint4 *>(cb + sw128(row, u0 + 1)) = w;
                        }
                    }
                    // this head's k and v scales of the 32 keys, published
                    // with K (the softmax of this tile needs both)
                    if (kv == 0 && dt < 2 * kRawKeys) {
                        const int n = dt % kRawKeys, which = dt / kRawKeys;
                        const float *sc = reinterpret_cast<const float *>(st + (which == 0 ? L.raw_ks : L.raw_vs));
                        float v = 0.f;
                        if (have && hkey0 + n < it.k_end) v = sc[(n / VA_PAGE_SIZE) * VA_PAGE_SIZE * Hkv +
                                                                 (n % VA_PAGE_SIZE) * Hkv + it.kvh];
                        (which == 0 ? ks_out : vs_out)[h * kRawKeys + n] = v;
                    }
                }
                if (!ok) break;
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar((kv == 0 ? kKFull : kVFull) + buf));
            }
            if (!ok) break;
            // both K and V of the two raw stages have been read
            __syncwarp();
            if (lane == 0)
                for (int h = 0; h < 2; ++h)
                    if (key0 + h * kRawKeys < it.k_end) mbar_arrive(bar(kRawEmpty + (2 * i + h) % kRawStages));
            (void)dwarp;
        }
    }

    if (!ok) atomicOr(p.flags, kFlagTimeout);
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
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

// 4-D view of a page pool [pages, 16, Hkv, D]: dims innermost first.
bool make_map(CUtensorMap *m, const void *base, int D, int Hkv, int num_pages, bool bf16) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t eb = bf16 ? 2 : 1;
    const cuuint64_t pages = num_pages > 0 ? (cuuint64_t)num_pages : (cuuint64_t)1 << 30;
    cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)Hkv, (cuuint64_t)VA_PAGE_SIZE, pages};
    cuuint64_t strides[3] = {D * eb, (cuuint64_t)Hkv * D * eb, (cuuint64_t)VA_PAGE_SIZE * Hkv * D * eb};
    cuuint32_t box[4] = {bf16 ? 64u : (cuuint32_t)D, 1u, (cuuint32_t)VA_PAGE_SIZE, 1u};
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
    const bool bf16 = DT == VA_BF16;
    if (!make_map(&mp.tm_k, p.k_pages, D, p.Hkv, p.num_pages, bf16) ||
        !make_map(&mp.tm_v, p.v_pages, D, p.Hkv, p.num_pages, bf16))
        return cudaErrorInvalidValue;
    const Smem<D, DT> L(p.Hkv);
    const size_t smem = L.total + 1024;  // + alignment slack
    auto k = mma_partial_kernel<D, DT>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    k<<<n, Cfg<D, DT>::kThreads, smem, s>>>(mp);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const PartialParams &p, int dtype, int n, cudaStream_t s) {
    switch (dtype) {
    case VA_BF16: return launch_one<D, VA_BF16>(p, n, s);
    case VA_FP8_E4M3: return launch_one<D, VA_FP8_E4M3>(p, n, s);
    default: return launch_one<D, VA_INT8>(p, n, s);
    }
}

}  // namespace

size_t mma_smem_bytes(int head_dim, int kv_dtype, int Hkv) {
    switch (head_dim) {
    case 64:
        return kv_dtype == VA_BF16 ? Smem<64, VA_BF16>(Hkv).total + 1024 : Smem<64, VA_INT8>(Hkv).total + 1024;
    case 128:
        return kv_dtype == VA_BF16 ? Smem<128, VA_BF16>(Hkv).total + 1024 : Smem<128, VA_INT8>(Hkv).total + 1024;
    default:
        return kv_dtype == VA_BF16 ? Smem<256, VA_BF16>(Hkv).total + 1024 : Smem<256, VA_INT8>(Hkv).total + 1024;
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
