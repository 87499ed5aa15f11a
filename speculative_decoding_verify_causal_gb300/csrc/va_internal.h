// Internal declarations shared by the library's translation units (never
// installed; the public surface is include/verify_attn.h).
#pragma once

#include <cuda_runtime.h>

#include <utility>
#include <stdint.h>

#include "verify_attn.h"

namespace va {

// One CTA's work: the packed rows of row group `rg` of kv head `kvh` of
// sequence `b`, over keys [k_begin, k_end).  `L` is the planned sequence
// length; `part` is the partial slot to write, or -1 when this item covers the
// whole sequence and writes the final output directly.
struct Item {
    int b, kvh, rg, k_begin, k_end, L, part, pad;
};

// One (sequence, kv head, row group) whose splits the combine merges.
struct Group {
    int b, kvh, rg, first_part, n, pad0, pad1, pad2;
};

enum : int { kFlagBadPage = 1, kFlagSeqLenMismatch = 2 };

// Everything a partial-attention kernel needs, passed by value.
struct PartialParams {
    const uint16_t *q;          // bf16 [B, T, Hq, D]
    const void *k_pages;        // [num_pages, 16, Hkv, D]
    const void *v_pages;
    const float *k_scale;       // [num_pages, 16, Hkv] or null (bf16)
    const float *v_scale;
    const int32_t *block_table; // [B, bt_stride]
    const int32_t *seq_lens;    // [B]
    uint16_t *out;              // bf16 [B, T, Hq, D]
    float *lse;                 // [B, T, Hq] or null
    const Item *items;
    float *o_part;              // [num_parts, rows_per_group, D]
    float *lse_part;            // [num_parts, rows_per_group]
    int *flags;
    int bt_stride, T, Hq, Hkv, G, R, rows_per_group, num_pages;
    int num_parts;              // split partials in o_part / lse_part
    float sm_scale_log2;        // log2(e) / sqrt(D)
};

struct CombineParams {
    const Group *groups;
    const float *o_part;
    const float *lse_part;
    uint16_t *out;
    float *lse;
    int T, Hq, G, R, rows_per_group, D;
};

// Launch `kernel` with programmatic dependent launch allowed: it may start
// while the previous kernel on the stream is finishing, and must execute
// griddepcontrol.wait before it touches memory that kernel may write.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Programmatic dependent launch, device side: wait until the previous grid on
// the stream has completed and its writes are visible.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Remember a failing CUDA call for verify_attn_last_cuda_error (thread-local).
void note_cuda_error(cudaError_t e);

// Whether the caller's pointers meet the alignment the partial kernel of
// `path` (a va_path, WARP or MMA) and the combine rely on.
bool aligned_for(int path, int kv_dtype, const void *q, const void *k_pages, const void *v_pages,
                 const float *k_scale, const float *v_scale, const int32_t *block_table,
                 const int32_t *seq_lens, const void *out, const float *lse);

// Kernel launchers (return cudaGetLastError() of the launch).
cudaError_t launch_warp_partial(const PartialParams &p, int head_dim, int kv_dtype,
                                int num_items, cudaStream_t s);
cudaError_t launch_combine(const CombineParams &p, int num_groups, int max_splits,
                           cudaStream_t s);
cudaError_t launch_mma_partial(const PartialParams &p, int head_dim, int kv_dtype,
                               int num_items, cudaStream_t s);
size_t mma_smem_bytes(int head_dim, int kv_dtype, int num_kv_heads);

// Geometry of each path.
constexpr int kWarpRows = 4;     // packed rows per work item, CUDA-core kernel
constexpr int kWarpTile = 32;    // split granularity (keys), CUDA-core kernel
constexpr int kWarpCtasPerSm = 4;  // resident CTAs of the CUDA-core kernel per SM (most variants)
// The CUDA-core kernel's register budget, and with it its resident CTAs per
// SM: four (128 registers) where that costs no spills, three for bf16 rows
// and the 4-row variant, whose wider slices spill at 128 (measured: 4 CTAs are
// 7-13 % faster on the 8-bit caches, 4 % slower on bf16).  The planner sizes
// the split for the same count, so that a plan is one wave.
__host__ __device__ constexpr int warp_rows_variant(int rows_per_item) {
    return rows_per_item <= 1 ? 1 : rows_per_item <= 2 ? 2 : 4;
}
__host__ __device__ constexpr int warp_ctas_per_sm(int kv_dtype, int rows_per_item) {
    return (kv_dtype == VA_BF16 || warp_rows_variant(rows_per_item) == 4) ? 3 : kWarpCtasPerSm;
}
// Packed rows per kv head up to which the planner picks the CUDA-core kernel:
// measured on GB300 (D = 128 / 256, bf16 / fp8 / int8 / int4, 256 to 262k
// tokens) it takes 0.54-0.81 of the tensor-core kernel's time at 1 row and
// 0.62-0.92 at 2, and from 3 rows on it is faster only at a few hundred
// tokens (0.94-1.21 of the time from 4k tokens).
constexpr int kWarpAutoMaxRows = 2;
inline int auto_path(int packed_rows) { return packed_rows <= kWarpAutoMaxRows ? VA_PATH_WARP : VA_PATH_MMA; }
constexpr int kMmaRows = 128;    // packed rows per work item, tcgen05 kernel (M)
constexpr int kMmaTile = 64;     // keys per tile, tcgen05 kernel (N of QK^T)
constexpr int kMmaMaxItemTokens = 16384;  // longest split of the tcgen05 kernel (page ids in smem)
constexpr size_t kMaxSmemPerBlock = 232448;  // opt-in dynamic shared memory per block (227 KB)

}  // namespace va
