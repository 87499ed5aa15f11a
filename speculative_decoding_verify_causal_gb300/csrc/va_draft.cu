// Lookup-augmented drafting ("I pushed Qwen3.8-27B to 381 tps for a single
// request on a RTX 3090", "Lookup-augmented drafting"): find the most recent
// earlier occurrence of the history's last tokens and propose what followed.
//
// One thread-block cluster per sequence (1 to 16 CTAs, from the history
// length bound; above 8, a non-portable size, used where the device can place
// it): CTA r scans the r-th slice of the end positions.  The last
// max_match tokens (reversed) sit in each CTA's shared memory; every thread
// walks end positions e (coalesced 4-byte loads of x[e], eight in flight per
// thread), extends a match
// backwards only when x[e] equals the last token, and keeps the best
// (length, e) as one 64-bit key (length in the high word, so the maximum is
// the longest match and, among equal lengths, the most recent end).  A block
// max-reduction, then CTA 0 reads the other CTAs' keys through distributed
// shared memory and its first num_draft threads copy the continuation.
#include <algorithm>
#include <atomic>

#include "va_internal.h"
#include "va_sm100.cuh"

namespace va {
namespace {

using namespace sm100;

constexpr int kThreads = 1024;
constexpr int kMaxMatch = 32;
constexpr int kMaxCluster = 8;          // portable cluster size (twice that where allowed)
constexpr int kTokensPerCta = 4096;     // history tokens per CTA of the cluster
constexpr int kUnroll = 8;              // end-token loads per thread in flight together

struct DraftParams {
    const int32_t *tokens;
    const int32_t *lens;
    int32_t *draft, *draft_len, *match_end, *match_len;
    int stride, min_match, max_match, num_draft;
};

__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long w = __shfl_xor_sync(0xffffffffu, v, o);
        v = w > v ? w : v;
    }
    return v;
}

__global__ void __launch_bounds__(kThreads) lookup_kernel(const DraftParams p) {
    __shared__ int32_t suf[kMaxMatch];                  // suf[i] = x[L - 1 - i]
    __shared__ unsigned long long wbest[kThreads / 32];
    griddep_wait();  // the history may come from the previous kernel on the stream
    const int b = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int rank = (int)cluster_rank(), nct = (int)cluster_size();
    const int32_t *x = p.tokens + (size_t)b * p.stride;
    int L = p.lens[b];
    if (L < 0 || L > p.stride) L = 0;  // out-of-contract length: treated as an empty history
    const int lmax = min(p.max_match, L);  // suffix tokens that exist
    if (tid < lmax) suf[tid] = x[L - 1 - tid];
    __syncthreads();
    unsigned long long best = 0;
    if (lmax >= p.min_match) {
        const int32_t last = suf[0];
        // this CTA's slice of end positions [0, L - 2]
        const int n_end = max(L - 1, 0), per = (n_end + nct - 1) / nct;
        const int e_hi = min(n_end, (rank + 1) * per);
        // kUnroll coalesced loads of end tokens per thread are issued before
        // any is compared, so that a thread's scan is a few memory round
        // trips instead of one per end position
        for (int e0 = rank * per + tid; e0 < e_hi; e0 += kThreads * kUnroll) {
            int32_t v[kUnroll];
#pragma unroll
            for (int k = 0; k < kUnroll; ++k) {
                const int e = e0 + k * kThreads;
                v[k] = e < e_hi ? x[e] : 0;
            }
#pragma unroll
            for (int k = 0; k < kUnroll; ++k) {
                const int e = e0 + k * kThreads;
                if (e >= e_hi || v[k] != last) continue;
                int l = 1;
                while (l < lmax && e - l >= 0 && x[e - l] == suf[l]) ++l;
                if (l >= p.min_match) {
                    const unsigned long long key = ((unsigned long long)l << 32) | (unsigned)e;
                    best = key > best ? key : best;
                }
            }
        }
    }
    best = warp_max_u64(best);
    if (lane == 0) wbest[warp] = best;
    __syncthreads();
    if (warp == 0) {
        best = warp_max_u64(lane < kThreads / 32 ? wbest[lane] : 0ull);
        if (lane == 0) wbest[0] = best;
    }
    cluster_sync();  // every CTA's key is in its shared memory
    if (rank == 0) {
        best = wbest[0];
        for (int r = 1; r < nct; ++r) {
            const unsigned long long o = ld_cluster_u64(&wbest[0], (uint32_t)r);
            best = o > best ? o : best;
        }
        const int e = best ? (int)(best & 0xffffffffull) : -1;
        const int n = best ? min(p.num_draft, L - 1 - e) : 0;
        for (int t = tid; t < p.num_draft; t += kThreads)
            p.draft[(size_t)b * p.num_draft + t] = t < n ? x[e + 1 + t] : -1;
        if (tid == 0) {
            p.draft_len[b] = n;
            if (p.match_end) p.match_end[b] = e;
            if (p.match_len) p.match_len[b] = best ? (int)(best >> 32) : 0;
        }
    }
    cluster_sync();  // the other CTAs' shared memory stays valid until CTA 0 has read it
}

}  // namespace
}  // namespace va

extern "C" int verify_attn_lookup_draft(const int32_t *tokens, int token_stride, const int32_t *lens,
                                        int num_seqs, int min_match, int max_match, int num_draft,
                                        int32_t *draft, int32_t *draft_len, int32_t *match_end,
                                        int32_t *match_len, void *stream) {
    if (!tokens || !lens || !draft || !draft_len) return VA_ERR_INVALID_ARGUMENT;
    if (num_seqs < 1 || num_seqs > 65535 || token_stride < 1 || min_match < 1 || max_match < min_match ||
        max_match > va::kMaxMatch || num_draft < 1 || num_draft > 256)
        return VA_ERR_INVALID_ARGUMENT;
    va::DraftParams p{};
    p.tokens = tokens;
    p.lens = lens;
    p.draft = draft;
    p.draft_len = draft_len;
    p.match_end = match_end;
    p.match_len = match_len;
    p.stride = token_stride;
    p.min_match = min_match;
    p.max_match = max_match;
    p.num_draft = num_draft;
    // cluster of CTAs per sequence: one per kTokensPerCta of the longest possible history,
    // up to 16 (a non-portable size, refused on parts that cannot place it: then 8)
    static std::atomic<int> s_wide{0};  // 0 unknown, 1 allowed, -1 refused
    int wide = s_wide.load(std::memory_order_relaxed);
    if (wide == 0) {
        // allowed, and at least one such cluster fits on the device
        wide = -1;
        if (cudaFuncSetAttribute(va::lookup_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
            cudaSuccess) {
            cudaLaunchConfig_t q = {};
            q.gridDim = dim3(2 * va::kMaxCluster, 1);
            q.blockDim = dim3(va::kThreads);
            cudaLaunchAttribute ca;
            ca.id = cudaLaunchAttributeClusterDimension;
            ca.val.clusterDim.x = 2 * va::kMaxCluster;
            ca.val.clusterDim.y = 1;
            ca.val.clusterDim.z = 1;
            q.attrs = &ca;
            q.numAttrs = 1;
            int nclusters = 0;
            if (cudaOccupancyMaxActiveClusters(&nclusters, va::lookup_kernel, &q) == cudaSuccess && nclusters >= 1)
                wide = 1;
        }
        (void)cudaGetLastError();
        s_wide.store(wide, std::memory_order_relaxed);
    }
    const int cap = wide > 0 ? 2 * va::kMaxCluster : va::kMaxCluster;
    int nct = std::min(cap, std::max(1, (token_stride + va::kTokensPerCta - 1) / va::kTokensPerCta));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(nct, num_seqs);
    cfg.blockDim = dim3(va::kThreads);
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = nct;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cudaError_t e = cudaLaunchKernelEx(&cfg, va::lookup_kernel, p);
    if (e != cudaSuccess && nct > va::kMaxCluster) {  // the wide cluster was refused: portable size
        (void)cudaGetLastError();
        s_wide.store(-1, std::memory_order_relaxed);
        nct = va::kMaxCluster;
        cfg.gridDim = dim3(nct, num_seqs);
        attr[0].val.clusterDim.x = nct;
        e = cudaLaunchKernelEx(&cfg, va::lookup_kernel, p);
    }
    if (e != cudaSuccess) {
        va::note_cuda_error(e);
        return VA_ERR_CUDA;
    }
    return VA_OK;
}
