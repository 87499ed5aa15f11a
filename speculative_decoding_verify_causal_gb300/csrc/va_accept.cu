// Speculative acceptance after the verify pass (the rejection sampler).
// Definition in verify_attn.h: greedy prefix match; sampled positions accept
// d[t] iff u q(d) < p(d) (q a point mass for lookup drafts, softmax of the raw
// draft logits with the temperature applied once otherwise); the first
// rejection emits a sample of max(0, p - q), a full acceptance the bonus
// sample of p_T, both as exponential races with Philox4x32-10 Gumbel variates.
//
// Two kernels.  stats_kernel, one thread-block cluster of 2, 4 or 8 CTAs per
// (sequence, position), each CTA a slice of the vocabulary, partial results
// exchanged through distributed shared memory (combined in rank order, so
// every CTA and every run gets the same binary32 value): the maximum and
// argmax of z / tau (of z when greedy), the log-sum-exp and p(d), and the
// same for the draft logits.  decide_kernel, a row of CTAs per sequence:
// every CTA evaluates all positions with those statistics in parallel (the
// same uniforms, so the same first rejection n), then each CTA runs the
// sequence's one race over its slice of the vocabulary and folds its best key
// into the sequence's slot with a 64-bit atomic maximum (order-free, so the
// winner does not depend on timing); the last CTA to finish writes the
// tokens.  Each vocabulary row is read once per pass, fp32, coalesced.
#include <math.h>

#include <algorithm>
#include <atomic>

#include "va_internal.h"
#include "va_sm100.cuh"

namespace va {
namespace {

using namespace sm100;

constexpr int kThreads = 1024;
// CTAs per vocabulary row in the statistics: 8 for up to 8 rows, 4 while the
// rows fit one wave of the GPU at that width, else 2 (measured on GB300 at
// 151,936 entries, greedy / sampled: 6 rows 6.8 / 14.2 us with 8 against
// 7.3 / 15.4 with 4; 17 rows 7.4 / 15.7 with 4 against 9.0 / 18.3 with 8;
// 384 rows 49.6 / 129.8 with 2 against 81.6 / 192.3 with 8 and 48.7 / 144.6
// with 1).  Larger slices per CTA amortise the cluster's barriers until too
// few SMs are left working.
constexpr int kClusterMax = 8;
constexpr int kClusterWide = 4;
constexpr int kClusterNarrow = 2;
constexpr int kClusterMaxRows = 8;
constexpr int kRaceThreads = 256;    // decide_kernel CTA size
constexpr int kRacePerThread = 4;    // vocabulary entries per race thread (sets the row of CTAs)
constexpr int kMaxRaceCtas = 1024;

struct PosStats {  // one (sequence, position); 32 bytes
    float lse_p, p_d, q_d, lse_q;
    int argmax, pad[3];
};

struct SeqSlot {  // one sequence's race, after the PosStats block; 16 bytes
    unsigned long long key;  // best (score, index) key so far
    unsigned int done;       // race CTAs finished
    unsigned int pad;
};

struct AcceptParams {
    const float *z;       // [B, T+1, V]
    const float *w;       // [B, T, V] or null
    const int32_t *d;     // [B, T]
    const float *tau;     // [B]
    PosStats *stats;      // [B, T+1]
    SeqSlot *slots;       // [B], cleared by stats_kernel
    int32_t *out;         // [B, T+1]
    int32_t *nacc;        // [B]
    unsigned long long seed;
    int B, T, V;
};

// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11): 10 rounds of two 32x32
// multiplies, the key bumped by the Weyl constants between rounds; all four
// output words (the compiler drops what a caller does not use).
__device__ __forceinline__ uint4 philox4(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3, uint32_t k0,
                                         uint32_t k1) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint32_t hi0 = __umulhi(0xD2511F53u, c0), lo0 = 0xD2511F53u * c0;
        const uint32_t hi1 = __umulhi(0xCD9E8D57u, c2), lo1 = 0xCD9E8D57u * c2;
        const uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
        c0 = n0;
        c1 = lo1;
        c2 = n2;
        c3 = lo0;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return make_uint4(c0, c1, c2, c3);
}

// U(b, t, i, k) = (j + 0.5) / 2^24 = (2j + 1) / 2^25, j the top 24 bits of word (i mod 4) of Philox
// on counter (i / 4, t, b, k): one Philox call serves four consecutive vocabulary entries.  The
// 25-bit odd numerator is exact in binary32 only below 2^24.
__device__ __forceinline__ uint4 uniform_bits4(const AcceptParams &p, int b, int t, int c, int k) {
    const uint4 w = philox4((uint32_t)c, (uint32_t)t, (uint32_t)b, (uint32_t)k, (uint32_t)p.seed,
                            (uint32_t)(p.seed >> 32));
    return make_uint4(w.x >> 8, w.y >> 8, w.z >> 8, w.w >> 8);
}

// U in binary32 rounded toward zero: within one ulp of U and strictly inside (0, 1) (rounding to
// nearest would give 1.0 for j = 2^24 - 1).
__device__ __forceinline__ float uniform01(uint32_t j) {
    return __uint2float_rz(2u * j + 1u) * 2.98023223876953125e-8f;  // 2^-25
}

// -ln U to a few ulps for every j, also where U is within 2^-24 of 1 and -ln U is as small as
// 2^-25: U = u_hi + u_lo with u_hi the nearest binary32 and u_lo = 0 or +-2^-25 (exact), and
// ln U = ln u_hi + ln(1 + u_lo / u_hi).  Below j = 2^23 the numerator 2j + 1 fits 24 bits and
// u_lo = 0; above, it lies halfway between 2j and 2j + 2 and rounds to the even significand (2j
// for even j, so u_lo = +2^-25; 2j + 2 for odd j, u_lo = -2^-25).  There u_hi is in [0.5, 1] and
// u_lo (2 - u_hi) stands for u_lo / u_hi to within half an ulp of -ln U.
__device__ __forceinline__ float neg_log_uniform(uint32_t j) {
    const float u_hi = __uint2float_rn(2u * j + 1u) * 2.98023223876953125e-8f;  // 2^-25
    const float u_lo = j < (1u << 23) ? 0.f : ((j & 1u) ? -2.98023223876953125e-8f : 2.98023223876953125e-8f);
    return -logf(u_hi) - u_lo * (2.f - u_hi);
}

// Order-preserving map of a float to uint32 (larger float, larger code).
__device__ __forceinline__ uint32_t ordered(float f) {
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float unordered(uint32_t o) {
    return __uint_as_float((o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o);
}

// key = (ordered value, smallest index wins ties); -0 is keyed as +0, so that
// equal values tie whatever their sign
__device__ __forceinline__ unsigned long long vkey(float v, int i) {
    return ((unsigned long long)ordered(v + 0.f) << 32) | (0xFFFFFFFFu - (uint32_t)i);
}

__device__ unsigned long long block_max_u64(unsigned long long v, unsigned long long *red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long x = __shfl_xor_sync(0xffffffffu, v, o);
        v = x > v ? x : v;
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();  // red may still be read by a previous reduction
    if (lane == 0) red[warp] = v;
    __syncthreads();
    v = lane < (int)(blockDim.x >> 5) ? red[lane] : 0ull;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long x = __shfl_xor_sync(0xffffffffu, v, o);
        v = x > v ? x : v;
    }
    return v;
}

__device__ float block_sum(float v, float *red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    v = lane < (int)(blockDim.x >> 5) ? red[lane] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Cluster-wide max of one 64-bit key per CTA (slot: this CTA's shared word).
__device__ unsigned long long cluster_max_u64(unsigned long long v, unsigned long long *slot) {
    if (threadIdx.x == 0) *slot = v;
    cluster_sync();
    unsigned long long m = 0;
    const uint32_t n = cluster_size();
    for (uint32_t r = 0; r < n; ++r) {
        const unsigned long long x = ld_cluster_u64(slot, r);
        m = x > m ? x : m;
    }
    cluster_sync();  // slots may be rewritten after this
    return m;
}

// Cluster-wide sum of one float per CTA, added in rank order.
__device__ float cluster_sum(float v, float *slot) {
    if (threadIdx.x == 0) *slot = v;
    cluster_sync();
    float s = 0.f;
    const uint32_t n = cluster_size();
    for (uint32_t r = 0; r < n; ++r) s += ld_cluster_f32(slot, r);
    cluster_sync();
    return s;
}

// This CTA's slice [lo, hi) of a V-long row; lo is a multiple of `unit`.
__device__ __forceinline__ void slice(int V, int &lo, int &hi, int unit = 1) {
    const int r = (int)cluster_rank(), n = (int)cluster_size();
    const int per = ((V + n - 1) / n + unit - 1) / unit * unit;
    lo = min(V, r * per);
    hi = min(V, lo + per);
}

constexpr int kVec = 4;  // 16-byte loads of a thread issued together in a row pass

// f(i, row[i]) for every i of [lo, hi).  With a 16-byte aligned row and V a
// multiple of 4 (then lo and hi are too): rounds of kVec unconditional
// 16-byte loads per thread, all issued before any is used, then single
// 16-byte loads for the rest; otherwise one entry at a time.
template <typename F>
__device__ __forceinline__ void row_pass(const float *row, int lo, int hi, bool vec, F f) {
    const int step = (int)blockDim.x;
    if (!vec) {
        for (int i = lo + (int)threadIdx.x; i < hi; i += step) f(i, row[i]);
        return;
    }
    const float4 *r4 = reinterpret_cast<const float4 *>(row);
    const int hi4 = hi >> 2;
    int j = (lo >> 2) + (int)threadIdx.x;
    for (; j + (kVec - 1) * step < hi4; j += kVec * step) {
        float4 x[kVec];
#pragma unroll
        for (int u = 0; u < kVec; ++u) x[u] = __ldg(r4 + j + u * step);
#pragma unroll
        for (int u = 0; u < kVec; ++u) {
            const int i = 4 * (j + u * step);
            f(i, x[u].x);
            f(i + 1, x[u].y);
            f(i + 2, x[u].z);
            f(i + 3, x[u].w);
        }
    }
    for (; j < hi4; j += step) {
        const float4 x = __ldg(r4 + j);
        f(4 * j, x.x);
        f(4 * j + 1, x.y);
        f(4 * j + 2, x.z);
        f(4 * j + 3, x.w);
    }
}

// Folds N scaled values (value k at vocabulary index index(k), increasing in
// k) into a thread's running maximum m, its first index mi and the sum s of
// exp(v - m): the round's maximum first; if it beats m, its first position
// in the round and one rescale of s; then the round's exponentials (two
// partial sums).
template <int N, typename I>
__device__ __forceinline__ void fold_round(float &m, int &mi, float &s, const float (&v)[N], I index) {
    float rm = v[0];
#pragma unroll
    for (int k = 1; k < N; ++k) rm = fmaxf(rm, v[k]);
    if (rm > m) {
        int ri = 0;
#pragma unroll
        for (int k = N - 1; k >= 0; --k)
            if (v[k] == rm) ri = index(k);
        s *= expf(m - rm);  // 0 while m is still -inf
        m = rm;
        mi = ri;
    }
    if (m > -INFINITY) {
        float a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int k = 0; k < N; k += 2) {
            a0 += expf(v[k] - m);
            if (k + 1 < N) a1 += expf(v[k + 1] - m);
        }
        s += a0 + a1;
    }
}

// Row statistics over the cluster: max (and its smallest index) of row * scale,
// and the log-sum-exp of row * scale when want_lse.
__device__ void row_stats(const float *row, int V, float scale, bool want_lse, unsigned long long *redk,
                          float *redf, unsigned long long *slot_k, float *slot_f, float &lse, int &argmax) {
    const bool vec = (V & 3) == 0 && (reinterpret_cast<uintptr_t>(row) & 15u) == 0;
    int lo, hi;
    slice(V, lo, hi, vec ? 4 : 1);
    // per thread: the largest value and its first index (a thread visits its
    // indices in increasing order, so a strict compare keeps the smallest
    // index of a tie); the 64-bit (value, index) key is formed once per thread
    float tmax = -INFINITY, tsum = 0.f;
    int tidx = -1;
    if (!want_lse) {
        row_pass(row, lo, hi, vec, [&](int i, float x) {
            const float v = x * scale;
            if (v > tmax) {
                tmax = v;
                tidx = i;
            }
        });
    } else if (vec) {
        // one read of the row: the running sum of exp(v - running max),
        // rescaled at most once per round of kVec 16-byte loads
        const int step = (int)blockDim.x;
        const float4 *r4 = reinterpret_cast<const float4 *>(row);
        const int hi4 = hi >> 2;
        int j = (lo >> 2) + (int)threadIdx.x;
        for (; j + (kVec - 1) * step < hi4; j += kVec * step) {
            float4 x[kVec];
#pragma unroll
            for (int u = 0; u < kVec; ++u) x[u] = __ldg(r4 + j + u * step);
            float v[4 * kVec];
#pragma unroll
            for (int u = 0; u < kVec; ++u) {
                v[4 * u] = x[u].x * scale;
                v[4 * u + 1] = x[u].y * scale;
                v[4 * u + 2] = x[u].z * scale;
                v[4 * u + 3] = x[u].w * scale;
            }
            fold_round(tmax, tidx, tsum, v, [&](int k) { return 4 * (j + (k >> 2) * step) + (k & 3); });
        }
        for (; j < hi4; j += step) {
            const float4 x = __ldg(r4 + j);
            const float v[4] = {x.x * scale, x.y * scale, x.z * scale, x.w * scale};
            fold_round(tmax, tidx, tsum, v, [&](int k) { return 4 * j + k; });
        }
    } else {
        for (int i = lo + (int)threadIdx.x; i < hi; i += (int)blockDim.x) {
            const float v[1] = {row[i] * scale};
            fold_round(tmax, tidx, tsum, v, [&](int) { return i; });
        }
    }
    unsigned long long k = 0;
    if (tidx >= 0) {
        k = vkey(tmax, tidx);
    } else {  // nothing above -inf here: the smallest index this thread visited
        const int first = vec ? 4 * ((lo >> 2) + (int)threadIdx.x) : lo + (int)threadIdx.x;
        if (first < hi) k = vkey(-INFINITY, first);
    }
    k = cluster_max_u64(block_max_u64(k, redk), slot_k);
    argmax = (int)(0xFFFFFFFFu - (uint32_t)(k & 0xFFFFFFFFull));
    if (!want_lse) return;
    const float m = unordered((uint32_t)(k >> 32));
    // this thread's sum moved from its own maximum to the row's (tmax <= m)
    float sum = tidx >= 0 ? tsum * expf(tmax - m) : 0.f;
    sum = cluster_sum(block_sum(sum, redf), slot_f);
    lse = m + logf(sum);
}

__global__ void __launch_bounds__(kThreads, 2) stats_kernel(const AcceptParams p) {
    __shared__ unsigned long long redk[kThreads / 32];
    __shared__ float redf[kThreads / 32];
    __shared__ unsigned long long slot_k;
    __shared__ float slot_f;
    griddep_wait();
    const int t = blockIdx.y, b = blockIdx.z;
    const float tau = p.tau[b];
    const bool greedy = !(tau > 0.f);
    const float inv = greedy ? 1.f : 1.f / tau;
    const float *z = p.z + ((size_t)b * (p.T + 1) + t) * p.V;
    if (t == 0 && cluster_rank() == 0 && threadIdx.x == 0) p.slots[b] = SeqSlot{};  // for decide_kernel
    PosStats st{};
    row_stats(z, p.V, inv, !greedy, redk, redf, &slot_k, &slot_f, st.lse_p, st.argmax);
    if (!greedy && t < p.T) {
        const int d = p.d[(size_t)b * p.T + t];
        const bool valid = d >= 0 && d < p.V;
        st.p_d = valid ? expf(z[d] * inv - st.lse_p) : 0.f;
        if (p.w) {
            const float *w = p.w + ((size_t)b * p.T + t) * p.V;
            int am;
            row_stats(w, p.V, inv, true, redk, redf, &slot_k, &slot_f, st.lse_q, am);
            st.q_d = valid ? expf(w[d] * inv - st.lse_q) : 0.f;
        } else {
            st.q_d = valid ? 1.f : 0.f;
        }
    }
    if (cluster_rank() == 0 && threadIdx.x == 0) p.stats[(size_t)b * (p.T + 1) + t] = st;
}

__device__ void write_tokens(const AcceptParams &p, int b, int n, int tok) {
    const int32_t *d = p.d + (size_t)b * p.T;
    for (int t = threadIdx.x; t <= p.T; t += blockDim.x)
        p.out[(size_t)b * (p.T + 1) + t] = t < n ? d[t] : (t == n ? tok : -1);
    if (threadIdx.x == 0) p.nacc[b] = n;
}

__global__ void __launch_bounds__(kRaceThreads) decide_kernel(const AcceptParams p) {
    __shared__ unsigned long long redk[kRaceThreads / 32];
    __shared__ int s_n;
    __shared__ int s_last;
    griddep_wait();
    const int b = blockIdx.y;
    const float tau = p.tau[b];
    const bool greedy = !(tau > 0.f);
    const PosStats *st = p.stats + (size_t)b * (p.T + 1);
    const int32_t *d = p.d + (size_t)b * p.T;
    // n = the first position whose draft is rejected (T if none is)
    if (threadIdx.x == 0) s_n = p.T;
    __syncthreads();
    for (int t = threadIdx.x; t < p.T; t += blockDim.x) {
        const bool valid = d[t] >= 0 && d[t] < p.V;
        const bool ok = greedy ? (valid && d[t] == st[t].argmax)
                               : (valid && uniform01(uniform_bits4(p, b, t, 0, 0).x) * st[t].q_d < st[t].p_d);
        if (!ok) atomicMin(&s_n, t);
    }
    __syncthreads();
    const int n = s_n;
    if (greedy) {
        if (blockIdx.x == 0) write_tokens(p, b, n, st[n].argmax);
        return;
    }
    // the race: this CTA's slice of the vocabulary, in groups of four
    // entries that share one Philox counter (16-byte loads of the logits
    // where the rows allow); scores in units of ln 2, the outer logarithm
    // of the Gumbel and ln r taken by the hardware base-2 logarithm
    // (absolute error about 1e-6, far below any race margin that matters)
    const float inv = 1.f / tau;
    const float *z = p.z + ((size_t)b * (p.T + 1) + n) * p.V;
    const bool bonus = n == p.T;
    const int dn = bonus ? -1 : d[n];
    const float *w = (!bonus && p.w) ? p.w + ((size_t)b * p.T + n) * p.V : nullptr;
    const bool vec = (p.V & 3) == 0 && (reinterpret_cast<uintptr_t>(z) & 15u) == 0 &&
                     (!w || (reinterpret_cast<uintptr_t>(w) & 15u) == 0);
    const float lse_p = st[n].lse_p, lse_q = st[n].lse_q;
    const int groups = (p.V + 3) >> 2;
    const int per = (groups + (int)gridDim.x - 1) / (int)gridDim.x;
    const int lo = min(groups, (int)blockIdx.x * per), hi = min(groups, lo + per);
    unsigned long long k = 0;
    for (int c = lo + (int)threadIdx.x; c < hi; c += blockDim.x) {
        const uint4 j4 = uniform_bits4(p, b, n, c, 1);
        const uint32_t js[4] = {j4.x, j4.y, j4.z, j4.w};
        const int i0 = 4 * c;
        float zv[4], wv[4];
        if (vec) {
            const float4 a = __ldg(reinterpret_cast<const float4 *>(z) + c);
            zv[0] = a.x, zv[1] = a.y, zv[2] = a.z, zv[3] = a.w;
            if (w) {
                const float4 e = __ldg(reinterpret_cast<const float4 *>(w) + c);
                wv[0] = e.x, wv[1] = e.y, wv[2] = e.z, wv[3] = e.w;
            }
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                zv[e] = i0 + e < p.V ? z[i0 + e] : 0.f;
                if (w) wv[e] = i0 + e < p.V ? w[i0 + e] : 0.f;
            }
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int i = i0 + e;
            if (i >= p.V) break;
            const float g2 = -__log2f(neg_log_uniform(js[e]));  // Gumbel / ln 2
            float score;  // in units of ln 2
            if (w) {
                const float r = expf(zv[e] * inv - lse_p) - expf(wv[e] * inv - lse_q);
                score = r > 0.f ? __log2f(r) + g2 : -INFINITY;
            } else {
                score = i == dn ? -INFINITY : fmaf(zv[e], inv * 1.4426950408889634f, g2);
            }
            const unsigned long long key = vkey(score, i);
            k = key > k ? key : k;
        }
    }
    k = block_max_u64(k, redk);
    SeqSlot *slot = p.slots + b;
    if (threadIdx.x == 0) {
        atomicMax(&slot->key, k);
        __threadfence();  // the maximum is visible before this CTA counts as done
        s_last = atomicAdd(&slot->done, 1u) == gridDim.x - 1;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    const unsigned long long best = atomicAdd(&slot->key, 0ull);  // every CTA's maximum is in
    write_tokens(p, b, n, (int)(0xFFFFFFFFu - (uint32_t)(best & 0xFFFFFFFFull)));
}

// Launch with a (cluster, 1, 1) cluster and programmatic dependent launch.
template <typename K>
cudaError_t launch_cluster(K kernel, dim3 grid, int cluster, cudaStream_t s, const AcceptParams &p) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kernel, p);
}

}  // namespace
}  // namespace va

extern "C" size_t verify_attn_accept_workspace_bytes(int num_seqs, int T) {
    if (num_seqs < 1 || T < 1) return 0;
    return sizeof(va::PosStats) * (size_t)num_seqs * (size_t)(T + 1) + sizeof(va::SeqSlot) * (size_t)num_seqs;
}

extern "C" int verify_attn_accept(const float *target_logits, const float *draft_logits,
                                  const int32_t *draft_tokens, const float *temperature, int num_seqs, int T,
                                  int vocab, uint64_t seed, void *workspace, int32_t *out_tokens,
                                  int32_t *num_accepted, void *stream) {
    if (!target_logits || !draft_tokens || !temperature || !workspace || !out_tokens || !num_accepted)
        return VA_ERR_INVALID_ARGUMENT;
    if (num_seqs < 1 || num_seqs > 65535 || T < 1 || T > 65535 || vocab < 1) return VA_ERR_INVALID_ARGUMENT;
    if ((reinterpret_cast<uintptr_t>(workspace) & 15u) != 0) return VA_ERR_INVALID_ARGUMENT;
    va::AcceptParams p{};
    p.z = target_logits;
    p.w = draft_logits;
    p.d = draft_tokens;
    p.tau = temperature;
    p.stats = static_cast<va::PosStats *>(workspace);
    p.slots = reinterpret_cast<va::SeqSlot *>(p.stats + (size_t)num_seqs * (size_t)(T + 1));
    p.out = out_tokens;
    p.nacc = num_accepted;
    p.seed = seed;
    p.B = num_seqs;
    p.T = T;
    p.V = vocab;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // resident race CTAs of the whole GPU (queried once per device)
    // the SM count and the race kernel's resident CTAs per SM, once per device
    static std::atomic<int> s_sms[64], s_race_per_sm[64];
    int dev = 0, sms = 0, race_per_sm = 0;
    if (cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < 64) {
        sms = s_sms[dev].load(std::memory_order_relaxed);
        race_per_sm = s_race_per_sm[dev].load(std::memory_order_relaxed);
        if (!sms || !race_per_sm) {
            if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) sms = 0;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&race_per_sm, va::decide_kernel, va::kRaceThreads, 0) !=
                cudaSuccess)
                race_per_sm = 0;
            s_sms[dev].store(sms, std::memory_order_relaxed);
            s_race_per_sm[dev].store(race_per_sm, std::memory_order_relaxed);
        }
    }
    cudaGetLastError();
    // statistics: two 1024-thread CTAs per SM are resident
    const long long rows = (long long)num_seqs * (T + 1);
    const int cluster = rows <= va::kClusterMaxRows                               ? va::kClusterMax
                        : (sms > 0 && rows * va::kClusterWide <= 2LL * sms) ? va::kClusterWide
                                                                            : va::kClusterNarrow;
    cudaError_t e = va::launch_cluster(va::stats_kernel, dim3(cluster, T + 1, num_seqs), cluster, s, p);
    const int slots = sms * race_per_sm;  // race CTAs resident on the whole GPU (0 if unknown)
    // A row of race CTAs per sequence: kRacePerThread vocabulary entries per
    // thread, but no more CTAs than one wave of the whole GPU spread over the
    // sequences (a greedy sequence's CTAs exit after the prefix match, so a
    // wide row only costs launches there; a sampled one loops over its slice).
    long long nrace = ((long long)vocab + va::kRaceThreads * va::kRacePerThread - 1) /
                      (va::kRaceThreads * va::kRacePerThread);
    if (slots > 0) nrace = std::min<long long>(nrace, std::max<long long>(1, slots / num_seqs));
    nrace = std::min<long long>(va::kMaxRaceCtas, std::max<long long>(1, nrace));
    if (e == cudaSuccess)
        e = va::launch_pdl(va::decide_kernel, dim3((unsigned)nrace, num_seqs), dim3(va::kRaceThreads), 0, s, p);
    if (e != cudaSuccess) {
        va::note_cuda_error(e);
        return VA_ERR_CUDA;
    }
    return VA_OK;
}
