// verify_attn_noalloc: the verify call for callers that cannot allocate
// device memory.
//
// A normal plan owns a cudaMalloc'ed workspace (work list + split partials).
// Some callers cannot call cudaMalloc at all: a serving runtime whose memory
// pool owns every byte of the device, a real-time path that must not take
// the allocator's locks, or an embedding that fixes its device footprint at
// start-up.  This entry point gives them the same kernels with their scratch
// in a file-scope device array of fixed size, VA_NOALLOC_SCRATCH_BYTES.
//
// In host code `g_noalloc_scratch` names a host-side stand-in, not device
// memory: its device address is fetched once per device with
// cudaGetSymbolAddress (that device current) and passed to the kernels.
// Every call shares the array and overwrites the previous call's contents;
// the flag word is cleared at the start of each call and can be read back
// with verify_attn_noalloc_flags.  The work list is staged in static host
// buffers and copied with cudaMemcpyAsync from pageable memory.  The partial
// kernel is the one a plan picks (CUDA cores up to two packed rows, tensor
// cores above), unless the tensor-core split partials cannot fit in the
// scratch at any split length its page-id staging allows: then the CUDA-core
// kernel runs, with splits as coarse as needed.
#include <cmath>
#include <mutex>

#include "va_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[VA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
constexpr size_t kFlagsBytes = 256;

std::mutex g_setup_mu;
void *g_scratch_dev[kMaxDevices];
int g_num_sms[kMaxDevices];

std::mutex g_host_mu;  // guards the host staging buffers below
// Work-list staging on the host (an item and a group are 32 bytes each);
// longer lists make the split coarser.
constexpr int kMaxItems = 65536;
va::Item g_host_items[kMaxItems];
va::Group g_host_groups[kMaxItems];

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

// Per-device set-up: the device address of the scratch array and the SM
// count, looked up once with the device current.
int device_setup(void **scratch, int *num_sms) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        va::note_cuda_error(e);
        cudaGetLastError();
        return VA_ERR_NO_DEVICE;
    }
    if (dev < 0 || dev >= kMaxDevices) return VA_ERR_NO_DEVICE;
    std::lock_guard<std::mutex> lk(g_setup_mu);
    if (!g_scratch_dev[dev]) {
        void *ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess || !ptr) {
            va::note_cuda_error(e);
            cudaGetLastError();
            return VA_ERR_CUDA;
        }
        int n = 0;
        e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess || n < 1) {
            va::note_cuda_error(e);
            cudaGetLastError();
            return VA_ERR_NO_DEVICE;
        }
        g_num_sms[dev] = n;
        g_scratch_dev[dev] = ptr;
    }
    *scratch = g_scratch_dev[dev];
    *num_sms = g_num_sms[dev];
    return VA_OK;
}

struct Layout {
    int rows_per_group, num_row_groups, tile, split;
    int num_items, num_groups, num_parts, max_splits;
    size_t off_items, off_groups, off_lse, off_o, total;
};

// Geometry of one split length; returns false if the counts overflow the
// host staging buffers.
bool layout_for(const int32_t *lens, int B, int Hkv, int D, int split, Layout &L) {
    L.split = split;
    long long items = 0, groups = 0, parts = 0;
    int max_splits = 1;
    for (int b = 0; b < B; ++b) {
        const int n = (lens[b] + split - 1) / split;
        max_splits = n > max_splits ? n : max_splits;
        const long long per = (long long)Hkv * L.num_row_groups;
        items += per * n;
        if (n > 1) {
            groups += per;
            parts += per * n;
        }
    }
    if (items > kMaxItems || groups > kMaxItems) return false;
    L.num_items = (int)items;
    L.num_groups = (int)groups;
    L.num_parts = (int)parts;
    L.max_splits = max_splits;
    L.off_items = kFlagsBytes;
    L.off_groups = align256(L.off_items + sizeof(va::Item) * items);
    L.off_lse = align256(L.off_groups + sizeof(va::Group) * groups);
    L.off_o = align256(L.off_lse + sizeof(float) * (size_t)parts * L.rows_per_group);
    L.total = align256(L.off_o + sizeof(float) * (size_t)parts * L.rows_per_group * D);
    return true;
}

// A failing CUDA call: remember it for verify_attn_last_cuda_error and
// reset the runtime's last-error state.
int cuda_fail(cudaError_t e) {
    va::note_cuda_error(e);
    cudaGetLastError();
    return VA_ERR_CUDA;
}

}  // namespace

extern "C" int verify_attn_noalloc(const int32_t *seq_lens_host, int B, int T, int Hq, int Hkv,
                                   int D, va_kv_dtype kv_dtype, const void *q, const void *k_pages,
                                   const void *v_pages, const float *k_scale,
                                   const float *v_scale, const int32_t *block_table,
                                   int block_table_stride, int num_pages, const int32_t *seq_lens,
                                   void *out, float *lse, void *stream) {
    if (!seq_lens_host || B < 1 || T < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv)
        return VA_ERR_INVALID_ARGUMENT;
    if (D != 64 && D != 128 && D != 256) return VA_ERR_UNSUPPORTED;
    if (kv_dtype < VA_BF16 || kv_dtype > VA_INT2) return VA_ERR_UNSUPPORTED;
    if (!q || !k_pages || !v_pages || !block_table || !seq_lens || !out)
        return VA_ERR_INVALID_ARGUMENT;
    if (kv_dtype != VA_BF16 && (!k_scale || !v_scale)) return VA_ERR_INVALID_ARGUMENT;
    int max_pages = 0;
    long long total_len = 0;
    int max_len = 0;
    for (int b = 0; b < B; ++b) {
        if (seq_lens_host[b] < T) return VA_ERR_INVALID_ARGUMENT;
        const int p = (seq_lens_host[b] + VA_PAGE_SIZE - 1) / VA_PAGE_SIZE;
        max_pages = p > max_pages ? p : max_pages;
        total_len += seq_lens_host[b];
        max_len = seq_lens_host[b] > max_len ? seq_lens_host[b] : max_len;
    }
    if (block_table_stride < 0 || (block_table_stride > 0 && block_table_stride < max_pages) || num_pages < 0)
        return VA_ERR_INVALID_ARGUMENT;
    const int bt_stride = block_table_stride > 0 ? block_table_stride : max_pages;

    // Geometry: the kernel a plan picks, with one wave of splits over the
    // SMs, made coarser until the split partials fit in the scratch; for the
    // tensor-core kernel (one resident CTA per SM) at most kMmaMaxItemTokens
    // keys per item, and when its partials cannot fit that way, the CUDA-core
    // kernel's geometry (several CTAs per SM, no limit on the split).  A
    // problem whose work list does not fit even unsplit is rejected here,
    // before any CUDA call.
    const int G = Hq / Hkv;
    const int R = G * T;
    auto geometry = [&](bool mma, Layout &L) {
        L = Layout{};
        L.num_row_groups = (R + (mma ? va::kMmaRows : va::kWarpRows) - 1) / (mma ? va::kMmaRows : va::kWarpRows);
        L.rows_per_group = (R + L.num_row_groups - 1) / L.num_row_groups;
        L.tile = mma ? va::kMmaTile : va::kWarpTile;
    };
    const bool mma_fits_smem = va::mma_smem_bytes(D, kv_dtype, Hkv) <= va::kMaxSmemPerBlock;
    Layout L{};
    geometry(false, L);
    const bool warp_possible = layout_for(seq_lens_host, B, Hkv, D, max_len, L) && L.total <= VA_NOALLOC_SCRATCH_BYTES;
    bool mma_possible = false;
    if (mma_fits_smem) {
        geometry(true, L);
        const int cap = max_len < va::kMmaMaxItemTokens ? max_len : va::kMmaMaxItemTokens;
        mma_possible = layout_for(seq_lens_host, B, Hkv, D, cap, L) && L.total <= VA_NOALLOC_SCRATCH_BYTES;
    }
    if (!warp_possible && !mma_possible) return VA_ERR_SCRATCH_TOO_SMALL;
    const bool mma = mma_possible && !(va::auto_path(R) == VA_PATH_WARP && warp_possible);
    if (!va::aligned_for(mma ? VA_PATH_MMA : VA_PATH_WARP, kv_dtype, q, k_pages, v_pages, k_scale, v_scale,
                         block_table, seq_lens, out, lse))
        return VA_ERR_INVALID_ARGUMENT;

    void *scratch = nullptr;
    int num_sms = 0;
    int rc = device_setup(&scratch, &num_sms);
    if (rc != VA_OK) return rc;
    geometry(mma, L);
    const int cap = mma ? (max_len < va::kMmaMaxItemTokens ? max_len : va::kMmaMaxItemTokens) : max_len;
    const long long slots = (long long)(mma ? 1 : va::warp_ctas_per_sm(kv_dtype, L.rows_per_group)) * num_sms;
    long long c = (total_len * Hkv * L.num_row_groups + slots - 1) / slots;
    c = (c + L.tile - 1) / L.tile * L.tile;
    if (c < 4 * L.tile) c = 4 * L.tile;
    bool fits = false;
    for (;;) {
        const int split = c > cap ? cap : (int)c;
        if (layout_for(seq_lens_host, B, Hkv, D, split, L) && L.total <= VA_NOALLOC_SCRATCH_BYTES) {
            fits = true;
            break;
        }
        if (split >= cap) break;  // as coarse as this kernel allows (checked above: not reached)
        c *= 2;
    }
    if (!fits) return VA_ERR_SCRATCH_TOO_SMALL;

    char *base = static_cast<char *>(scratch);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    std::lock_guard<std::mutex> lk(g_host_mu);
    int ni = 0, ng = 0, part = 0;
    for (int b = 0; b < B; ++b) {
        const int len = seq_lens_host[b];
        const int n = (len + L.split - 1) / L.split;
        for (int kvh = 0; kvh < Hkv; ++kvh)
            for (int rg = 0; rg < L.num_row_groups; ++rg) {
                const int first = n > 1 ? part : -1;
                if (n > 1) {
                    g_host_groups[ng++] = va::Group{b, kvh, rg, part, n, 0, 0, 0};
                    part += n;
                }
                for (int i = 0; i < n; ++i) {
                    const int k1 = (i + 1) * L.split < len ? (i + 1) * L.split : len;
                    g_host_items[ni++] = va::Item{b, kvh, rg, i * L.split, k1, len,
                                                  n > 1 ? first + i : -1, 0};
                }
            }
    }
    // Pageable sources: each copy has read the host buffer when it returns.
    cudaError_t e = cudaMemsetAsync(base, 0, kFlagsBytes, s);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(base + L.off_items, g_host_items, sizeof(va::Item) * ni, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess && ng > 0)
        e = cudaMemcpyAsync(base + L.off_groups, g_host_groups, sizeof(va::Group) * ng, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return cuda_fail(e);

    va::PartialParams pp{};
    pp.q = static_cast<const uint16_t *>(q);
    pp.k_pages = k_pages;
    pp.v_pages = v_pages;
    pp.k_scale = k_scale;
    pp.v_scale = v_scale;
    pp.block_table = block_table;
    pp.seq_lens = seq_lens;
    pp.out = static_cast<uint16_t *>(out);
    pp.lse = lse;
    pp.items = reinterpret_cast<const va::Item *>(base + L.off_items);
    pp.o_part = reinterpret_cast<float *>(base + L.off_o);
    pp.lse_part = reinterpret_cast<float *>(base + L.off_lse);
    pp.flags = reinterpret_cast<int *>(base);
    pp.bt_stride = bt_stride;
    pp.T = T;
    pp.Hq = Hq;
    pp.Hkv = Hkv;
    pp.G = G;
    pp.R = R;
    pp.rows_per_group = L.rows_per_group;
    pp.num_pages = num_pages;  // 0: block-table entries unchecked
    pp.num_parts = L.num_parts;
    pp.sm_scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)D));
    e = mma ? va::launch_mma_partial(pp, D, kv_dtype, ni, s) : va::launch_warp_partial(pp, D, kv_dtype, ni, s);
    if (e != cudaSuccess) return cuda_fail(e);
    if (ng > 0) {
        va::CombineParams cp{};
        cp.groups = reinterpret_cast<const va::Group *>(base + L.off_groups);
        cp.o_part = pp.o_part;
        cp.lse_part = pp.lse_part;
        cp.out = pp.out;
        cp.lse = lse;
        cp.T = T;
        cp.Hq = Hq;
        cp.G = G;
        cp.R = R;
        cp.rows_per_group = L.rows_per_group;
        cp.D = D;
        e = va::launch_combine(cp, ng, L.max_splits, s);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    return VA_OK;
}

extern "C" int verify_attn_noalloc_flags(int clear, int *flags, void *stream) {
    if (!flags) return VA_ERR_INVALID_ARGUMENT;
    void *scratch = nullptr;
    int num_sms = 0;
    int rc = device_setup(&scratch, &num_sms);
    if (rc != VA_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int host = 0;
    cudaError_t e = cudaMemcpyAsync(&host, scratch, sizeof(int), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e == cudaSuccess && clear) e = cudaMemsetAsync(scratch, 0, sizeof(int), s);
    if (e != cudaSuccess) return cuda_fail(e);
    *flags = host;
    return VA_OK;
}
