// Host side of the library: the split planner, plan lifetime, argument
// validation and the two launches of one verify call.
//
// The planner sizes the split-KV geometry from the live sequence lengths and
// the SM count only.  The reason is the lesson of "Four Tesla V100s from 2017
// matched my RTX 5090 on single-request Qwen 3.8 decode" (sections "This is a
// server, not a GEMM screenshot" and "What about long context?"): a declared
// maximum context that leaked into the partition geometry made short requests
// slow.  The split itself is the method of "I pushed Qwen3.8-27B to 124 tps on
// a single request on a RTX 3090", bullet "Split-KV attention kernel for the
// verify step": cut the cache along its length so that a few verify queries
// still occupy every SM, then merge the partial softmaxes by log-sum-exp.
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <functional>
#include <new>
#include <queue>
#include <vector>

#include "va_internal.h"

struct va_plan {
    int num_seqs, T, Hq, Hkv, D, kv_dtype;
    int path, rows_per_group, num_row_groups, tile;
    int tokens_per_split, bt_stride, num_pages, num_sms;
    int num_items, num_parts, num_groups, max_splits;
    std::vector<int32_t> seq_lens;
    int device;
    void *dev_mem;  // one allocation: items | groups | flags | lse_part | o_part
    va::Item *items;
    va::Group *groups;
    int *flags;
    float *lse_part;
    float *o_part;
    long long workspace_bytes;
    cudaEvent_t ev_before, ev_after;  // optional measurement hook
};

namespace {

thread_local va_plan *t_current_plan = nullptr;
thread_local int t_last_cuda_error = 0;

struct Geometry {
    int path, rows_per_group, num_row_groups, tile, tokens_per_split, slots;
    int max_splits;
    std::vector<va::Item> items;
    std::vector<va::Group> groups;
    int num_parts;
};

int head_dim_ok(int D) { return D == 64 || D == 128 || D == 256; }

// Bits per cached element.
int kv_bits(int dtype) {
    return dtype == VA_BF16 ? 16 : dtype == VA_INT4 ? 4 : dtype == VA_INT2 ? 2 : 8;
}

// Splits of one sequence for a nominal split length c: equal parts rounded up
// to the key tile, so every split but the last is a whole number of tiles.
int split_length(int L, int c, int tile) {
    int n = (L + c - 1) / c;
    int base = (L + n - 1) / n;
    base = (base + tile - 1) / tile * tile;
    return base;
}

// Longest-processing-time makespan of `costs` on `slots` identical workers.
double lpt_makespan(std::vector<double> costs, int slots) {
    std::sort(costs.begin(), costs.end(), std::greater<double>());
    if ((int)costs.size() <= slots) return costs.empty() ? 0.0 : costs.front();
    std::priority_queue<double, std::vector<double>, std::greater<double>> load;
    for (int i = 0; i < slots; ++i) load.push(0.0);
    double worst = 0.0;
    for (double c : costs) {
        double l = load.top();
        load.pop();
        l += c;
        worst = std::max(worst, l);
        load.push(l);
    }
    return worst;
}

int validate(const int32_t *seq_lens, int B, int T, int Hq, int Hkv, int D, int dtype,
             const va_plan_options *opts) {
    if (!seq_lens || B < 1 || T < 1 || Hq < 1 || Hkv < 1) return VA_ERR_INVALID_ARGUMENT;
    if (Hq % Hkv != 0) return VA_ERR_INVALID_ARGUMENT;
    if (!head_dim_ok(D)) return VA_ERR_UNSUPPORTED;
    if (dtype < VA_BF16 || dtype > VA_INT2) return VA_ERR_UNSUPPORTED;
    int max_pages = 0;
    for (int b = 0; b < B; ++b) {
        if (seq_lens[b] < T) return VA_ERR_INVALID_ARGUMENT;
        max_pages = std::max(max_pages, (seq_lens[b] + VA_PAGE_SIZE - 1) / VA_PAGE_SIZE);
    }
    if (opts) {
        if (opts->block_table_stride < 0 || opts->tokens_per_split < 0 || opts->num_pages < 0)
            return VA_ERR_INVALID_ARGUMENT;
        if (opts->block_table_stride > 0 && opts->block_table_stride < max_pages)
            return VA_ERR_INVALID_ARGUMENT;
        if (opts->path < VA_PATH_AUTO || opts->path > VA_PATH_MMA) return VA_ERR_INVALID_ARGUMENT;
    }
    return VA_OK;
}

// The CUDA-core kernel for one or two packed rows per kv head (a T = 1 decode
// with one or two query heads per kv head, say), the tensor-core kernel from
// three rows on: the crossover measured on GB300 (va::auto_path).
int choose_path(int R, int Hkv, const va_plan_options *opts) {
    (void)Hkv;
    int want = opts ? opts->path : VA_PATH_AUTO;
    return want != VA_PATH_AUTO ? want : va::auto_path(R);
}

int plan_geometry(const int32_t *seq_lens, int B, int T, int Hq, int Hkv, int D, int dtype,
                  int num_sms, const va_plan_options *opts, Geometry &g) {
    const int G = Hq / Hkv;
    const int R = G * T;
    g.path = choose_path(R, Hkv, opts);
    if (g.path == VA_PATH_MMA && va::mma_smem_bytes(D, dtype, Hkv) > va::kMaxSmemPerBlock) {
        // the page scale blocks of a large kv-head count do not fit next to the tiles
        if (opts && opts->path == VA_PATH_MMA) return VA_ERR_UNSUPPORTED;
        g.path = VA_PATH_WARP;
    }
    const bool mma = g.path == VA_PATH_MMA;
    const int max_rows = mma ? va::kMmaRows : va::kWarpRows;
    g.tile = mma ? va::kMmaTile : va::kWarpTile;
    g.num_row_groups = (R + max_rows - 1) / max_rows;
    g.rows_per_group = (R + g.num_row_groups - 1) / g.num_row_groups;
    // the tcgen05 kernel holds a whole SM; the CUDA-core kernel's residency
    // depends on its variant
    g.slots = mma ? num_sms : num_sms * va::warp_ctas_per_sm(dtype, g.rows_per_group);

    int maxL = 0;
    double total = 0.0;
    for (int b = 0; b < B; ++b) {
        maxL = std::max(maxL, seq_lens[b]);
        total += seq_lens[b];
    }
    const int per_seq_items = Hkv * g.num_row_groups;
    // Cost model in key-token units: a fixed start-up cost per item (q load,
    // pipeline fill) and, for split sequences, the partial write + combine
    // read of rows x D fp32 relative to one token's KV bytes.
    const double token_bytes = 2.0 * D * kv_bits(dtype) / 8.0 + (dtype == VA_BF16 ? 0 : 8);
    const double c_item = mma ? 384.0 : 128.0;
    const double c_split = 2.0 * g.rows_per_group * (D + 1) * 4.0 / token_bytes;

    auto cost_of = [&](int c, std::vector<double> *costs) {
        if (costs) costs->clear();
        std::vector<double> tmp;
        std::vector<double> &v = costs ? *costs : tmp;
        for (int b = 0; b < B; ++b) {
            int L = seq_lens[b];
            int base = split_length(L, c, g.tile);
            int n = (L + base - 1) / base;
            for (int i = 0; i < n; ++i) {
                int len = std::min(base, L - i * base);
                double cst = c_item + len + (n > 1 ? c_split : 0.0);
                for (int k = 0; k < per_seq_items; ++k) v.push_back(cst);
            }
        }
        return lpt_makespan(v, g.slots);
    };

    // the tcgen05 kernel stages an item's page ids in shared memory
    const int cap = mma ? va::kMmaMaxItemTokens : (1 << 30);
    int chosen;
    if (opts && opts->tokens_per_split > 0) {
        chosen = (opts->tokens_per_split + g.tile - 1) / g.tile * g.tile;
        chosen = std::min(chosen, cap);
    } else {
        // Candidates: the one-wave length and a few multiples of the slot
        // count, plus "no split"; the smallest LPT makespan wins (ties go to
        // longer splits: fewer partials).
        std::vector<int> cand;
        const double units = total * per_seq_items;
        for (double waves : {0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, 8.0}) {
            double c = units / (g.slots * waves);  // key tokens per item for `waves` items per slot
            int ci = (int)std::ceil(c / g.tile) * g.tile;
            ci = std::max(ci, 4 * g.tile);
            cand.push_back(std::min(ci, cap));
        }
        cand.push_back(std::min(std::max(maxL, g.tile), cap));
        std::sort(cand.begin(), cand.end());
        cand.erase(std::unique(cand.begin(), cand.end()), cand.end());
        double best = 1e300;
        chosen = cand.back();
        for (int c : cand) {
            double m = cost_of(c, nullptr);
            if (m < best * (1.0 - 1e-9) || (m <= best * (1.0 + 1e-9) && c > chosen)) {
                best = std::min(best, m);
                chosen = c;
            }
        }
    }
    g.tokens_per_split = chosen;

    // Materialise items; order them longest first (the hardware hands out
    // CTAs in launch order, which then approximates LPT).
    struct Tmp {
        va::Item it;
        double cost;
    };
    std::vector<Tmp> tmp;
    g.groups.clear();
    g.max_splits = 1;
    int parts = 0;
    for (int b = 0; b < B; ++b) {
        int L = seq_lens[b];
        int base = split_length(L, chosen, g.tile);
        int n = (L + base - 1) / base;
        g.max_splits = std::max(g.max_splits, n);
        for (int kvh = 0; kvh < Hkv; ++kvh)
            for (int rg = 0; rg < g.num_row_groups; ++rg) {
                int first = -1;
                if (n > 1) {
                    first = parts;
                    parts += n;
                    g.groups.push_back({b, kvh, rg, first, n, 0, 0, 0});
                }
                for (int i = 0; i < n; ++i) {
                    va::Item it{b, kvh, rg, i * base, std::min(L, (i + 1) * base), L,
                                n > 1 ? first + i : -1, 0};
                    double cst = c_item + (it.k_end - it.k_begin) + (n > 1 ? c_split : 0.0);
                    tmp.push_back({it, cst});
                }
            }
    }
    std::stable_sort(tmp.begin(), tmp.end(), [](const Tmp &a, const Tmp &b) { return a.cost > b.cost; });
    g.items.clear();
    for (auto &t : tmp) g.items.push_back(t.it);
    g.num_parts = parts;
    return VA_OK;
}

int query_num_sms(int *num_sms, int *device) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return VA_ERR_NO_DEVICE;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) {
        cudaGetLastError();
        return VA_ERR_NO_DEVICE;
    }
    *num_sms = n;
    *device = dev;
    return VA_OK;
}

void fill_info(const va_plan &p, va_plan_info *info) {
    info->num_seqs = p.num_seqs;
    info->T = p.T;
    info->num_q_heads = p.Hq;
    info->num_kv_heads = p.Hkv;
    info->head_dim = p.D;
    info->kv_dtype = p.kv_dtype;
    info->path = p.path;
    info->rows_per_group = p.rows_per_group;
    info->num_row_groups = p.num_row_groups;
    info->tokens_per_split = p.tokens_per_split;
    info->num_items = p.num_items;
    info->num_split_groups = p.num_groups;
    info->max_splits = p.max_splits;
    info->num_sms = p.num_sms;
    info->workspace_bytes = p.workspace_bytes;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace

namespace va {
void note_cuda_error(cudaError_t e) {
    if (e != cudaSuccess) t_last_cuda_error = (int)e;
}

bool aligned_for(int path, int kv_dtype, const void *q, const void *k_pages, const void *v_pages,
                 const float *k_scale, const float *v_scale, const int32_t *block_table,
                 const int32_t *seq_lens, const void *out, const float *lse) {
    auto ok = [](const void *ptr, uintptr_t a) { return (reinterpret_cast<uintptr_t>(ptr) & (a - 1)) == 0; };
    const bool quant = kv_dtype != VA_BF16;
    // cache rows move in 16-byte units in both kernels (TMA boxes, or
    // 16 / 8 / 4-byte vector loads at 16-byte aligned row offsets)
    if (!ok(k_pages, 16) || !ok(v_pages, 16)) return false;
    if (!ok(q, 2) || !ok(out, 2) || !ok(block_table, 4) || !ok(seq_lens, 4) || (lse && !ok(lse, 4))) return false;
    if (quant && (!ok(k_scale, 4) || !ok(v_scale, 4))) return false;
    // the tensor-core kernel moves q, out and the scales in 16-byte units too
    if (path == VA_PATH_MMA && (!ok(q, 16) || !ok(out, 16) || (quant && (!ok(k_scale, 16) || !ok(v_scale, 16)))))
        return false;
    return true;
}
}  // namespace va

extern "C" {

int verify_attn_last_cuda_error(void) { return t_last_cuda_error; }

const char *verify_attn_last_cuda_error_string(void) {
    return cudaGetErrorString(static_cast<cudaError_t>(t_last_cuda_error));
}

int verify_attn_validate_host(const int32_t *seq_lens, int B, int T, const int32_t *block_table,
                              int bt_stride, int num_pages, int *bad_seq, int *bad_block) {
    if (bad_seq) *bad_seq = -1;
    if (bad_block) *bad_block = -1;
    if (!seq_lens || !block_table || B < 1 || T < 1 || bt_stride < 1 || num_pages < 1)
        return VA_ERR_INVALID_ARGUMENT;
    for (int b = 0; b < B; ++b) {
        const long long L = seq_lens[b];
        if (L < T || L > (long long)VA_PAGE_SIZE * bt_stride) {
            if (bad_seq) *bad_seq = b;
            return VA_ERR_INVALID_ARGUMENT;
        }
        const int used = (int)((L + VA_PAGE_SIZE - 1) / VA_PAGE_SIZE);
        const int32_t *row = block_table + (size_t)b * bt_stride;
        for (int i = 0; i < used; ++i) {
            if (row[i] < 0 || row[i] >= num_pages) {
                if (bad_seq) *bad_seq = b;
                if (bad_block) *bad_block = i;
                return VA_ERR_INVALID_ARGUMENT;
            }
        }
    }
    return VA_OK;
}

const char *verify_attn_status_string(int status) {
    switch (status) {
    case VA_OK: return "ok";
    case VA_ERR_INVALID_ARGUMENT: return "invalid argument";
    case VA_ERR_UNSUPPORTED: return "unsupported head_dim, dtype or path";
    case VA_ERR_PLAN_MISMATCH: return "call arguments do not match the plan";
    case VA_ERR_NO_PLAN: return "no current plan on this thread";
    case VA_ERR_CUDA: return "CUDA runtime error";
    case VA_ERR_OUT_OF_MEMORY: return "device workspace allocation failed";
    case VA_ERR_NO_DEVICE: return "no usable CUDA device";
    case VA_ERR_SCRATCH_TOO_SMALL:
        return "work list exceeds the static scratch of verify_attn_noalloc (VA_NOALLOC_SCRATCH_BYTES)";
    default: return "unknown status";
    }
}

int verify_attn_plan_describe(const int32_t *seq_lens, int B, int T, int Hq, int Hkv, int D,
                              va_kv_dtype kv_dtype, int num_sms, const va_plan_options *opts,
                              va_plan_info *info, int32_t *items, int max_items) {
    int rc = validate(seq_lens, B, T, Hq, Hkv, D, kv_dtype, opts);
    if (rc != VA_OK) return rc;
    if (num_sms < 1 || !info || (items && max_items < 0)) return VA_ERR_INVALID_ARGUMENT;
    Geometry g;
    rc = plan_geometry(seq_lens, B, T, Hq, Hkv, D, kv_dtype, num_sms, opts, g);
    if (rc != VA_OK) return rc;
    va_plan p{};
    p.num_seqs = B;
    p.T = T;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.D = D;
    p.kv_dtype = kv_dtype;
    p.path = g.path;
    p.rows_per_group = g.rows_per_group;
    p.num_row_groups = g.num_row_groups;
    p.tokens_per_split = g.tokens_per_split;
    p.num_items = (int)g.items.size();
    p.num_groups = (int)g.groups.size();
    p.max_splits = g.max_splits;
    p.num_sms = num_sms;
    p.workspace_bytes = (long long)g.num_parts * g.rows_per_group * (D + 1) * 4;
    fill_info(p, info);
    if (items) {
        int n = std::min(max_items, (int)g.items.size());
        for (int i = 0; i < n; ++i) {
            const va::Item &it = g.items[i];
            items[5 * i + 0] = it.b;
            items[5 * i + 1] = it.kvh;
            items[5 * i + 2] = it.rg;
            items[5 * i + 3] = it.k_begin;
            items[5 * i + 4] = it.k_end;
        }
    }
    return VA_OK;
}

int verify_attn_plan_ex(const int32_t *seq_lens, int B, int T, int Hq, int Hkv, int D,
                        va_kv_dtype kv_dtype, int num_sms, const va_plan_options *opts,
                        va_plan **out_plan) {
    if (!out_plan) return VA_ERR_INVALID_ARGUMENT;
    *out_plan = nullptr;
    int rc = validate(seq_lens, B, T, Hq, Hkv, D, kv_dtype, opts);
    if (rc != VA_OK) return rc;
    int device = 0, sms = 0;
    rc = query_num_sms(&sms, &device);
    if (rc != VA_OK) return rc;
    if (num_sms < 0) return VA_ERR_INVALID_ARGUMENT;
    if (num_sms == 0) num_sms = sms;
    Geometry g;
    rc = plan_geometry(seq_lens, B, T, Hq, Hkv, D, kv_dtype, num_sms, opts, g);
    if (rc != VA_OK) return rc;

    va_plan *p = new (std::nothrow) va_plan();
    if (!p) return VA_ERR_OUT_OF_MEMORY;
    p->num_seqs = B;
    p->T = T;
    p->Hq = Hq;
    p->Hkv = Hkv;
    p->D = D;
    p->kv_dtype = kv_dtype;
    p->path = g.path;
    p->rows_per_group = g.rows_per_group;
    p->num_row_groups = g.num_row_groups;
    p->tile = g.tile;
    p->tokens_per_split = g.tokens_per_split;
    int max_pages = 0;
    for (int b = 0; b < B; ++b) max_pages = std::max(max_pages, (seq_lens[b] + VA_PAGE_SIZE - 1) / VA_PAGE_SIZE);
    p->bt_stride = (opts && opts->block_table_stride > 0) ? opts->block_table_stride : max_pages;
    p->num_pages = opts ? opts->num_pages : 0;
    p->num_sms = num_sms;
    p->num_items = (int)g.items.size();
    p->num_parts = g.num_parts;
    p->num_groups = (int)g.groups.size();
    p->max_splits = g.max_splits;
    p->seq_lens.assign(seq_lens, seq_lens + B);
    p->device = device;

    size_t off_items = 0;
    size_t off_groups = align_up(off_items + sizeof(va::Item) * g.items.size(), 256);
    size_t off_flags = align_up(off_groups + sizeof(va::Group) * std::max<size_t>(1, g.groups.size()), 256);
    size_t off_lse = align_up(off_flags + 256, 256);
    size_t n_lse = (size_t)g.num_parts * g.rows_per_group;
    size_t off_o = align_up(off_lse + sizeof(float) * std::max<size_t>(1, n_lse), 256);
    size_t n_o = (size_t)g.num_parts * g.rows_per_group * D;
    size_t total = align_up(off_o + sizeof(float) * std::max<size_t>(1, n_o), 256);
    void *mem = nullptr;
    if (cudaMalloc(&mem, total) != cudaSuccess) {
        cudaGetLastError();
        delete p;
        return VA_ERR_OUT_OF_MEMORY;
    }
    char *base = static_cast<char *>(mem);
    p->dev_mem = mem;
    p->items = reinterpret_cast<va::Item *>(base + off_items);
    p->groups = reinterpret_cast<va::Group *>(base + off_groups);
    p->flags = reinterpret_cast<int *>(base + off_flags);
    p->lse_part = reinterpret_cast<float *>(base + off_lse);
    p->o_part = reinterpret_cast<float *>(base + off_o);
    p->workspace_bytes = (long long)total;
    bool ok = cudaMemcpy(p->items, g.items.data(), sizeof(va::Item) * g.items.size(),
                         cudaMemcpyHostToDevice) == cudaSuccess;
    if (ok && !g.groups.empty())
        ok = cudaMemcpy(p->groups, g.groups.data(), sizeof(va::Group) * g.groups.size(),
                        cudaMemcpyHostToDevice) == cudaSuccess;
    if (ok) ok = cudaMemset(p->flags, 0, 256) == cudaSuccess;
    if (!ok) {
        cudaGetLastError();
        cudaFree(mem);
        delete p;
        return VA_ERR_CUDA;
    }
    *out_plan = p;
    t_current_plan = p;
    return VA_OK;
}

int verify_attn_plan(const int32_t *seq_lens, int B, int T, int Hq, int Hkv, int D,
                     va_kv_dtype kv_dtype, int num_sms, va_plan **out_plan) {
    return verify_attn_plan_ex(seq_lens, B, T, Hq, Hkv, D, kv_dtype, num_sms, nullptr, out_plan);
}

void verify_attn_plan_destroy(va_plan *p) {
    if (!p) return;
    if (t_current_plan == p) t_current_plan = nullptr;
    if (p->dev_mem) cudaFree(p->dev_mem);
    delete p;
}

int verify_attn_plan_get_info(const va_plan *p, va_plan_info *info) {
    if (!p || !info) return VA_ERR_INVALID_ARGUMENT;
    fill_info(*p, info);
    return VA_OK;
}

int verify_attn_plan_device_flags(const va_plan *p, int clear, int *flags, void *stream) {
    if (!p || !flags) return VA_ERR_INVALID_ARGUMENT;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int host = 0;
    if (cudaMemcpyAsync(&host, p->flags, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess) {
        cudaGetLastError();
        return VA_ERR_CUDA;
    }
    if (clear && cudaMemsetAsync(p->flags, 0, sizeof(int), s) != cudaSuccess) {
        cudaGetLastError();
        return VA_ERR_CUDA;
    }
    *flags = host;
    return VA_OK;
}

int verify_attn_with_plan(const va_plan *p, const void *q, const void *k_pages,
                          const void *v_pages, const float *k_scale, const float *v_scale,
                          const int32_t *block_table, const int32_t *seq_lens, int T, void *out,
                          float *lse, void *stream) {
    if (!p) return VA_ERR_NO_PLAN;
    if (!q || !k_pages || !v_pages || !block_table || !seq_lens || !out)
        return VA_ERR_INVALID_ARGUMENT;
    if (p->kv_dtype != VA_BF16 && (!k_scale || !v_scale)) return VA_ERR_INVALID_ARGUMENT;
    if (T != p->T) return VA_ERR_PLAN_MISMATCH;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

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
    pp.items = p->items;
    pp.o_part = p->o_part;
    pp.lse_part = p->lse_part;
    pp.flags = p->flags;
    pp.bt_stride = p->bt_stride;
    pp.T = p->T;
    pp.Hq = p->Hq;
    pp.Hkv = p->Hkv;
    pp.G = p->Hq / p->Hkv;
    pp.R = pp.G * p->T;
    pp.rows_per_group = p->rows_per_group;
    pp.num_pages = p->num_pages;
    pp.num_parts = p->num_parts;
    pp.sm_scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)p->D));

    if (!va::aligned_for(p->path, p->kv_dtype, q, k_pages, v_pages, k_scale, v_scale, block_table, seq_lens,
                         out, lse))
        return VA_ERR_INVALID_ARGUMENT;
    if (p->ev_before && cudaEventRecordWithFlags(p->ev_before, s, cudaEventRecordExternal) != cudaSuccess)
        return VA_ERR_CUDA;
    cudaError_t e = p->path == VA_PATH_MMA
                        ? va::launch_mma_partial(pp, p->D, p->kv_dtype, p->num_items, s)
                        : va::launch_warp_partial(pp, p->D, p->kv_dtype, p->num_items, s);
    if (e != cudaSuccess) {
        va::note_cuda_error(e);
        cudaGetLastError();
        return VA_ERR_CUDA;
    }
    if (p->ev_after && cudaEventRecordWithFlags(p->ev_after, s, cudaEventRecordExternal) != cudaSuccess)
        return VA_ERR_CUDA;
    if (p->num_groups > 0) {
        va::CombineParams cp{};
        cp.groups = p->groups;
        cp.o_part = p->o_part;
        cp.lse_part = p->lse_part;
        cp.out = pp.out;
        cp.lse = lse;
        cp.T = p->T;
        cp.Hq = p->Hq;
        cp.G = pp.G;
        cp.R = pp.R;
        cp.rows_per_group = p->rows_per_group;
        cp.D = p->D;
        e = va::launch_combine(cp, p->num_groups, p->max_splits, s);
        if (e != cudaSuccess) {
            va::note_cuda_error(e);
            cudaGetLastError();
            return VA_ERR_CUDA;
        }
    }
    return VA_OK;
}

int verify_attn_plan_set_events(va_plan *p, void *ev_before, void *ev_after) {
    if (!p || (!ev_before) != (!ev_after)) return VA_ERR_INVALID_ARGUMENT;
    p->ev_before = static_cast<cudaEvent_t>(ev_before);
    p->ev_after = static_cast<cudaEvent_t>(ev_after);
    return VA_OK;
}

int verify_attn(const void *q, const void *k_pages, const void *v_pages, const float *k_scale,
                const float *v_scale, const int32_t *block_table, const int32_t *seq_lens, int T,
                void *out, float *lse, void *stream) {
    if (!t_current_plan) return VA_ERR_NO_PLAN;
    return verify_attn_with_plan(t_current_plan, q, k_pages, v_pages, k_scale, v_scale,
                                 block_table, seq_lens, T, out, lse, stream);
}

}  // extern "C"
