/*
 * verify_attn.h -- C ABI of the GB300 (sm_103a) verify-attention library.
 *
 * The operation.  Speculative decoding drafts a short block of T tokens and
 * checks them with one forward pass of the target model ("I pushed
 * Qwen3.8-27B to 124 tps on a single request on a RTX 3090", bullets "MTP-4
 * drafts" -> T = 5 and "Split-KV attention kernel for the verify step";
 * "I pushed Qwen3.8-27B to 381 tps for a single request on a RTX 3090",
 * "Longer verify blocks" -> T = 16).  In every attention layer of that pass,
 * the T verify queries attend causally to a long paged KV cache.  With G =
 * num_q_heads / num_kv_heads query heads per kv head, the G*T query rows of
 * one kv head share every key, so the library packs them into one tile and
 * reads each KV byte once per kv head.  The cache length is split across the
 * GPU's SMs ("split-KV") and the per-split partial results are merged by
 * log-sum-exp, so that a handful of queries still fill the chip (the same
 * bullet: FlashAttention-2 split KV only for one query and left most SMs
 * idle).  The split geometry is chosen from the live context lengths only,
 * never from a declared maximum ("Four Tesla V100s from 2017 matched my RTX
 * 5090 on single-request Qwen 3.8 decode", sections "This is a server, not a
 * GEMM screenshot" and "What about long context?": a declared max context
 * that leaked into the partition geometry taxed short requests).
 *
 * Definition (exact up to rounding), for sequence b with L_b cached tokens
 * (L_b includes the T verify tokens), verify token t, query head h and kv
 * head g = h / G:
 *     Khat[j] = decode(k_pages[block_table[b][j/16], j%16, g, :]) * k_scale[...]
 *     s_j     = (1/sqrt(head_dim)) * <q[b,t,h,:], Khat[j]>,  j <= L_b - T + t
 *     lse     = ln sum_j exp(s_j)
 *     out     = sum_j exp(s_j - lse) * Vhat[j]
 * bf16 caches use scale 1 (scale pointers may be NULL).
 *
 * Memory layouts (row-major, contiguous, all on the device unless noted):
 *     q            bf16  [B, T, Hq, D]
 *     k_pages      [num_pages, 16, Hkv, D] of bf16 / fp8-e4m3 / int8, or
 *                  [num_pages, 16, Hkv, D * bits / 8] bytes for the packed
 *                  4-bit / 2-bit caches: code d of a row is the two's-
 *                  complement field at bit (d * bits) % 8 of byte
 *                  d * bits / 8 (the first element in the low bits)
 *     v_pages      same layout as k_pages
 *     k_scale      fp32  [num_pages, 16, Hkv]   (one scale per token, kv head)
 *     v_scale      fp32  [num_pages, 16, Hkv]
 *     block_table  int32 [B, block_table_stride]  physical page of each
 *                  16-token logical block; stride defaults to
 *                  max_b ceil(L_b / 16)
 *     seq_lens     int32 [B]   same values as given to the planner
 *     out          bf16  [B, T, Hq, D]
 *     lse          fp32  [B, T, Hq]   natural-log log-sum-exp of the scaled
 *                  scores (may be NULL when not wanted)
 * The 4-bit and 2-bit caches follow the "KVarN 4/2-bit KV cache" bullet of
 * "I pushed Qwen3.8-27B to 381 tps for a single request on a RTX 3090", which
 * names the bit widths but not the format; the library takes the int8 rule
 * with fewer bits (symmetric absmax scale per token and kv head, codes
 * clamped to +-7 / +-1, decode = code * scale), so every cached format shares
 * one definition of decode().
 * Alignment: k_pages and v_pages start on a 16-byte boundary; on the tensor-
 * core path (the default) so do q, out and the scales; every other pointer
 * is aligned to its element type.  A call that breaks this returns
 * VA_ERR_INVALID_ARGUMENT before anything is launched.
 * Row r of a kv head's packed tile is verify token t = r / G, query head
 * h = g*G + r % G.
 *
 * Ownership.  The caller owns every tensor and the stream.  A plan owns its
 * device work list and split-partial workspace and frees them in
 * verify_attn_plan_destroy.  Calls on one plan share that workspace, so they
 * must be ordered on one stream (or otherwise serialised).
 *
 * Errors.  Every int-returning call returns VA_OK (0) or a negative va_status.
 * Nothing throws across the ABI and nothing traps on the device.  Launches
 * are asynchronous: a VA_OK from verify_attn means the work was enqueued.
 * When the plan knows the page-pool size (va_plan_options.num_pages > 0) the
 * kernels check every block-table entry; a bad entry is skipped (its keys
 * read as absent) and recorded in a device flag word that
 * verify_attn_plan_device_flags returns.  A device seq_lens value that
 * differs from the planned one is recorded the same way.
 */
#ifndef VERIFY_ATTN_H
#define VERIFY_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Tokens per KV page (vLLM's default block size, kept for attention layers
 * by "I pushed Qwen3.8-27B to 381 tps ...", "DFlash2 past 64k"). */
#define VA_PAGE_SIZE 16

typedef struct va_plan va_plan;

typedef enum {
    VA_BF16 = 0,     /* 2-byte bfloat16 cache, no scales */
    VA_FP8_E4M3 = 1, /* OCP fp8 e4m3, fp32 scale per (token, kv head) */
    VA_INT8 = 2,     /* int8, fp32 scale per (token, kv head) */
    VA_INT4 = 3,     /* 4-bit two's complement, two per byte, fp32 scale per (token, kv head) */
    VA_INT2 = 4      /* 2-bit two's complement, four per byte, fp32 scale per (token, kv head) */
} va_kv_dtype;

typedef enum {
    VA_OK = 0,
    VA_ERR_INVALID_ARGUMENT = -1, /* null or misaligned pointer, T < 1, Hq % Hkv != 0, L_b < T ... */
    VA_ERR_UNSUPPORTED = -2,      /* head_dim not in {64, 128, 256}, unknown dtype */
    VA_ERR_PLAN_MISMATCH = -3,    /* call arguments disagree with the plan */
    VA_ERR_NO_PLAN = -4,          /* verify_attn with no current plan on this thread */
    VA_ERR_CUDA = -5,             /* a CUDA runtime call or launch failed */
    VA_ERR_OUT_OF_MEMORY = -6,    /* workspace allocation failed */
    VA_ERR_NO_DEVICE = -7,        /* no usable CUDA device */
    VA_ERR_SCRATCH_TOO_SMALL = -8 /* verify_attn_noalloc: the work list alone does not
                                     fit in VA_NOALLOC_SCRATCH_BYTES */
} va_status;

/* Which partial-attention kernel a plan uses. */
typedef enum {
    VA_PATH_AUTO = 0,  /* the CUDA-core kernel for 1 or 2 packed rows per kv head,
                          tensor cores from 3 (the measured crossover) */
    VA_PATH_WARP = 1,  /* CUDA-core kernel: warp-shuffle reductions, any row count
                          (4 rows per work item; more rows re-read the cache) */
    VA_PATH_MMA = 2    /* tcgen05 tensor-core kernel (TMEM accumulators) */
} va_path;

/* Optional planner settings; zero-initialise for defaults. */
typedef struct {
    int block_table_stride; /* entries per block_table row; 0 = max_b ceil(L_b/16) */
    int tokens_per_split;   /* force the split length (rounded up to the kernel's
                               key tile); 0 = chosen by the planner */
    int path;               /* va_path */
    int num_pages;          /* page-pool size for device bound checks; 0 = no checks */
} va_plan_options;

/* Read-only summary of a plan (host data). */
typedef struct {
    int num_seqs, T, num_q_heads, num_kv_heads, head_dim, kv_dtype;
    int path;               /* the va_path actually used */
    int rows_per_group;     /* packed rows per work item (<= G*T) */
    int num_row_groups;     /* ceil(G*T / rows_per_group) */
    int tokens_per_split;   /* split length chosen */
    int num_items;          /* work items (CTAs of the partial kernel) */
    int num_split_groups;   /* (seq, kv head, row group) triples merged by the combine */
    int max_splits;         /* largest split count of any sequence */
    int num_sms;            /* SM count the plan was sized for */
    long long workspace_bytes;
} va_plan_info;

/* Build a plan for one batch shape.  Host only: reads seq_lens_host
 * (length num_seqs), chooses the split geometry from the live lengths and
 * num_sms (0 = query the current device), uploads the work list and
 * allocates the partial workspace on the current device.  On success
 * *out_plan owns that memory and becomes the calling thread's current plan
 * (used by verify_attn). */
int verify_attn_plan(const int32_t *seq_lens_host, int num_seqs, int T,
                     int num_q_heads, int num_kv_heads, int head_dim,
                     va_kv_dtype kv_dtype, int num_sms, va_plan **out_plan);

/* Same, with options (opts may be NULL). */
int verify_attn_plan_ex(const int32_t *seq_lens_host, int num_seqs, int T,
                        int num_q_heads, int num_kv_heads, int head_dim,
                        va_kv_dtype kv_dtype, int num_sms,
                        const va_plan_options *opts, va_plan **out_plan);

/* Verify attention with the calling thread's current plan (the one most
 * recently built on this thread and not yet destroyed).  stream is a
 * cudaStream_t (NULL = legacy default stream).  Asynchronous. */
int verify_attn(const void *q, const void *k_pages, const void *v_pages,
                const float *k_scale, const float *v_scale,
                const int32_t *block_table, const int32_t *seq_lens, int T,
                void *out, float *lse, void *stream);

/* Verify attention with an explicit plan (preferred form). */
int verify_attn_with_plan(const va_plan *plan, const void *q,
                          const void *k_pages, const void *v_pages,
                          const float *k_scale, const float *v_scale,
                          const int32_t *block_table, const int32_t *seq_lens,
                          int T, void *out, float *lse, void *stream);

/* Free a plan's device memory (NULL is a no-op).  Clears the thread's
 * current plan if it was this one.  The caller must make sure no call that
 * uses the plan is still running on the device. */
void verify_attn_plan_destroy(va_plan *plan);

/* Static English text for a va_status code. */
const char *verify_attn_status_string(int status);

/* Copy a plan's summary into *info (host only). */
int verify_attn_plan_get_info(const va_plan *plan, va_plan_info *info);

/* Pure host planning (no CUDA call, usable without a GPU): fills *info and,
 * when items != NULL, up to max_items work items as 5 ints each
 * (seq, kv_head, row_group, key_begin, key_end), in launch order. */
int verify_attn_plan_describe(const int32_t *seq_lens_host, int num_seqs, int T,
                              int num_q_heads, int num_kv_heads, int head_dim,
                              va_kv_dtype kv_dtype, int num_sms,
                              const va_plan_options *opts, va_plan_info *info,
                              int32_t *items, int max_items);

/* Host-side check of a batch's paging inputs before they go to the device
 * (no CUDA call, usable without a GPU): every sequence length satisfies
 * T <= seq_lens[b] <= 16 * block_table_stride, and every block-table entry
 * that a sequence uses (entries 0 .. ceil(L_b / 16) - 1 of row b) lies in
 * [0, num_pages).  Layouts as for verify_attn, both arrays in host memory.
 * Returns VA_OK, or VA_ERR_INVALID_ARGUMENT for null pointers, non-positive
 * sizes or the first violation found; *bad_seq and *bad_block (either may be
 * NULL) then name it: the sequence, and the block index within its row (-1
 * when the length itself is at fault); both are -1 on success.  The device
 * kernels make the same page check themselves when a plan knows num_pages;
 * this call lets a caller reject a bad batch before launching anything. */
int verify_attn_validate_host(const int32_t *seq_lens_host, int num_seqs, int T,
                              const int32_t *block_table_host, int block_table_stride,
                              int num_pages, int *bad_seq, int *bad_block);

/* Read (and if clear != 0, reset) the plan's device flag word:
 *   bit 0 (1) = a block-table entry outside [0, num_pages) was skipped;
 *   bit 1 (2) = a device seq_lens value differed from the planned one;
 *   bit 2 (4) = a wait inside the tensor-core kernel's pipeline gave up after
 *               its time limit (2 s); the CTA stopped early and its rows of
 *               out / lse are not valid.  It means a hardware or scheduling
 *               fault, never a property of the inputs.
 * Synchronises the stream. */
int verify_attn_plan_device_flags(const va_plan *plan, int clear, int *flags,
                                  void *stream);

/* Measurement hook.  When set (both non-NULL), every later call with this
 * plan records ev_before just before its partial-attention kernel and
 * ev_after just after it, on the call's stream, so that a caller can time
 * the dominant kernel alone (cudaEventElapsedTime).  The events are
 * cudaEvent_t handles owned by the caller; pass NULL, NULL to stop.  Works
 * under CUDA-graph capture (the records become graph nodes). */
int verify_attn_plan_set_events(va_plan *plan, void *ev_before, void *ev_after);

/* The cudaError_t value of the most recent CUDA call made by this library on
 * the calling thread that failed (0 if none): the detail behind a
 * VA_ERR_CUDA status.  verify_attn_last_cuda_error_string gives its text. */
int verify_attn_last_cuda_error(void);
const char *verify_attn_last_cuda_error_string(void);

/* Size of the library's built-in scratch for verify_attn_noalloc: a
 * file-scope device array that every GPU which loads the library holds until
 * the process exits. */
#define VA_NOALLOC_SCRATCH_BYTES (32u << 20)

/* Verify attention without any memory allocation, for callers that cannot
 * call cudaMalloc: code running where the allocator is off limits (inside a
 * custom memory pool's accounting, a real-time or signal-safe path, or an
 * embedding runtime that owns all device memory), or that must not grow the
 * device footprint after start-up.  (The method's sources describe no such
 * entry: it exists for deployment.)
 *
 * It plans from seq_lens_host on every call (host work only, no heap) and
 * keeps the work list and the split partials in a static device array of
 * VA_NOALLOC_SCRATCH_BYTES instead of a plan's workspace.  The caller passes
 * every input and output exactly as for verify_attn (same layouts), plus the
 * block-table row stride (0 = max_b ceil(L_b / 16)) and the page-pool size
 * num_pages (> 0: every block-table entry is checked against [0, num_pages),
 * a bad one is skipped and flagged as with a plan; 0: unchecked).  When the
 * partials of the default split do not fit, the split is made coarser until
 * they do; a problem whose work list alone does not fit returns
 * VA_ERR_SCRATCH_TOO_SMALL before anything touches the device.  Nothing is
 * allocated: no cudaMalloc, no cudaFree, no allocating library call.
 *
 * It runs the partial kernel a plan picks with a one-wave split, made
 * coarser while the partials do not fit; only a problem whose tensor-core
 * partials cannot fit at any split of up to 16384 keys runs the CUDA-core
 * kernel instead (unsplit if need be), which is several times slower at long
 * contexts with many packed rows.  Pointer alignment is checked as for
 * verify_attn_with_plan.
 *
 * The first call on a device looks up the array's device address there
 * (cudaGetSymbolAddress, with that device current).  All calls share the one
 * array, and each call overwrites what the previous one left there (its flag
 * word is cleared at the start of every call): calls that overlap on the GPU
 * race, so order them on one stream.  The work list is copied from static,
 * pageable host buffers with cudaMemcpyAsync on every call.  Asynchronous
 * like verify_attn. */
int verify_attn_noalloc(const int32_t *seq_lens_host, int num_seqs, int T,
                        int num_q_heads, int num_kv_heads, int head_dim,
                        va_kv_dtype kv_dtype, const void *q,
                        const void *k_pages, const void *v_pages,
                        const float *k_scale, const float *v_scale,
                        const int32_t *block_table, int block_table_stride,
                        int num_pages, const int32_t *seq_lens, void *out,
                        float *lse, void *stream);

/* The flag word that the most recent verify_attn_noalloc call on the current
 * device left in the static scratch (same bits as
 * verify_attn_plan_device_flags); clear != 0 resets it.  Synchronises the
 * stream. */
int verify_attn_noalloc_flags(int clear, int *flags, void *stream);

/* KV append with quantise-on-write: the step just before verify attention.
 * The verify forward computes K and V for its T tokens and stores them in the
 * paged cache before attending ("I pushed Qwen3.8-27B to 381 tps for a single
 * request on a RTX 3090", "DFlash2 past 64k": an int8 cache in 16-token
 * pages; "I pushed Qwen3.8-27B to 124 tps on a single request on a RTX
 * 3090", "What we had": an fp8 cache).  For sequence b (L_b = seq_lens[b]
 * includes the T new tokens), verify token t and kv head g:
 *     pos  = L_b - T + t,  page = block_table[b][pos / 16],  slot = pos % 16
 *     x    = k_new[b, t, g, :]                (bf16, exact in fp32)
 *     a    = max_d |x_d|
 *     s    = a / qmax in fp32, qmax = 448 (e4m3), 127 (int8), 7 (int4) or
 *            1 (int2); s = 1 if a = 0
 *     y_d  = x_d / s in fp32 (correctly rounded)
 *     e4m3: byte_d = round-to-nearest-even e4m3 of clamp(y_d, -448, 448)
 *     int8: byte_d = clamp(round-half-even(y_d), -127, 127)
 *     int4 / int2: code_d = clamp(round-half-even(y_d), -qmax, qmax), packed
 *           as the cache layout above states
 *     k_pages[page, slot, g, :] = bytes,  k_scale[page, slot, g] = s
 * and the same for v.  A bf16 cache receives the bf16 bits unchanged (the
 * scale pointers are ignored and may be NULL).  This is the per-(token, kv
 * head) absmax quantisation the verify inputs are built with, so appending
 * and attending agree on the cache format.
 *
 * Layouts: k_new, v_new bf16 [num_seqs, T, Hkv, D] on the device; the cache,
 * block table (row stride block_table_stride >= 1) and device seq_lens as for
 * verify_attn.  head_dim in {64, 128, 256}.  Checks: rows whose position is
 * negative (seq_lens[b] < T) or whose page is outside [0, num_pages) (when
 * num_pages > 0) are skipped and set bit 0 of *flags (a device int, may be
 * NULL; the library only ORs into it).  Returns VA_OK when enqueued on
 * stream, VA_ERR_INVALID_ARGUMENT for null or non-positive arguments,
 * VA_ERR_UNSUPPORTED for another head_dim or dtype, VA_ERR_CUDA if the launch
 * fails.  Rows of one call write disjoint cache slots as long as the block
 * table does not map two of them to the same page and slot. */
int verify_attn_kv_append(const void *k_new, const void *v_new, int num_seqs, int T,
                          int num_kv_heads, int head_dim, va_kv_dtype kv_dtype,
                          void *k_pages, void *v_pages, float *k_scale, float *v_scale,
                          const int32_t *block_table, int block_table_stride,
                          const int32_t *seq_lens, int num_pages, int *flags, void *stream);

/* Lookup-augmented drafting: propose draft tokens by finding the most recent
 * earlier occurrence of the request's last generated tokens in its own token
 * history and copying what followed ("I pushed Qwen3.8-27B to 381 tps for a
 * single request on a RTX 3090", "Lookup-augmented drafting": the last 6-12
 * tokens are looked up in the whole history, far beyond a block drafter's
 * window).  For sequence b with history x[0 .. L-1] (L = lens[b]):
 *     l(e)  = the largest l <= max_match with x[e - i] == x[L - 1 - i] for all
 *             i < l (and e - i >= 0), for every end position e <= L - 2
 *             (so that at least one token follows the occurrence);
 *     best  = the e with the largest min(l(e), max_match) among those with
 *             l(e) >= min_match, the largest e (the most recent) on a tie;
 *     draft = x[e + 1 .. min(e + 1 + num_draft, L) - 1]
 * draft_len[b] = its length (0 when no e qualifies), draft slots past it are
 * -1, match_end[b] = e or -1 (may be NULL), match_len[b] = min(l(e),
 * max_match) or 0 (may be NULL).  Integer work: the result is exact.
 *
 * Layouts (device): tokens int32 [num_seqs, token_stride]; lens int32
 * [num_seqs] (0 <= lens[b] <= token_stride); draft int32 [num_seqs,
 * num_draft]; draft_len, match_end, match_len int32 [num_seqs].  Limits:
 * 1 <= min_match <= max_match <= 32, 1 <= num_draft <= 256.  Returns VA_OK
 * when enqueued, VA_ERR_INVALID_ARGUMENT otherwise, VA_ERR_CUDA if the launch
 * fails.  One thread-block cluster scans each sequence: one CTA per 4,096
 * tokens of token_stride, at most 16 where the device can place a cluster of
 * that (non-portable) size and 8 otherwise, the CTAs' best matches combined
 * through distributed shared memory. */
int verify_attn_lookup_draft(const int32_t *tokens, int token_stride, const int32_t *lens,
                             int num_seqs, int min_match, int max_match, int num_draft,
                             int32_t *draft, int32_t *draft_len, int32_t *match_end,
                             int32_t *match_len, void *stream);

/* Speculative acceptance after the verify pass (the rejection sampler).
 * "I pushed Qwen3.8-27B to 124 tps ...": speculative decoding is exact by
 * construction (the sampled distribution is the target's); "I pushed
 * Qwen3.8-27B to 381 tps ...", "Lookup-augmented drafting": greedy never reads
 * the draft distribution, and sampled positions of a lookup draft get a
 * point-mass proposal q, which is a legal proposal for the rejection sampler;
 * "DFlash2 drafting": a model drafter's proposal is softmax of its raw logits
 * with the temperature applied once.
 *
 * For sequence b with draft d[0..T-1], target logits z[t] (t = 0..T, z[T] is
 * the position after the last draft) and temperature tau = temperature[b]:
 *   tau <= 0 (greedy): y_t = argmax_i z[t][i] (smallest i on ties); accept
 *     d[t] while d[t] == y_t; the first mismatch emits y_t, otherwise the
 *     bonus y_T is emitted.
 *   tau > 0: p_t = softmax(z[t] / tau); q_t = the one-hot of d[t] when
 *     draft_logits is NULL, else softmax(draft_logits[t] / tau).  Draft t is
 *     accepted iff u_t * q_t(d[t]) < p_t(d[t]), u_t = U(b, t, 0, 0).  At the
 *     first rejection the token emitted is argmax_i [ln r_i + G_i] over
 *     r_i = max(0, p_t(i) - q_t(i)) > 0 (the residual distribution sampled by
 *     an exponential race); if every draft is accepted the bonus token is
 *     argmax_i [z[T][i] / tau + G_i] (a sample of p_T).  G_i = -ln(-ln
 *     U(b, t, i, 1)) are Gumbel variates of the emitting position t.
 *   U(b, t, i, k) = (floor(w / 2^8) + 0.5) / 2^24 with w word number
 *     (i mod 4) of Philox4x32-10 (Salmon et al., SC'11) on counter
 *     (floor(i / 4), t, b, k) and key (seed low word, seed high word):
 *     uniform in (0, 1), reproducible, one Philox call per four entries.
 * Outputs: out_tokens[b, 0 .. n-1] = d[0 .. n-1], out_tokens[b, n] = the
 * emitted token, -1 after it; num_accepted[b] = n (0 .. T).
 * Layouts (device): target_logits fp32 [num_seqs, T + 1, vocab];
 * draft_logits fp32 [num_seqs, T, vocab] or NULL; draft_tokens int32
 * [num_seqs, T]; temperature fp32 [num_seqs]; out_tokens int32 [num_seqs,
 * T + 1]; num_accepted int32 [num_seqs]; workspace: at least
 * verify_attn_accept_workspace_bytes(num_seqs, T) bytes, 16-byte aligned,
 * owned by the caller; its contents need no initialisation, and calls that
 * share one workspace must be ordered on one stream.  The decisions are taken in binary32 (the scores,
 * exponentials and logarithms of the CUDA math library; u_t is U rounded toward zero, so below 1,
 * and each Gumbel takes -ln U to a few ulps from the exact U, whose nearest binary32 value can be
 * 1 or lose the low bit that decides -ln U near 1; the race ranks scores in units of ln 2, with
 * the hardware base-2 logarithm (absolute error about 1e-6) for ln(-ln U) and ln r), so a CPU restatement
 * in another precision agrees except where two scores, or u and p/q, are
 * within a few ulps.  Returns VA_OK when enqueued, VA_ERR_INVALID_ARGUMENT
 * for bad arguments (T >= 1, vocab >= 1, draft tokens outside [0, vocab) are
 * rejected as drafts), VA_ERR_CUDA if a launch fails. */
size_t verify_attn_accept_workspace_bytes(int num_seqs, int T);
int verify_attn_accept(const float *target_logits, const float *draft_logits,
                       const int32_t *draft_tokens, const float *temperature, int num_seqs,
                       int T, int vocab, uint64_t seed, void *workspace, int32_t *out_tokens,
                       int32_t *num_accepted, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* VERIFY_ATTN_H */
