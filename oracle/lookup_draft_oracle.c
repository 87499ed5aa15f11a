/*
 * CPU oracle for lookup-augmented drafting.  TEST INFRASTRUCTURE ONLY (the
 * tests and the benchmark's CPU-baseline leg); it shares no code with the
 * CUDA library.
 *
 * What it computes ("I pushed Qwen3.8-27B to 381 tps for a single request on
 * a RTX 3090", "Lookup-augmented drafting": the request's own token history
 * is scanned for the most recent occurrence of the last 6-12 generated tokens
 * and what followed that occurrence is proposed as the draft), taken in the
 * plainest order: for n = max_match down to min_match, the latest end
 * position e <= L - 2 (a token must follow) with x[e - i] == x[L - 1 - i] for
 * all i < n; the first n that has one wins, and the draft is
 * x[e + 1 .. min(e + 1 + num_draft, L) - 1].
 */
#include <stdint.h>

/* Returns the draft length (0 = no match); *match_end / *match_len get e and
 * n (-1 and 0 without a match); draft gets num_draft entries, -1 past the
 * proposal. */
int oracle_lookup_draft(const int32_t *x, int L, int min_match, int max_match, int num_draft, int32_t *draft,
                        int32_t *match_end, int32_t *match_len)
{
    int best_e = -1, best_n = 0;
    for (int n = max_match; n >= min_match && best_e < 0; --n) {
        if (n > L)
            continue;
        for (int e = L - 2; e >= n - 1; --e) {
            int i = 0;
            while (i < n && x[e - i] == x[L - 1 - i])
                ++i;
            if (i == n) {
                best_e = e;
                best_n = n;
                break;
            }
        }
    }
    int len = 0;
    if (best_e >= 0) {
        len = L - 1 - best_e;
        if (len > num_draft)
            len = num_draft;
    }
    for (int t = 0; t < num_draft; ++t)
        draft[t] = t < len ? x[best_e + 1 + t] : -1;
    *match_end = best_e;
    *match_len = best_n;
    return len;
}
