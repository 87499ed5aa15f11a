"""Pins of the lookup-drafting oracle (CPU): against an independent search
with Python's bytes.rfind (a library routine) over many random histories,
planted copies with a known answer, and the edge cases the definition fixes."""
import numpy as np
import pytest

import oracle
from speculative_decoding_verify_causal_gb300 import workloads as wl


def rfind_reference(x, min_match, max_match, num_draft):
    """Longest n first; the most recent occurrence of the last n tokens that
    ends at or before L - 2, found with bytes.rfind on a 4-byte encoding."""
    L = len(x)
    enc = np.asarray(x, ">i4").tobytes()
    for n in range(max_match, min_match - 1, -1):
        if n > L:
            continue
        sub = enc[(L - n) * 4:]
        end = (L - 1) * 4  # the occurrence must end at token L - 2 or earlier
        while True:
            i = enc.rfind(sub, 0, end)
            if i < 0:
                break
            if i % 4 == 0:
                e = i // 4 + n - 1
                length = min(num_draft, L - 1 - e)
                draft = [int(v) for v in x[e + 1:e + 1 + length]] + [-1] * (num_draft - length)
                return draft, length, e, n
            end = i + len(sub) - 1  # misaligned hit: search before it
    return [-1] * num_draft, 0, -1, 0


@pytest.mark.parametrize("vocab", [2, 3, 5, 50, 151_936])
def test_matches_bytes_rfind_on_random_histories(vocab):
    rng = np.random.default_rng(vocab)
    for trial in range(60):
        L = int(rng.integers(1, 400))
        x = wl.token_history(1000 * vocab + trial, L, vocab=vocab, copy_frac=0.4, seg_range=(3, 20))
        lo = int(rng.integers(1, 8))
        hi = int(rng.integers(lo, 20))
        k = int(rng.integers(1, 12))
        d, n, e, m = oracle.lookup_draft(x, lo, hi, k)
        rd, rn, re_, rm = rfind_reference(x, lo, hi, k)
        assert (list(d), n, e, m) == (rd, rn, re_, rm), (L, lo, hi, k)


def test_planted_copy_is_found():
    x = wl.token_history(5, 5000, copy_frac=0.0)
    x[-12:] = x[1000:1012]  # the last 12 tokens occurred earlier, ending at 1011
    d, n, e, m = oracle.lookup_draft(x, 6, 12, 8)
    assert (e, m, n) == (1011, 12, 8) and list(d) == list(x[1012:1020])


def test_most_recent_occurrence_wins_on_equal_length():
    x = wl.token_history(6, 3000, copy_frac=0.0)
    x[-12:] = x[500:512]
    x[2000:2012] = x[500:512]
    d, n, e, m = oracle.lookup_draft(x, 6, 12, 4)
    assert (e, m) == (2011, 12) and list(d) == list(x[2012:2016])


def test_longer_match_beats_more_recent_shorter_one():
    x = wl.token_history(7, 3000, copy_frac=0.0)
    x[-12:] = x[500:512]          # 12-token occurrence ending at 511
    x[2000:2006] = x[-6:]         # a more recent 6-token occurrence ending at 2005
    d, n, e, m = oracle.lookup_draft(x, 6, 12, 4)
    assert (e, m) == (511, 12)


def test_edges():
    assert oracle.lookup_draft(np.array([7], np.int32), 1, 4, 3)[1:] == (0, -1, 0)
    # periodic history: the overlapping occurrence one period back is the most recent
    x = np.array([1, 2, 3] * 10, np.int32)
    d, n, e, m = oracle.lookup_draft(x, 6, 12, 5)
    assert (e, m, n) == (26, 12, 3) and list(d) == [1, 2, 3, -1, -1]
    # draft truncated by the end of the history
    x = np.array([9, 9, 9, 9, 9, 9, 9, 4], np.int32)
    d, n, e, m = oracle.lookup_draft(x, 1, 3, 8)
    assert n == 0 or list(d[:n]) == list(x[e + 1:e + 1 + n])
