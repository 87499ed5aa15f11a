"""Pins of the acceptance-sampler oracle (CPU): Philox4x32-10 against the
published known-answer vectors, the greedy rule against its plain statement,
and the exactness theorem the pages rely on (the emitted tokens follow the
target distribution, whatever the proposal) checked statistically."""
import math

import numpy as np
import pytest

from oracle import sampler


def test_philox_known_answers():
    cases = [((0, 0, 0, 0), (0, 0), (0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8)),
             ((0xFFFFFFFF,) * 4, (0xFFFFFFFF,) * 2, (0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD)),
             ((0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344), (0xA4093822, 0x299F31D0),
              (0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1))]
    for ctr, key, want in cases:
        got = sampler.philox4x32_10(*ctr, *key)
        assert tuple(int(np.asarray(v)) for v in got) == want


def test_uniform_is_open_unit_interval_and_flat():
    u = sampler.uniform(123, 0, 0, np.arange(200000, dtype=np.uint64), 1)
    assert u.min() > 0 and u.max() < 1
    hist = np.histogram(u, bins=20, range=(0, 1))[0]
    assert np.all(np.abs(hist - 10000) < 600)


def test_uniform_words_of_one_counter_are_flat_and_uncorrelated():
    # four consecutive entries share a Philox counter, one word each: every
    # word position must be flat on its own, and neighbours (same counter or
    # across counters) uncorrelated -- a wrong word choice (say the first
    # word for all four) repeats values and fails both
    n = 400_000
    u = sampler.uniform(7, 3, 2, np.arange(n, dtype=np.uint64), 1)
    # 24-bit values: about n^2 / 2^25 repeats by chance (4,800 here)
    assert len(np.unique(u)) > n - 1.2 * n * n / 2 ** 25
    for r in range(4):
        hist = np.histogram(u[r::4], bins=10, range=(0, 1))[0]
        assert np.all(np.abs(hist - n / 40) < 0.06 * n / 40)
    for lag in (1, 2, 3, 4):
        c = np.corrcoef(u[:-lag], u[lag:])[0, 1]
        assert abs(c) < 0.01
    # entry 0 of every position is word 0 of counter (0, t, b, k)
    w0 = sampler.philox4x32_10(0, 2, 3, 1, 7, 0)[0]
    assert u[0] == ((int(w0) >> 8) + 0.5) / 2 ** 24


def test_greedy_prefix_rule():
    rng = np.random.default_rng(1)
    B, T, V = 50, 6, 9
    z = rng.standard_normal((B, T + 1, V))
    y = z.argmax(-1)
    d = y[:, :T].copy()
    cut = rng.integers(0, T + 1, B)
    for b in range(B):
        if cut[b] < T:
            d[b, cut[b]] = (y[b, cut[b]] + 1) % V
    out, n = sampler.accept(z, d, np.zeros(B), seed=5)
    for b in range(B):
        assert n[b] == cut[b]
        assert list(out[b, :n[b]]) == list(d[b, :n[b]])
        assert out[b, n[b]] == y[b, n[b]]
        assert np.all(out[b, n[b] + 1:] == -1)


def _chi2_ok(counts, probs, n):
    exp = probs * n
    keep = exp > 5
    chi2 = float(np.sum((counts[keep] - exp[keep]) ** 2 / exp[keep]))
    dof = int(keep.sum()) - 1
    # p-value > 1e-6 via the Wilson-Hilferty normal approximation
    zz = ((chi2 / dof) ** (1 / 3) - (1 - 2 / (9 * dof))) / math.sqrt(2 / (9 * dof))
    return zz < 4.75


@pytest.mark.parametrize("proposal", ["point", "model"])
def test_emitted_tokens_follow_the_target_distribution(proposal):
    """Speculative sampling is exact: the first emitted token is distributed as
    p_0 = softmax(z[0] / tau), for a point-mass draft and for a model draft
    with its own distribution q (drawn from q, as a drafter would)."""
    V, T, tau, N = 7, 3, 0.8, 12000
    rng = np.random.default_rng(2)
    z = rng.standard_normal((1, T + 1, V)) * 1.5
    w = rng.standard_normal((1, T, V)) * 1.5
    p0 = np.exp(z[0, 0] / tau - np.log(np.sum(np.exp(z[0, 0] / tau))))
    q0 = np.exp(w[0, 0] / tau) / np.sum(np.exp(w[0, 0] / tau))
    counts = np.zeros(V)
    draw = np.random.default_rng(3)
    for s in range(N):
        if proposal == "point":
            d = np.array([[3, 1, 4]])
            out, n = sampler.accept(z, d, [tau], seed=s)
        else:
            d = np.array([[draw.choice(V, p=q0), 0, 0]])
            out, n = sampler.accept(z, d, [tau], seed=s, draft_logits=w)
        counts[out[0, 0]] += 1
    assert _chi2_ok(counts, p0, N)


def test_bonus_token_follows_the_last_position():
    V, T, tau, N = 5, 2, 1.3, 8000
    rng = np.random.default_rng(4)
    z = rng.standard_normal((1, T + 1, V))
    z[0, 0, 2] = 40.0  # drafts certain to be accepted
    z[0, 1, 0] = 40.0
    pT = np.exp(z[0, T] / tau) / np.sum(np.exp(z[0, T] / tau))
    counts = np.zeros(V)
    for s in range(N):
        out, n = sampler.accept(z, np.array([[2, 0]]), [tau], seed=s)
        assert n[0] == T
        counts[out[0, T]] += 1
    assert _chi2_ok(counts, pT, N)


def test_out_of_vocab_draft_is_rejected():
    z = np.zeros((1, 3, 4))
    out, n = sampler.accept(z, np.array([[7, 1]]), [1.0], seed=1)
    assert n[0] == 0 and 0 <= out[0, 0] < 4
