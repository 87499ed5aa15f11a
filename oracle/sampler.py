"""CPU oracle for speculative acceptance (the rejection sampler after the
verify pass).  TEST INFRASTRUCTURE ONLY; numpy, fp64 arithmetic, shares no
code with the CUDA library.

What it computes.  Speculative decoding is exact by construction: the tokens
it emits follow the target model's distribution ("I pushed Qwen3.8-27B to 124
tps on a single request on a RTX 3090", closing paragraph).  Greedy decoding
never reads the draft distribution and a lookup draft is a point-mass proposal
q, a legal proposal for the rejection sampler ("I pushed Qwen3.8-27B to 381
tps for a single request on a RTX 3090", "Lookup-augmented drafting"); a model
drafter's proposal is the softmax of its raw logits with the temperature
applied once ("DFlash2 drafting").  The rule, step by step:

  greedy (tau <= 0): accept draft t while it equals argmax z[t] (smallest index
    on ties); the first mismatch emits that argmax, otherwise the bonus
    argmax z[T] is emitted.
  sampled: p_t = softmax(z[t] / tau); q_t = one-hot(d[t]) or softmax(w[t] / tau).
    Accept d[t] iff u_t q_t(d[t]) < p_t(d[t]).  At the first rejection emit a
    sample of the residual max(0, p_t - q_t) (normalised), else the bonus: a
    sample of p_T.  Samples are exponential races: argmax_i ln r_i + G_i with
    Gumbel variates G_i = -ln(-ln U_i).
  U(b, t, i, k): word number (i mod 4) of the four that Philox4x32-10
    (Salmon, Moraes, Dror and Shaw, "Parallel random numbers: as easy as 1, 2,
    3", SC'11) gives for counter (floor(i / 4), t, b, k) and key (seed low,
    seed high 32 bits), mapped to (floor(w / 2^8) + 0.5) / 2^24: one Philox
    call serves four consecutive vocabulary entries.  (The pages fix no
    random-number generator; this mapping is a reading.)
"""
from __future__ import annotations

import numpy as np

_M0, _M1 = np.uint64(0xD2511F53), np.uint64(0xCD9E8D57)
_W0, _W1 = np.uint64(0x9E3779B9), np.uint64(0xBB67AE85)
_MASK = np.uint64(0xFFFFFFFF)


def philox4x32_10(c0, c1, c2, c3, k0, k1):
    """Philox4x32-10 on arrays of counters (broadcast); returns 4 uint32 arrays."""
    c = [np.asarray(v, np.uint64) & _MASK for v in (c0, c1, c2, c3)]
    k = [np.uint64(int(k0) & 0xFFFFFFFF), np.uint64(int(k1) & 0xFFFFFFFF)]
    for _ in range(10):
        p0 = _M0 * c[0]
        p1 = _M1 * c[2]
        hi0, lo0 = p0 >> np.uint64(32), p0 & _MASK
        hi1, lo1 = p1 >> np.uint64(32), p1 & _MASK
        c = [(hi1 ^ c[1] ^ k[0]) & _MASK, lo1, (hi0 ^ c[3] ^ k[1]) & _MASK, lo0]
        k = [(k[0] + _W0) & _MASK, (k[1] + _W1) & _MASK]
    return [v.astype(np.uint32) for v in c]


def uniform(seed: int, b: int, t: int, i, k: int):
    """U(b, t, i, k) for a scalar or an array of vocabulary indices i."""
    i = np.asarray(i, np.uint64)
    words = philox4x32_10(i // np.uint64(4), t, b, k, seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF)
    w = np.choose((i % np.uint64(4)).astype(np.int64), words)
    return ((w >> np.uint32(8)).astype(np.float64) + 0.5) / 2.0 ** 24


def _softmax_stats(x):
    m = np.max(x)
    lse = m + np.log(np.sum(np.exp(x - m)))
    return lse


def accept(target_logits, draft_tokens, temperature, seed, draft_logits=None, details=False):
    """target_logits [B, T+1, V], draft_tokens [B, T], temperature [B] (<= 0:
    greedy), draft_logits [B, T, V] or None.  Returns (out_tokens [B, T+1] with
    -1 after the emitted token, num_accepted [B]); with details=True also a
    per-sequence record of the decision quantities (for near-tie checks)."""
    z = np.asarray(target_logits, np.float64)
    d = np.asarray(draft_tokens, np.int64)
    B, T1, V = z.shape
    T = T1 - 1
    out = np.full((B, T1), -1, np.int32)
    nacc = np.zeros(B, np.int32)
    recs = []
    for b in range(B):
        tau = float(temperature[b])
        rec = {"accept_margins": [], "race": None}
        n = T
        if not tau > 0:
            for t in range(T):
                y = int(np.argmax(z[b, t]))
                if d[b, t] != y:
                    n = t
                    break
            tok = int(np.argmax(z[b, n]))
        else:
            for t in range(T):
                valid = 0 <= d[b, t] < V
                v = z[b, t] / tau
                lse = _softmax_stats(v)
                p_d = float(np.exp(v[d[b, t]] - lse)) if valid else 0.0
                if draft_logits is None:
                    q_d = 1.0 if valid else 0.0
                else:
                    wv = np.asarray(draft_logits[b, t], np.float64) / tau
                    q_d = float(np.exp(wv[d[b, t]] - _softmax_stats(wv))) if valid else 0.0
                u = float(uniform(seed, b, t, 0, 0))
                rec["accept_margins"].append((u * q_d, p_d))
                if not (valid and u * q_d < p_d):
                    n = t
                    break
            i = np.arange(V, dtype=np.uint64)
            g = -np.log(-np.log(uniform(seed, b, n, i, 1)))
            v = z[b, n] / tau
            if n == T:
                score = v + g
            elif draft_logits is None:
                score = v + g
                if 0 <= d[b, n] < V:
                    score[d[b, n]] = -np.inf
            else:
                p = np.exp(v - _softmax_stats(v))
                wv = np.asarray(draft_logits[b, n], np.float64) / tau
                q = np.exp(wv - _softmax_stats(wv))
                r = p - q
                with np.errstate(divide="ignore", invalid="ignore"):
                    score = np.where(r > 0, np.log(np.where(r > 0, r, 1.0)) + g, -np.inf)
            tok = int(np.argmax(score))
            rec["race"] = score
        out[b, :n] = d[b, :n]
        out[b, n] = tok
        nacc[b] = n
        recs.append(rec)
    return (out, nacc, recs) if details else (out, nacc)
