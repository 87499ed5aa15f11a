"""GPU parity of the acceptance sampler (through the C ABI) against the CPU
oracle: greedy decisions exact; sampled decisions equal except where the
oracle's fp64 decision quantities are within a few binary32 ulps (the kernel
decides in binary32 with the CUDA math library) -- such near-ties are counted
and must be rare and genuine."""
import numpy as np
import pytest

from oracle import sampler

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from speculative_decoding_verify_causal_gb300 import build
    build.build()


def make(seed, B, T, V, greedy_frac=0.3, match_frac=0.7, model=False):
    rng = np.random.default_rng(seed)
    z = (rng.standard_normal((B, T + 1, V)) * rng.uniform(0.5, 4, (B, 1, 1))).astype(np.float32)
    y = z.argmax(-1)
    d = y[:, :T].copy()
    flip = rng.random((B, T)) > match_frac
    d[flip] = rng.integers(0, V, flip.sum())
    tau = np.where(rng.random(B) < greedy_frac, 0.0, rng.uniform(0.3, 1.5, B)).astype(np.float32)
    w = (z[:, :T] + rng.standard_normal((B, T, V)).astype(np.float32)) if model else None
    return z, d.astype(np.int32), tau, w


def run(z, d, tau, seed, w=None):
    import speculative_decoding_verify_causal_gb300 as va
    out, n = va.verify_attn_accept(torch.from_numpy(z).cuda(), torch.from_numpy(d).cuda(),
                                   torch.from_numpy(tau).cuda(), seed,
                                   None if w is None else torch.from_numpy(w).cuda())
    torch.cuda.synchronize()
    return out.cpu().numpy(), n.cpu().numpy()


def near_tie(rec, n_gpu, tok_gpu, n_ref, tau_b):
    """True if the CPU and GPU may legitimately differ: an acceptance test whose
    u q and p are within 1e-5 relative, or a race whose best two fp64 scores
    (the GPU's pick and the true maximum) are within 1e-4."""
    for uq, p in rec["accept_margins"][:min(n_gpu, n_ref) + 1]:
        if abs(uq - p) <= 1e-5 * max(abs(p), 1e-30):
            return True
    if rec["race"] is not None and n_gpu == n_ref:
        sc = rec["race"]
        return np.isfinite(sc[tok_gpu]) and sc.max() - sc[tok_gpu] <= 1e-4 * (1 + abs(sc.max()))
    return False


def check_against_oracle(z, d, tau, seed, w, out, n):
    """Greedy rows exact; sampled rows equal or at a genuine near-tie, and
    such rows rare; every row well formed."""
    B, T = d.shape
    V = z.shape[2]
    ref_out, ref_n, recs = sampler.accept(z, d, tau, seed, draft_logits=w, details=True)
    mism = 0
    for b in range(B):
        same = n[b] == ref_n[b] and np.array_equal(out[b], ref_out[b])
        if same:
            continue
        assert not tau[b] <= 0, f"greedy sequence {b} differs"
        assert near_tie(recs[b], int(n[b]), int(out[b, n[b]]), int(ref_n[b]), tau[b]), b
        mism += 1
    assert mism <= max(1, B // 50)
    # structure of every row: accepted drafts, then one token, then -1
    for b in range(B):
        assert np.array_equal(out[b, :n[b]], d[b, :n[b]]) and 0 <= out[b, n[b]] < V
        assert np.all(out[b, n[b] + 1:] == -1)


@pytest.mark.parametrize("B,T,V,model", [(64, 5, 50, False), (32, 16, 1000, False), (16, 8, 32000, False),
                                         (32, 5, 1000, True), (4, 16, 151_936, False), (64, 5, 151_936, False),
                                         (8, 4, 777, True), (6, 3, 50, True)])
def test_accept_matches_oracle(B, T, V, model):
    # the last three: the benchmark's batch of 64 sequences over the full
    # vocabulary (race grid capped at one GPU wave), and model drafters on
    # vocabularies that are not a multiple of 4 (scalar loads in both kernels)
    z, d, tau, w = make(B * 7 + T + V, B, T, V, model=model)
    seed = 0x1234_5678_9ABC + V
    out, n = run(z, d, tau, seed, w)
    check_against_oracle(z, d, tau, seed, w, out, n)


def test_accept_logits_off_a_16_byte_boundary():
    # V a multiple of 4, but both logit arrays start 4 bytes past a 16-byte
    # boundary: both kernels must take their scalar loads
    import speculative_decoding_verify_causal_gb300 as va
    B, T, V = 16, 4, 1000
    z, d, tau, w = make(77, B, T, V, model=True)

    def shifted(a):
        buf = torch.empty(a.size + 1, dtype=torch.float32, device="cuda")
        t = buf[1:].view(a.shape)
        t.copy_(torch.from_numpy(a))
        assert t.data_ptr() % 16 == 4
        return t

    seed = 4242
    out, n = va.verify_attn_accept(shifted(z), torch.from_numpy(d).cuda(), torch.from_numpy(tau).cuda(), seed,
                                   shifted(w))
    torch.cuda.synchronize()
    check_against_oracle(z, d, tau, seed, w, out.cpu().numpy(), n.cpu().numpy())


def test_accept_all_greedy_exact_and_bonus():
    B, T, V = 20, 16, 777
    z, d, tau, _ = make(9, B, T, V, greedy_frac=1.0, match_frac=1.0)
    out, n = run(z, d, tau, 3)
    ref_out, ref_n = sampler.accept(z, d, tau, 3)
    assert np.array_equal(n, ref_n) and np.array_equal(out, ref_out)
    assert np.all(n == T)


def test_accept_argument_errors():
    import ctypes
    import speculative_decoding_verify_causal_gb300 as va
    lib = va.library()
    P = ctypes.c_void_p
    assert lib.verify_attn_accept(P(0), P(0), P(0), P(0), 1, 1, 10, 0, P(0), P(0), P(0), P(0)) == -1
    assert lib.verify_attn_accept_workspace_bytes(0, 1) == 0
    with pytest.raises(ValueError):
        va.verify_attn_accept(torch.zeros((2, 3, 4), device="cuda"), torch.zeros((2, 3), dtype=torch.int32,
                              device="cuda"), torch.ones(2, device="cuda"), 1)


def _one_hot_prefix(T, V, d_tok, rng):
    """Positions 0..T-1 put logit 100 on the draft token (binary32 p(d) is
    exactly 1, fp64 p(d) is 1 - V e^-100 = 1.0), so every draft is accepted
    whenever u < 1; position T is a random row."""
    z = np.zeros((1, T + 1, V), np.float32)
    z[0, :T, d_tok] = 100.0
    z[0, T] = rng.standard_normal(V).astype(np.float32)
    return z, np.full((1, T), d_tok, np.int32), np.ones(1, np.float32)


def test_accept_uniform_at_the_top_of_its_range():
    # seed 46 draws j = 2^24 - 1 for the acceptance uniform of position 342,
    # so U = 1 - 2^-25; its binary32 value must stay below 1 or the draft with
    # p(d) = 1 would be rejected
    seed, T, V = 46, 400, 8
    assert sampler.uniform(seed, 0, 342, 0, 0) == 1.0 - 2.0 ** -25
    z, d, tau = _one_hot_prefix(T, V, 3, np.random.default_rng(1))
    out, n = run(z, d, tau, seed)
    ref_out, ref_n, recs = sampler.accept(z, d, tau, seed, details=True)
    assert ref_n[0] == T and n[0] == T
    assert out[0, T] == ref_out[0, T] or near_tie(recs[0], int(n[0]), int(out[0, T]), int(ref_n[0]), tau[0])


def test_race_gumbel_at_the_top_of_the_uniform_range():
    # seed 4714 draws j = 2^24 - 1 for the race uniform of entry 2687 at
    # position 2: its Gumbel is ln 2^25 = 17.33, finite, so with logit -30 it
    # must lose to the zero-logit entries (an infinite Gumbel would win)
    seed, T, V, i_top = 4714, 2, 4096, 2687
    assert sampler.uniform(seed, 0, T, i_top, 1) == 1.0 - 2.0 ** -25
    z, d, tau = _one_hot_prefix(T, V, 7, np.random.default_rng(2))
    z[0, T] = 0.0
    z[0, T, i_top] = -30.0
    out, n = run(z, d, tau, seed)
    ref_out, ref_n, recs = sampler.accept(z, d, tau, seed, details=True)
    assert ref_n[0] == T and n[0] == T and ref_out[0, T] != i_top
    assert out[0, T] != i_top
    assert out[0, T] == ref_out[0, T] or near_tie(recs[0], int(n[0]), int(out[0, T]), int(ref_n[0]), tau[0])


def test_race_gumbels_track_the_oracle_near_u_one():
    # equal logits make the race a pure Gumbel maximum, decided among the
    # largest uniforms, where -ln U is smallest (2^-25 at the top) and must
    # be formed without rounding U to binary32 first: the winner must match
    # the oracle's in every sequence (near ties excepted)
    B, T, V = 32, 1, 50_000
    rng = np.random.default_rng(4)
    z = np.zeros((B, T + 1, V), np.float32)
    z[:, 0, 5] = 100.0
    d = np.full((B, T), 5, np.int32)
    tau = np.ones(B, np.float32)
    out, n = run(z, d, tau, 99)
    ref_out, ref_n, recs = sampler.accept(z, d, tau, 99, details=True)
    assert np.all(n == T) and np.all(ref_n == T)
    bad = [b for b in range(B) if out[b, T] != ref_out[b, T]
           and not near_tie(recs[b], int(n[b]), int(out[b, T]), int(ref_n[b]), tau[b])]
    assert not bad, bad
