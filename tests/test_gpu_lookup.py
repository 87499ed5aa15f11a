"""GPU parity of lookup-augmented drafting (through the C ABI) against the
CPU oracle: draft, draft length, match end and match length exact for every
sequence of random batches (small vocabularies for many accidental matches,
the real vocabulary with copied segments, long histories), and argument
errors."""
import numpy as np
import pytest

import oracle
from speculative_decoding_verify_causal_gb300 import workloads as wl

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from speculative_decoding_verify_causal_gb300 import build
    build.build()


def run_batch(hists, lo, hi, k, stride=None):
    import speculative_decoding_verify_causal_gb300 as va
    B = len(hists)
    stride = stride or max(1, max(len(h) for h in hists))
    toks = np.full((B, stride), -7, np.int32)
    for b, h in enumerate(hists):
        toks[b, :len(h)] = h
    lens = np.array([len(h) for h in hists], np.int32)
    me = torch.empty(B, dtype=torch.int32, device="cuda")
    ml = torch.empty(B, dtype=torch.int32, device="cuda")
    draft, dlen = va.verify_attn_lookup_draft(torch.from_numpy(toks).cuda(), torch.from_numpy(lens).cuda(), k,
                                              min_match=lo, max_match=hi, match_end=me, match_len=ml)
    torch.cuda.synchronize()
    return draft.cpu().numpy(), dlen.cpu().numpy(), me.cpu().numpy(), ml.cpu().numpy()


@pytest.mark.parametrize("vocab,lo,hi,k", [(2, 3, 12, 8), (4, 6, 12, 16), (16, 2, 32, 7), (151_936, 6, 12, 16),
                                           (151_936, 1, 1, 256)])
def test_lookup_batch_exact(vocab, lo, hi, k):
    rng = np.random.default_rng(vocab + hi)
    hists = [wl.token_history(int(rng.integers(1 << 30)), int(L), vocab=vocab, copy_frac=0.3)
             for L in rng.integers(0, 5000, 40)]
    hists += [np.zeros(0, np.int32), np.array([5], np.int32), np.arange(3, dtype=np.int32)]
    draft, dlen, me, ml = run_batch(hists, lo, hi, k)
    for b, h in enumerate(hists):
        d, n, e, m = oracle.lookup_draft(h, lo, hi, k)
        assert (dlen[b], me[b], ml[b]) == (n, e, m), b
        assert np.array_equal(draft[b], d), b


@pytest.mark.parametrize("L", [25_016, 262_160])
def test_lookup_long_history(L):
    h = wl.token_history(L, L, copy_frac=0.3)
    h[-10:] = h[L // 3:L // 3 + 10]  # a known 10-token occurrence far back
    draft, dlen, me, ml = run_batch([h], 6, 12, 16)
    d, n, e, m = oracle.lookup_draft(h, 6, 12, 16)
    assert (dlen[0], me[0], ml[0]) == (n, e, m) and np.array_equal(draft[0], d)
    assert m >= 10


def test_lookup_argument_errors():
    import ctypes
    import speculative_decoding_verify_causal_gb300 as va
    lib = va.library()
    P = ctypes.c_void_p
    t = torch.zeros((1, 8), dtype=torch.int32, device="cuda")
    ptr = P(t.data_ptr())
    assert lib.verify_attn_lookup_draft(P(0), 8, ptr, 1, 6, 12, 4, ptr, ptr, P(0), P(0), P(0)) == -1
    assert lib.verify_attn_lookup_draft(ptr, 8, ptr, 1, 6, 33, 4, ptr, ptr, P(0), P(0), P(0)) == -1  # max_match
    assert lib.verify_attn_lookup_draft(ptr, 8, ptr, 1, 7, 6, 4, ptr, ptr, P(0), P(0), P(0)) == -1   # min > max
    assert lib.verify_attn_lookup_draft(ptr, 8, ptr, 1, 6, 12, 0, ptr, ptr, P(0), P(0), P(0)) == -1  # num_draft
