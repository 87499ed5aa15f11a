"""GPU parity of the KV append with quantise-on-write (through the C ABI)
against the CPU oracle: every code byte and every scale bit-exact (integer
work decided by binary32 quotients on both sides), untouched slots unchanged,
skipped rows flagged, and argument errors reported."""
import numpy as np
import pytest

import oracle

from test_kv_append_oracle import make_case

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from speculative_decoding_verify_causal_gb300 import build
    build.build()


def dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    return t.cuda() if dtype is None else t.view(dtype).cuda()


def run_gpu(k_new, v_new, pages, scale, bt, lens, T, kv_dtype, num_pages=0):
    import speculative_decoding_verify_causal_gb300 as va
    kp, vp = dev(pages), dev(pages)
    ks = None if scale is None else dev(scale)
    vs = None if scale is None else dev(scale)
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    va.verify_attn_kv_append(dev(k_new.view(np.int16), torch.bfloat16), dev(v_new.view(np.int16), torch.bfloat16),
                             kp, vp, ks, vs, dev(bt), dev(lens), T, kv_dtype, num_pages=num_pages, flags=flags)
    torch.cuda.synchronize()
    out = [kp.cpu().numpy(), vp.cpu().numpy(), None if ks is None else ks.cpu().numpy(),
           None if vs is None else vs.cpu().numpy()]
    return out, int(flags.item())


CASES = [(B, T, Hkv, D, dt) for (B, T, Hkv) in ((1, 1, 1), (3, 5, 4), (2, 16, 4), (64, 5, 4))
         for D in (64, 128, 256) for dt in ("fp8_e4m3", "int8", "bf16", "int4", "int2")]


@pytest.mark.parametrize("B,T,Hkv,D,kv_dtype", CASES)
def test_kv_append_bit_exact(B, T, Hkv, D, kv_dtype):
    k_new, v_new, pages, scale, bt, lens, num_pages = make_case(100 + B + T + Hkv + D, B, T, Hkv, D, kv_dtype)
    (kp, vp, ks, vs), flags = run_gpu(k_new, v_new, pages, scale, bt, lens, T, kv_dtype)
    rk, rv, rks, rvs, skipped = oracle.kv_append(k_new, v_new, pages, pages, scale, scale, bt, lens, kv_dtype)
    assert skipped == 0 and flags == 0
    assert np.array_equal(kp, rk) and np.array_equal(vp, rv)
    if scale is not None:
        assert np.array_equal(ks.view(np.uint32), rks.view(np.uint32))
        assert np.array_equal(vs.view(np.uint32), rvs.view(np.uint32))


@pytest.mark.parametrize("kv_dtype", ["fp8_e4m3", "int8", "int4", "int2"])
def test_kv_append_extreme_rows(kv_dtype):
    """Rows of ties, tiny (subnormal-scale) and huge magnitudes, all-equal rows."""
    B, T, Hkv, D = 1, 8, 2, 64
    k_new, v_new, pages, scale, bt, lens, _ = make_case(7, B, T, Hkv, D, kv_dtype)
    f = (k_new.astype(np.uint32) << 16).view(np.float32).copy()
    f[0, 0, 0] = 1e-38                         # tiny row: s underflows towards subnormal
    f[0, 1, 0] = 3e38                          # huge row
    f[0, 2, 0] = np.linspace(-1, 1, D)         # many ties after scaling
    f[0, 3, 1] = 2.5                           # all equal
    f[0, 4, 1, :] = 0.0
    f[0, 4, 1, 7] = -1e-3
    k_new = (torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16))
    (kp, vp, ks, vs), flags = run_gpu(k_new, v_new, pages, scale, bt, lens, T, kv_dtype)
    rk, rv, rks, rvs, _ = oracle.kv_append(k_new, v_new, pages, pages, scale, scale, bt, lens, kv_dtype)
    assert np.array_equal(kp, rk) and np.array_equal(vp, rv)
    assert np.array_equal(ks.view(np.uint32), rks.view(np.uint32))


def test_kv_append_skips_and_flags_bad_rows():
    B, T, Hkv, D = 2, 4, 2, 128
    k_new, v_new, pages, scale, bt, lens, num_pages = make_case(9, B, T, Hkv, D, "int8", extra_pages=8)
    lens = lens.copy()
    bt = bt.copy()
    lens[1] = 2  # positions -2, -1: skipped
    pos = lens[0] - T
    bt[0, pos // 16] = num_pages + 3  # allocated (see below) but outside the planned pool
    big = np.concatenate([pages, np.zeros((8,) + pages.shape[1:], pages.dtype)])  # pool larger than num_pages
    big_scale = np.concatenate([scale, np.zeros((8,) + scale.shape[1:], scale.dtype)])
    (kp, vp, ks, vs), flags = run_gpu(k_new, v_new, big, big_scale, bt, lens, T, "int8", num_pages=num_pages)
    rk, rv, rks, rvs, skipped = oracle.kv_append(k_new, v_new, big, big, big_scale, big_scale, bt, lens, "int8",
                                                 num_pages=num_pages)
    assert skipped > 0 and flags & 1
    assert np.array_equal(kp, rk) and np.array_equal(vp, rv) and np.array_equal(ks, rks)


def test_kv_append_argument_errors():
    import speculative_decoding_verify_causal_gb300 as va
    k_new, v_new, pages, scale, bt, lens, _ = make_case(3, 1, 2, 1, 64, "int8")
    kn = dev(k_new.view(np.int16), torch.bfloat16)
    with pytest.raises(ValueError):  # the binding refuses a quantised cache without scales
        va.verify_attn_kv_append(kn, kn, dev(pages), dev(pages), None, None, dev(bt), dev(lens), 2, "int8")
    lib = va.library()
    import ctypes
    P = ctypes.c_void_p
    kp = dev(pages)
    btd, lsd = dev(bt), dev(lens)
    ptr = lambda t: P(t.data_ptr())
    # null scales through the C ABI itself
    assert lib.verify_attn_kv_append(ptr(kn), ptr(kn), 1, 2, 1, 64, 2, ptr(kp), ptr(kp), P(0), P(0), ptr(btd),
                                     bt.shape[1], ptr(lsd), 0, P(0), P(0)) == -1
    assert lib.verify_attn_kv_append(P(0), P(0), 1, 2, 1, 64, 2, P(0), P(0), P(0), P(0), P(0), 1, P(0), 0, P(0),
                                     P(0)) == -1
    k96 = torch.zeros((1, 2, 1, 96), dtype=torch.bfloat16, device="cuda")
    p96 = torch.zeros((4, 16, 1, 96), dtype=torch.int8, device="cuda")
    s96 = torch.zeros((4, 16, 1), dtype=torch.float32, device="cuda")
    with pytest.raises(va.VerifyAttnError):  # head_dim 96 unsupported
        va.verify_attn_kv_append(k96, k96, p96, p96, s96, s96, dev(bt), dev(lens), 2, "int8")
