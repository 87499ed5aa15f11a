"""Pins of the KV-append oracle (CPU): its e4m3 and int8 encoders against the
library casts, the whole append against an independent numpy / torch
restatement of the per-(token, kv head) absmax quantisation, and the
invariants the definition fixes (absmax element at the top code, a zero row
keeps scale 1, round trip within half a code step, untouched slots)."""
import numpy as np
import pytest
import torch

import oracle


def torch_e4m3(y):
    return torch.from_numpy(np.asarray(y, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def e4m3_values():
    """All finite e4m3 magnitudes, ascending (0 .. 448)."""
    codes = np.arange(0, 0x7F, dtype=np.uint8)  # 0x7F is NaN
    return torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()


# ------------------------------------------------------------ encoders
def test_e4m3_encoder_matches_torch_on_every_bf16_value_in_range():
    bits = np.arange(0, 1 << 16, dtype=np.uint32)
    vals = (bits << 16).view(np.float32)
    vals = vals[np.isfinite(vals) & (np.abs(vals) <= 448.0)]
    ours = np.array([oracle.e4m3_encode(v) for v in vals], dtype=np.uint8)
    assert np.array_equal(ours, torch_e4m3(vals))


def test_e4m3_encoder_ties_round_to_even():
    mag = e4m3_values()
    mids = (mag[:-1] + mag[1:]) / 2  # exact in binary32
    for v in np.concatenate([mids, -mids]):
        assert oracle.e4m3_encode(v) == torch_e4m3([v])[0], v
    # a tie between codes 0x38 (1.0) and 0x39 (1.125) goes to the even code
    assert oracle.e4m3_encode(1.0625) == 0x38
    assert oracle.e4m3_encode(1.1875) == 0x3A


def test_e4m3_encoder_random_binary32():
    rng = np.random.default_rng(11)
    mag = np.exp(rng.uniform(np.log(1e-6), np.log(448.0), 20000)).astype(np.float32)
    vals = mag * rng.choice([-1.0, 1.0], mag.size).astype(np.float32)
    ours = np.array([oracle.e4m3_encode(v) for v in vals], dtype=np.uint8)
    assert np.array_equal(ours, torch_e4m3(vals))


def test_e4m3_encoder_signed_zero_and_extremes():
    assert oracle.e4m3_encode(0.0) == 0x00
    assert oracle.e4m3_encode(-0.0) == 0x80
    assert oracle.e4m3_encode(448.0) == 0x7E and oracle.e4m3_encode(-448.0) == 0xFE
    assert oracle.e4m3_encode(2.0 ** -9) == 0x01          # smallest subnormal
    assert oracle.e4m3_encode(2.0 ** -10) == 0x00         # tie with 0 -> even
    assert oracle.e4m3_encode(0.875 * 2.0 ** -6) == 0x07  # largest subnormal
    assert oracle.e4m3_encode(2.0 ** -6) == 0x08          # smallest normal


def test_int8_encoder_half_even_and_clamp():
    rng = np.random.default_rng(12)
    vals = np.concatenate([rng.uniform(-130, 130, 5000), np.arange(-130, 131) + 0.5]).astype(np.float32)
    ours = np.array([oracle.int8_encode(v) for v in vals])
    assert np.array_equal(ours, np.clip(np.rint(vals), -127, 127))


# ------------------------------------------------------------ the append
def reference_quantise(x, kv_dtype):
    """Independent restatement with numpy / torch: rows x [..., D] fp32."""
    a = np.abs(x).max(axis=-1).astype(np.float32)
    qmax = np.float32(448.0 if kv_dtype == "fp8_e4m3" else 127.0)
    s = np.where(a > 0, a / qmax, np.float32(1.0)).astype(np.float32)
    y = (x / s[..., None]).astype(np.float32)
    if kv_dtype == "fp8_e4m3":
        codes = torch_e4m3(np.clip(y, -448.0, 448.0))
    else:
        codes = np.clip(np.rint(y), -127, 127).astype(np.int8).view(np.uint8)
    return codes, s


def bf16_bits(x):
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(
        np.uint16)


def bits_to_f32(b):
    return (b.astype(np.uint32) << 16).view(np.float32)


def make_case(seed, B, T, Hkv, D, kv_dtype, extra_pages=3):
    rng = np.random.default_rng(seed)
    lens = rng.integers(T, 80, B) + T
    npages_seq = (lens + 15) // 16
    num_pages = int(npages_seq.sum()) + extra_pages
    perm = rng.permutation(num_pages)
    bt = np.zeros((B, int(npages_seq.max())), np.int32)
    o = 0
    for b in range(B):
        bt[b, :npages_seq[b]] = perm[o:o + npages_seq[b]]
        o += npages_seq[b]
    x = rng.standard_normal((2, B, T, Hkv, D)).astype(np.float32) * rng.uniform(0.01, 50, (2, B, T, Hkv, 1))
    x[0, 0, 0, 0] = 0.0           # a zero row
    x[1, -1, -1, -1, 3] = -0.0    # a negative zero
    k_new, v_new = bf16_bits(x[0]), bf16_bits(x[1])
    if kv_dtype == "bf16":
        pages = np.full((num_pages, 16, Hkv, D), 0x1234, np.uint16)
        scale = None
    elif kv_dtype in ("int4", "int2"):  # packed bytes, D * bits / 8 per row
        bits = 4 if kv_dtype == "int4" else 2
        pages = np.full((num_pages, 16, Hkv, D * bits // 8), 0x5A, np.uint8)
        scale = np.full((num_pages, 16, Hkv), 7.0, np.float32)
    else:
        pages = np.full((num_pages, 16, Hkv, D), 0x5A, np.int8 if kv_dtype == "int8" else np.uint8)
        scale = np.full((num_pages, 16, Hkv), 7.0, np.float32)
    return k_new, v_new, pages, scale, bt, lens.astype(np.int32), num_pages


@pytest.mark.parametrize("kv_dtype", ["fp8_e4m3", "int8", "bf16"])
@pytest.mark.parametrize("D", [64, 256])
def test_append_matches_independent_restatement(kv_dtype, D):
    B, T, Hkv = 3, 5, 4
    k_new, v_new, pages, scale, bt, lens, num_pages = make_case(5 + D, B, T, Hkv, D, kv_dtype)
    kp, vp, ks, vs, skipped = oracle.kv_append(k_new, v_new, pages, pages, scale, scale, bt, lens, kv_dtype)
    assert skipped == 0
    written = np.zeros((num_pages, 16), bool)
    for b in range(B):
        for t in range(T):
            pos = lens[b] - T + t
            page, slot = bt[b, pos // 16], pos % 16
            written[page, slot] = True
            for src, dst, dsc in ((k_new, kp, ks), (v_new, vp, vs)):
                row = bits_to_f32(src[b, t])  # [Hkv, D]
                if kv_dtype == "bf16":
                    assert np.array_equal(dst[page, slot], src[b, t])
                else:
                    codes, s = reference_quantise(row, kv_dtype)
                    assert np.array_equal(dst[page, slot].view(np.uint8), codes)
                    assert np.array_equal(dsc[page, slot], s)
    # every other slot untouched
    assert np.array_equal(kp[~written], pages[~written]) and np.array_equal(vp[~written], pages[~written])
    if scale is not None:
        assert np.array_equal(ks[~written], scale[~written])


def packbits_codes(codes, bits):
    """Signed codes [..., D] -> bytes [..., D * bits / 8] through numpy's
    little-endian bit packing (independent of the oracle's shifts)."""
    u = (codes.astype(np.int64) & ((1 << bits) - 1))
    b = ((u[..., None] >> np.arange(bits)) & 1).astype(np.uint8)  # [..., D, bits], low bit first
    return np.packbits(b.reshape(*codes.shape[:-1], -1), axis=-1, bitorder="little")


@pytest.mark.parametrize("kv_dtype,bits,qmax", [("int4", 4, 7), ("int2", 2, 1)])
@pytest.mark.parametrize("D", [64, 256])
def test_append_packed_matches_independent_restatement(kv_dtype, bits, qmax, D):
    """4-bit / 2-bit caches: every written row equals the int8 rule with
    qmax 7 / 1 (binary32 absmax scale, round-half-even, clamp) packed with
    numpy's bit packing; every other byte and scale is untouched."""
    B, T, Hkv = 3, 5, 4
    k_new, v_new, pages, scale, bt, lens, num_pages = make_case(7 + D + bits, B, T, Hkv, D, kv_dtype)
    assert pages.shape == (num_pages, 16, Hkv, D * bits // 8) and pages.dtype == np.uint8
    kp, vp, ks, vs, skipped = oracle.kv_append(k_new, v_new, pages, pages, scale, scale, bt, lens, kv_dtype)
    assert skipped == 0
    written = np.zeros((num_pages, 16), bool)
    for b in range(B):
        for t in range(T):
            pos = lens[b] - T + t
            page, slot = bt[b, pos // 16], pos % 16
            written[page, slot] = True
            for src, dst, dsc in ((k_new, kp, ks), (v_new, vp, vs)):
                x = bits_to_f32(src[b, t])  # [Hkv, D]
                a = np.abs(x).max(axis=-1).astype(np.float32)
                sc = np.where(a > 0, a / np.float32(qmax), np.float32(1.0)).astype(np.float32)
                codes = np.clip(np.rint((x / sc[:, None]).astype(np.float32)), -qmax, qmax)
                assert np.array_equal(dst[page, slot], packbits_codes(codes, bits))
                assert np.array_equal(dsc[page, slot], sc)
    assert np.array_equal(kp[~written], pages[~written]) and np.array_equal(vp[~written], pages[~written])
    assert np.array_equal(ks[~written], scale[~written])


@pytest.mark.parametrize("kv_dtype", ["fp8_e4m3", "int8"])
def test_append_invariants(kv_dtype):
    B, T, Hkv, D = 2, 16, 2, 128
    k_new, v_new, pages, scale, bt, lens, num_pages = make_case(21, B, T, Hkv, D, kv_dtype)
    kp, vp, ks, vs, _ = oracle.kv_append(k_new, v_new, pages, pages, scale, scale, bt, lens, kv_dtype)
    top = 0x7E if kv_dtype == "fp8_e4m3" else 127
    for b in range(B):
        for t in range(T):
            pos = lens[b] - T + t
            page, slot = bt[b, pos // 16], pos % 16
            for g in range(Hkv):
                x = bits_to_f32(k_new[b, t, g])
                codes, s = kp[page, slot, g].view(np.uint8), ks[page, slot, g]
                if not np.any(x):
                    assert s == 1.0 and not np.any(codes)
                    continue
                if kv_dtype == "fp8_e4m3":
                    dec = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).float().numpy()
                    # absmax element at +-448; round trip within half a step (2^-4 relative, or 2^-10 s)
                    assert (codes[np.argmax(np.abs(x))] & 0x7F) == top
                    err = np.abs(dec * s - x)
                    assert np.all(err <= np.maximum(np.abs(x) * 2.0 ** -4, s * 2.0 ** -10) * 1.0001)
                else:
                    dec = codes.view(np.int8).astype(np.float32)
                    assert abs(int(codes.view(np.int8)[np.argmax(np.abs(x))])) == top
                    assert np.all(np.abs(dec * s - x) <= 0.5 * s * 1.0001)


def test_append_skips_rows_outside_the_pool():
    B, T, Hkv, D = 2, 4, 1, 64
    k_new, v_new, pages, scale, bt, lens, num_pages = make_case(31, B, T, Hkv, D, "int8")
    lens = lens.copy()
    lens[1] = 2                     # fewer tokens than T: positions -2, -1 are skipped
    bt = bt.copy()
    pos = lens[0] - T               # first new token of sequence 0
    bt[0, pos // 16] = num_pages + 5  # a page outside the pool
    kp, vp, ks, vs, skipped = oracle.kv_append(k_new, v_new, pages, pages, scale, scale, bt, lens, "int8",
                                               num_pages=num_pages)
    n_bad_page = sum(1 for t in range(T) if (lens[0] - T + t) // 16 == pos // 16)
    assert skipped == 2 * Hkv * (n_bad_page + 2)


def test_append_rejects_bad_arguments():
    k_new, v_new, pages, scale, bt, lens, _ = make_case(41, 1, 2, 1, 64, "int8")
    with pytest.raises(ValueError):
        oracle.kv_append(k_new, v_new, pages, pages, None, None, bt, lens, "int8")
