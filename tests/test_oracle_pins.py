"""Pins for the CPU oracle: each test checks it against something other than
itself (a library routine, a closed form, an invariant or a brute-force
restatement), so that a dropped term, a wrong sign or index or a transposed
operand in the oracle fails at least one of them.  CPU only."""
import math

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verify_causal_gb300 import workloads as wl

PAGE = 16


# ---------------------------------------------------------------- helpers
PACKED_BITS = {"int4": 4, "int2": 2}


def unpack_codes(raw, bits, D):
    """Packed bytes [..., D * bits / 8] -> signed codes [..., D], through
    numpy's little-endian bit unpacking (a different route from the oracle's
    shifts and masks): field d is bits d*bits .. d*bits+bits-1 of the row."""
    b = np.unpackbits(np.ascontiguousarray(raw, np.uint8)[..., None], axis=-1, bitorder="little")
    b = b.reshape(*raw.shape[:-1], D, bits).astype(np.int64)
    u = (b * (1 << np.arange(bits))).sum(-1)
    return np.where(u >= (1 << (bits - 1)), u - (1 << bits), u)


def dense_kv(w, which):
    """Independent dequantisation with torch dtypes: [B][L_b, Hkv, D] float64."""
    raw = w[which + "_pages"]
    dt = w["kv_dtype"]
    t = torch.from_numpy(np.ascontiguousarray(raw))
    if dt == "bf16":
        vals = t.view(torch.bfloat16).to(torch.float64)
    elif dt == "fp8_e4m3":
        vals = t.view(torch.float8_e4m3fn).to(torch.float64)
    elif dt in PACKED_BITS:
        vals = torch.from_numpy(unpack_codes(raw, PACKED_BITS[dt], w["D"]).astype(np.float64))
    else:
        vals = t.to(torch.float64)
    if dt != "bf16":
        sc = torch.from_numpy(w[which + "_scale"]).to(torch.float64)
        vals = vals * sc[..., None]
    flat = vals.reshape(-1, w["Hkv"], w["D"])
    out = []
    for b, L in enumerate(w["seq_lens"]):
        tok = np.arange(L)
        phys = w["block_table"][b, tok // PAGE].astype(np.int64) * PAGE + tok % PAGE
        out.append(flat[torch.from_numpy(phys)])
    return out


def q_f64(w):
    return torch.from_numpy(w["q"].view(np.int16)).view(torch.bfloat16).to(torch.float64)


def sdpa_reference(w):
    """Brute force with torch's SDPA in float64, explicit bottom-right causal
    mask and GQA by repeat_interleave."""
    T, Hq, Hkv, D = w["T"], w["Hq"], w["Hkv"], w["D"]
    G = Hq // Hkv
    q = q_f64(w)
    K = dense_kv(w, "k")
    V = dense_kv(w, "v")
    outs, lses = [], []
    for b, L in enumerate(w["seq_lens"]):
        qb = q[b].permute(1, 0, 2)  # [Hq, T, D]
        kb = K[b].permute(1, 0, 2).repeat_interleave(G, dim=0)  # [Hq, L, D]
        vb = V[b].permute(1, 0, 2).repeat_interleave(G, dim=0)
        t = torch.arange(T)[:, None]
        j = torch.arange(L)[None, :]
        mask = j <= (L - T + t)
        o = torch.nn.functional.scaled_dot_product_attention(
            qb, kb, vb, attn_mask=mask, scale=1.0 / math.sqrt(D))
        s = torch.matmul(qb, kb.transpose(1, 2)) / math.sqrt(D)
        s = s.masked_fill(~mask, float("-inf"))
        outs.append(o.permute(1, 0, 2).numpy())
        lses.append(torch.logsumexp(s, dim=-1).permute(1, 0).numpy())
    return np.stack(outs), np.stack(lses)


def small_workload(seed, lens, T, Hq, Hkv, D, dt, **kw):
    return wl.make_workload(seed, lens, T, Hq, Hkv, D, dt, **kw)


# ---------------------------------------------------------------- decoders
def test_e4m3_decoder_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.decode_e4m3(int(c)) for c in codes])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert nan.sum() == 2  # S.1111.111 only
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.nanmax(got) == 448.0 and np.nanmin(got) == -448.0
    assert oracle.decode_e4m3(0x01) == 2.0 ** -9  # smallest subnormal


@pytest.mark.parametrize("bits", [4, 2])
def test_packed_decoder_all_bytes(bits):
    """Every byte value at every field position: the oracle's packed decoder
    against numpy's bit unpacking and the two's-complement rule."""
    data = np.arange(256, dtype=np.uint8)
    per = 8 // bits
    got = np.array([oracle.decode_packed(data, i, bits) for i in range(256 * per)])
    ref = unpack_codes(data.reshape(256, 1), bits, per).reshape(-1)
    assert np.array_equal(got, ref)
    assert got.min() == -(1 << (bits - 1)) and got.max() == (1 << (bits - 1)) - 1


@pytest.mark.parametrize("dt,qmax", [("int4", 7), ("int2", 1)])
def test_packed_generator_round_trip(dt, qmax):
    """Rows quantised by the input generator come back, through the oracle's
    decoder, within half a code step: |x - code * s| <= s / 2, |code| <= qmax,
    each row's largest |x| on a top code, an all-zero row on code 0."""
    rng = np.random.Generator(np.random.PCG64(31))
    x = (rng.standard_normal((50, 64)) * rng.uniform(0.01, 30.0, (50, 1))).astype(np.float32)
    x[7] = 0.0
    raw, s = wl._quantise(x, dt)
    bits = PACKED_BITS[dt]
    codes = np.array([[oracle.decode_packed(raw[r], d, bits) for d in range(64)] for r in range(50)])
    assert np.abs(codes).max() <= qmax
    err = np.abs(x.astype(np.float64) - codes * s[:, None].astype(np.float64))
    assert (err <= s[:, None] * (0.5 + 1e-6)).all()
    nz = np.arange(50) != 7
    assert (np.abs(codes[nz][np.arange(49), np.abs(x[nz]).argmax(1)]) == qmax).all()
    assert (codes[7] == 0).all() and s[7] == 1.0


def test_bf16_decoder_random_codes():
    rng = np.random.default_rng(1)
    codes = rng.integers(0, 1 << 16, size=4096, dtype=np.uint16)
    ref = torch.from_numpy(codes.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.decode_bf16(int(c)) for c in codes])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


# ---------------------------------------------------------------- brute force
@pytest.mark.parametrize("dt", ["bf16", "fp8_e4m3", "int8", "int4", "int2"])
@pytest.mark.parametrize("T,Hq,Hkv,D,lens", [
    (5, 4, 1, 64, [37]),
    (3, 6, 2, 16, [19, 40]),
    (1, 4, 4, 8, [5, 16, 17]),
    (16, 8, 2, 32, [16, 50]),
])
def test_oracle_matches_sdpa_float64(dt, T, Hq, Hkv, D, lens):
    w = small_workload(100 + T + D, lens, T, Hq, Hkv, D, dt, extra_pages=3)
    out, lse = oracle.verify_attn(w)
    ref_out, ref_lse = sdpa_reference(w)
    np.testing.assert_allclose(out, ref_out, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-13, atol=1e-12)


# ---------------------------------------------------------------- invariants
def _set_all_v_to_one(w):
    dt = w["kv_dtype"]
    if dt == "bf16":
        w["v_pages"][...] = 0x3F80
    elif dt == "fp8_e4m3":
        w["v_pages"][...] = 0x38  # 1.0 in e4m3
        w["v_scale"][...] = 1.0
    elif dt in PACKED_BITS:  # code 1 in every field
        bits = PACKED_BITS[dt]
        w["v_pages"][...] = sum(1 << (bits * k) for k in range(8 // bits))
        w["v_scale"][...] = 1.0
    else:
        w["v_pages"][...] = 1
        w["v_scale"][...] = 1.0


@pytest.mark.parametrize("dt", ["bf16", "fp8_e4m3", "int8", "int4", "int2"])
def test_softmax_rows_sum_to_one(dt):
    w = small_workload(7, [23, 64], 4, 6, 3, 32, dt)
    _set_all_v_to_one(w)
    out, _ = oracle.verify_attn(w)
    np.testing.assert_allclose(out, 1.0, rtol=0, atol=1e-12)


@pytest.mark.parametrize("dt", ["bf16", "int8", "int4", "int2"])
def test_T1_is_plain_decode_of_last_verify_token(dt):
    T = 5
    w = small_workload(11, [70], T, 4, 2, 16, dt)
    out, lse = oracle.verify_attn(w)
    w1 = dict(w)
    w1["q"] = np.ascontiguousarray(w["q"][:, T - 1:T])
    w1["T"] = 1
    out1, lse1 = oracle.verify_attn(w1)
    assert np.array_equal(out1[:, 0], out[:, T - 1])
    assert np.array_equal(lse1[:, 0], lse[:, T - 1])
    # and plain (non-causal) decode over all L keys, by torch softmax
    q = q_f64(w1)[0, 0]  # [Hq, D]
    K = dense_kv(w, "k")[0]
    V = dense_kv(w, "v")[0]
    G = 2
    for h in range(4):
        s = (K[:, h // G, :] @ q[h]) / 4.0
        p = torch.softmax(s, dim=0)
        np.testing.assert_allclose(out1[0, 0, h], (p[:, None] * V[:, h // G, :]).sum(0).numpy(),
                                   rtol=0, atol=1e-12)


@pytest.mark.parametrize("dt", ["bf16", "fp8_e4m3", "int8", "int4", "int2"])
def test_identical_keys_closed_form(dt):
    T, Hq, Hkv, D, L = 6, 4, 2, 16, 40
    w = small_workload(13, [L], T, Hq, Hkv, D, dt)
    kp = w["k_pages"]
    # every key row (and its scale) of each kv head equal to the head's first row
    for g in range(Hkv):
        row0 = kp[w["block_table"][0, 0], 0, g].copy()
        kp[:, :, g, :] = row0
        if w["k_scale"] is not None:
            w["k_scale"][:, :, g] = w["k_scale"][w["block_table"][0, 0], 0, g]
    out, lse = oracle.verify_attn(w)
    q = q_f64(w)[0]  # [T, Hq, D]
    K = dense_kv(w, "k")[0]
    V = dense_kv(w, "v")[0]
    for t in range(T):
        n = L - T + t + 1
        for h in range(Hq):
            g = h // (Hq // Hkv)
            s = float(q[t, h] @ K[0, g]) / math.sqrt(D)
            np.testing.assert_allclose(out[0, t, h], V[:n, g].mean(0).numpy(), rtol=0, atol=1e-12)
            assert abs(lse[0, t, h] - (s + math.log(n))) < 1e-12


@pytest.mark.parametrize("split", [1, 7, 16, 33, 64])
def test_split_lse_merge_equals_direct(split):
    w = small_workload(17, [97], 4, 4, 2, 16, "fp8_e4m3")
    out, lse = oracle.verify_attn(w)
    L = 97
    for (t, h) in [(0, 0), (3, 3), (2, 1)]:
        parts = [oracle.verify_attn_partial(w, 0, t, h, a, min(a + split, L)) for a in range(0, L, split)]
        lses = np.array([p[1] for p in parts])
        m = lses.max()
        tot = m + math.log(np.exp(lses - m).sum())
        o = sum(np.exp(l - tot) * p[0] for p, l in zip(parts, lses) if np.isfinite(l))
        assert abs(tot - lse[0, t, h]) < 1e-12
        np.testing.assert_allclose(o, out[0, t, h], rtol=0, atol=1e-12)
        # a split entirely beyond the causal limit reports lse = -inf and out = 0
    o_m, l_m = oracle.verify_attn_partial(w, 0, 0, 0, L - 2, L)
    assert l_m == -math.inf and not o_m.any()


@pytest.mark.parametrize("dt", ["bf16", "fp8_e4m3", "int8", "int4", "int2"])
def test_page_permutation_invariance(dt):
    w = small_workload(19, [45, 33], 3, 4, 2, 16, dt, extra_pages=4)
    out, lse = oracle.verify_attn(w)
    rng = np.random.default_rng(5)
    perm = rng.permutation(w["num_pages"])  # new position of old page p is perm[p]
    w2 = dict(w)
    for key in ("k_pages", "v_pages", "k_scale", "v_scale"):
        if w[key] is not None:
            a = np.empty_like(w[key])
            a[perm] = w[key]
            w2[key] = a
    w2["block_table"] = perm[w["block_table"]].astype(np.int32)
    out2, lse2 = oracle.verify_attn(w2)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def test_needle_dominates():
    T, Hq, Hkv, D, L = 5, 4, 1, 64, 261
    w = small_workload(23, [L], T, Hq, Hkv, D, "int8", needles=lambda rng, b, L: [100])
    out, lse = oracle.verify_attn(w)
    K = dense_kv(w, "k")[0][:, 0]
    V = dense_kv(w, "v")[0][:, 0]
    q = q_f64(w)[0, 0, 0]
    s = (K @ q) / math.sqrt(D)
    p = torch.softmax(s, 0)
    non_needle = 1.0 - float(p[100])
    assert non_needle < 1e-3  # the planted key carries the row
    bound = non_needle * float((V - V[100]).abs().max())
    assert np.abs(out[0, 0, 0] - V[100].numpy()).max() <= bound + 1e-12
    # lse = s_needle - ln p_needle exactly, so it sits within -ln(1 - mass) above s_needle
    gap = lse[0, 0, 0] - float(s[100])
    assert 0.0 <= gap <= -math.log1p(-non_needle) + 1e-12


def test_rows_api_matches_full_output():
    w = small_workload(29, [33, 18], 2, 6, 3, 16, "fp8_e4m3")
    out, lse = oracle.verify_attn(w)
    rows = [(0, 0, 0), (1, 1, 5), (0, 1, 3), (1, 0, 2)]
    o, l = oracle.verify_attn_rows(w, rows)
    for i, (b, t, h) in enumerate(rows):
        assert np.array_equal(o[i], out[b, t, h]) and l[i] == lse[b, t, h]


def test_bad_arguments_rejected():
    w = small_workload(31, [20], 4, 4, 2, 16, "int8")
    bad = dict(w)
    bad["seq_lens"] = np.array([3], np.int32)  # shorter than T
    with pytest.raises(ValueError):
        oracle.verify_attn(bad)
    bad = dict(w)
    bad["k_scale"] = None  # quantised cache without scales
    with pytest.raises(ValueError):
        oracle.verify_attn(bad)
    with pytest.raises(ValueError):
        oracle.verify_attn_rows(w, [(0, 4, 0)])  # t out of range


def test_golden_regression_fixture():
    """Stored oracle values (written by tests/golden/make_golden.py, which
    calls only the oracle and the input generator)."""
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "tiny_oracle_rows.txt")
    rows, outs, lses = [], [], []
    with open(path) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            parts = line.split()
            rows.append(tuple(int(x) for x in parts[:3]))
            lses.append(float(parts[3]))
            outs.append([float(x) for x in parts[4:]])
    w = wl.config_workload("tiny")
    o, l = oracle.verify_attn_rows(w, rows)
    np.testing.assert_allclose(l, lses, rtol=0, atol=1e-12)
    np.testing.assert_allclose(o, np.array(outs), rtol=0, atol=1e-12)
