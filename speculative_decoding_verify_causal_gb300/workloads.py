"""Seeded synthetic workloads for verify attention.

This module only *makes inputs*: random numbers, rounding to the stored
formats, page shuffling and the planted needles / peaks.  It holds none of the
attention arithmetic, so the CUDA path and the CPU oracle can both be fed from
it without sharing any of the method's code.

Input recipe (the same for tests, smoke check and benchmark):

* RNG: ``numpy.random.Generator(PCG64(seed))``; the named configs use
  ``seed = 20260 + index``.
* q, k, v ~ N(0, 1) in fp32, rounded to bf16 (round-to-nearest-even).
* Quantised caches store one fp32 scale per (token, kv-head):
  ``a = max |x|`` over head_dim; fp8-e4m3 uses ``s = a / 448`` and stores
  ``e4m3(x / s)`` (round-to-nearest-even, clamped to +-448); int8 uses
  ``s = a / 127`` and stores ``clamp(rint(x / s), -127, 127)``; ``a == 0``
  gives ``s = 1``.  int4 / int2 follow int8 with ``qmax`` = 7 / 1 and pack the
  two's-complement codes little-end first (element d at bit (d * bits) % 8 of
  byte d * bits / 8): a row of head_dim codes is head_dim / 2 or / 4 bytes.
* Paged cache: 16-token pages, page ids shuffled by the seed; a batch draws its
  pages from one shared pool assigned in order after the shuffle; slots past
  the end of a sequence are zero.
* Needles: key ``20 * qhat`` with ``qhat`` the unit vector of query 0 (first
  q-head of the kv-head's group, verify token 0), planted before quantisation.
* Peaks: a seeded 1 % of (token, kv-head) key rows multiplied by 4 before
  quantisation.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

PAGE = 16
KV_ELEM_BYTES = {"bf16": 2, "fp8_e4m3": 1, "int8": 1}  # whole-byte formats
KV_ELEM_BITS = {"bf16": 16, "fp8_e4m3": 8, "int8": 8, "int4": 4, "int2": 2}
PACKED_QMAX = {"int4": 7, "int2": 1}


def pack_codes(codes: np.ndarray, bits: int) -> np.ndarray:
    """Signed integer codes [..., D] -> packed bytes [..., D * bits / 8], code d
    in bits (d * bits) % 8 .. of byte d * bits / 8 (two's complement)."""
    per = 8 // bits
    c = (codes.astype(np.int16) & ((1 << bits) - 1)).astype(np.uint8)
    c = c.reshape(*codes.shape[:-1], codes.shape[-1] // per, per)
    out = np.zeros(c.shape[:-1], np.uint8)
    for k in range(per):
        out |= (c[..., k] << (bits * k)).astype(np.uint8)
    return out
_CHUNK_TOKENS = 8192  # fixed draw granularity: keeps the stream reproducible


@dataclasses.dataclass(frozen=True)
class Config:
    name: str
    index: int
    seq_lens: tuple  # context lengths before adding T (one per sequence), or None
    T: int
    Hq: int
    Hkv: int
    D: int
    kv_dtype: str
    needles: str = ""  # "random3" | "depths" | ""
    peaks: float = 0.0
    batch: int = 1
    ctx_range: tuple = ()  # (lo, hi) uniform context lengths for a batch

    @property
    def description(self):
        return _DESCRIPTIONS[self.name]


_DESCRIPTIONS = {
    "tiny": "1 seq, 256+5 tokens, 4 q / 1 kv heads, D=64, bf16 KV",
    "mtp4": "1 seq, 1536+5 tokens, 24 q / 4 kv heads, D=256, fp8-e4m3 KV, 3 needles per kv head",
    "lookup16": "1 seq, 25000+16 tokens, 24 q / 4 kv heads, D=256, int8 KV, 1% keys x4",
    "batched": "64 seqs, U[1000,8000]+5 tokens, 24 q / 4 kv heads, D=256, fp8-e4m3 KV, shared page pool",
    "maxctx": "1 seq, 262144+16 tokens, 24 q / 4 kv heads, D=256, int8 KV, needles at 10/50/90/99%",
}

CONFIGS = {
    "tiny": Config("tiny", 0, (256,), 5, 4, 1, 64, "bf16"),
    "mtp4": Config("mtp4", 1, (1536,), 5, 24, 4, 256, "fp8_e4m3", needles="random3"),
    "lookup16": Config("lookup16", 2, (25000,), 16, 24, 4, 256, "int8", peaks=0.01),
    "batched": Config("batched", 3, None, 5, 24, 4, 256, "fp8_e4m3", batch=64, ctx_range=(1000, 8000)),
    "maxctx": Config("maxctx", 4, (262144,), 16, 24, 4, 256, "int8", needles="depths"),
}


def _bf16_round(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 (RNE) -> fp32."""
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16).float().numpy()


def _bf16_bits(x: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _quantise(x: np.ndarray, kv_dtype: str):
    """Store rows x [..., D] (fp32) in the cache format: (raw, scale or None)."""
    if kv_dtype == "bf16":
        return _bf16_bits(x), None
    a = np.max(np.abs(x), axis=-1).astype(np.float32)
    if kv_dtype in PACKED_QMAX:
        qm = PACKED_QMAX[kv_dtype]
        s = np.where(a > 0, a / np.float32(qm), np.float32(1.0)).astype(np.float32)
        y = (x / s[..., None]).astype(np.float32)
        codes = np.clip(np.rint(y), -qm, qm).astype(np.int8)
        return pack_codes(codes, KV_ELEM_BITS[kv_dtype]), s
    qmax = np.float32(448.0 if kv_dtype == "fp8_e4m3" else 127.0)
    s = np.where(a > 0, a / qmax, np.float32(1.0)).astype(np.float32)
    y = (x / s[..., None]).astype(np.float32)
    if kv_dtype == "fp8_e4m3":
        y = np.clip(y, -448.0, 448.0)
        raw = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    else:
        raw = np.clip(np.rint(y), -127, 127).astype(np.int8)
    return raw, s


def _normal_rows(rng, n_tokens, Hkv, D):
    out = np.empty((n_tokens, Hkv, D), np.float32)
    for s in range(0, n_tokens, _CHUNK_TOKENS):
        e = min(n_tokens, s + _CHUNK_TOKENS)
        out[s:e] = rng.standard_normal((e - s, Hkv, D), dtype=np.float32)
    return out


def make_workload(seed, seq_lens, T, Hq, Hkv, D, kv_dtype, *, needles=None, peaks=0.0,
                  extra_pages=0, bt_stride=None, name="custom", k_std=1.0, v_std=1.0):
    """Build one synthetic verify-attention problem.

    ``seq_lens`` are the full lengths L_b (they include the T verify tokens).
    ``needles``: None, or a callable ``(rng, b, L) -> list of token positions``
    at which every kv head gets a needle key.  ``k_std`` / ``v_std`` scale the
    N(0, 1) key / value rows before rounding and quantisation (1 leaves the
    stream of the named configurations unchanged).  Returns a dict of host
    arrays.
    """
    seq_lens = [int(x) for x in seq_lens]
    B = len(seq_lens)
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    G = Hq // Hkv
    rng = np.random.Generator(np.random.PCG64(seed))

    q32 = _bf16_round(rng.standard_normal((B, T, Hq, D), dtype=np.float32))
    pages_per_seq = [(L + PAGE - 1) // PAGE for L in seq_lens]
    num_pages = sum(pages_per_seq) + int(extra_pages)
    perm = rng.permutation(num_pages).astype(np.int32)
    stride = max(pages_per_seq) if bt_stride is None else int(bt_stride)
    if stride < max(pages_per_seq):
        raise ValueError("bt_stride too small")
    block_table = np.zeros((B, stride), np.int32)
    off = 0
    for b, n in enumerate(pages_per_seq):
        block_table[b, :n] = perm[off:off + n]
        off += n

    raw_dtype = {"bf16": np.uint16, "fp8_e4m3": np.uint8, "int8": np.int8, "int4": np.uint8, "int2": np.uint8}[kv_dtype]
    row_elems = D * KV_ELEM_BITS[kv_dtype] // 8 if kv_dtype in PACKED_QMAX else D
    k_pages = np.zeros((num_pages, PAGE, Hkv, row_elems), raw_dtype)
    v_pages = np.zeros((num_pages, PAGE, Hkv, row_elems), raw_dtype)
    quant = kv_dtype != "bf16"
    k_scale = np.zeros((num_pages, PAGE, Hkv), np.float32) if quant else None
    v_scale = np.zeros((num_pages, PAGE, Hkv), np.float32) if quant else None
    needle_pos = []
    k_flat = k_pages.reshape(num_pages * PAGE, Hkv, row_elems)
    v_flat = v_pages.reshape(num_pages * PAGE, Hkv, row_elems)
    for b, L in enumerate(seq_lens):
        k = _normal_rows(rng, L, Hkv, D)
        v = _normal_rows(rng, L, Hkv, D)
        if k_std != 1.0:
            k *= np.float32(k_std)
        if v_std != 1.0:
            v *= np.float32(v_std)
        k = _bf16_round(k)
        v = _bf16_round(v)
        pos = []
        if needles is not None:
            pos = list(needles(rng, b, L))
            for g in range(Hkv):
                q0 = q32[b, 0, g * G].astype(np.float64)
                qhat = (q0 / np.linalg.norm(q0)).astype(np.float32)
                for j in pos:
                    k[j, g] = np.float32(20.0) * qhat
        needle_pos.append(pos)
        if peaks > 0:
            n_pk = int(round(peaks * L * Hkv))
            pick = rng.choice(L * Hkv, size=n_pk, replace=False)
            k.reshape(L * Hkv, D)[pick] *= np.float32(4.0)
        tok = np.arange(L)
        phys = block_table[b, tok // PAGE].astype(np.int64) * PAGE + tok % PAGE
        kr, ks = _quantise(k, kv_dtype)
        vr, vs = _quantise(v, kv_dtype)
        k_flat[phys] = kr
        v_flat[phys] = vr
        if quant:
            k_scale.reshape(-1, Hkv)[phys] = ks
            v_scale.reshape(-1, Hkv)[phys] = vs
        del k, v, kr, vr
    return {
        "name": name,
        "seed": seed,
        "q": _bf16_bits(q32),
        "k_pages": k_pages,
        "v_pages": v_pages,
        "k_scale": k_scale,
        "v_scale": v_scale,
        "block_table": block_table,
        "seq_lens": np.asarray(seq_lens, np.int32),
        "T": T,
        "Hq": Hq,
        "Hkv": Hkv,
        "D": D,
        "kv_dtype": kv_dtype,
        "num_pages": num_pages,
        "needle_pos": needle_pos,
        "k_std": float(k_std),
        "v_std": float(v_std),
    }


def variant_name(name: str, kv_dtype: str | None = None, T: int | None = None, Hq: int | None = None,
                 ctx: int | None = None) -> str:
    """Label of a named configuration with some of its fields replaced."""
    tags = [f"{k}{v}" if k != "kv" else str(v)
            for k, v in (("kv", kv_dtype), ("T", T), ("Hq", Hq), ("ctx", ctx)) if v is not None]
    return "/".join([name] + tags)


def describe(name: str, kv_dtype: str | None = None, T: int | None = None, Hq: int | None = None,
             ctx: int | None = None) -> str:
    """One-line description of a (possibly modified) named configuration."""
    c = CONFIGS[name]
    d = c.description
    if ctx is not None:
        d = d.replace(f"{c.seq_lens[0]}+", f"{ctx}+")
    if kv_dtype is not None:
        d = d.replace(f"{c.kv_dtype.replace('_', '-')} KV", f"{kv_dtype.replace('_', '-')} KV")
    if T is not None:
        d = d.replace(f"+{c.T} tokens", f"+{T} tokens")
    if Hq is not None:
        d = d.replace(f"{c.Hq} q / ", f"{Hq} q / ")
    return d


def config_workload(name: str, kv_dtype: str | None = None, T: int | None = None, Hq: int | None = None,
                    ctx: int | None = None):
    """One of the five named configurations, fully materialised.  ``kv_dtype``,
    ``T`` (verify tokens), ``Hq`` (query heads, a multiple of the kv heads)
    and ``ctx`` (the cached context of a single-sequence configuration)
    replace its fields; the seed and the needle depths (as fractions of the
    context) stay those of the configuration."""
    c = CONFIGS[name]
    if T is not None or Hq is not None or ctx is not None:
        if ctx is not None and c.batch > 1:
            raise ValueError("ctx replaces the context of a single-sequence configuration")
        c = dataclasses.replace(c, T=T if T is not None else c.T, Hq=Hq if Hq is not None else c.Hq,
                                seq_lens=(ctx,) if ctx is not None else c.seq_lens)
    seed = 20260 + c.index
    if c.batch > 1:
        lens_rng = np.random.Generator(np.random.PCG64(seed + 1000))
        ctx = lens_rng.integers(c.ctx_range[0], c.ctx_range[1] + 1, size=c.batch)
        seq_lens = [int(x) + c.T for x in ctx]
    else:
        seq_lens = [x + c.T for x in c.seq_lens]
    needles = None
    if c.needles == "random3":
        def needles(rng, b, L, T=c.T):
            return sorted(int(x) for x in rng.choice(L - T, size=3, replace=False))
    elif c.needles == "depths":
        def needles(rng, b, L, ctx=c.seq_lens[0]):
            return [int(math.floor(p * ctx)) for p in (0.10, 0.50, 0.90, 0.99)]
    return make_workload(seed, seq_lens, c.T, c.Hq, c.Hkv, c.D, kv_dtype or c.kv_dtype,
                         needles=needles, peaks=c.peaks, name=variant_name(name, kv_dtype, T, Hq, ctx))


def algorithmic_bytes(w) -> int:
    """Bytes one verify call must move at minimum: every live KV row of every
    kv head (plus its two scales when quantised), q, out (bf16), lse (fp32),
    the block-table entries in use and seq_lens.  Split partials excluded."""
    Hkv, D, T, Hq = w["Hkv"], w["D"], w["T"], w["Hq"]
    row_bytes = D * KV_ELEM_BITS[w["kv_dtype"]] // 8
    quant = w["kv_dtype"] != "bf16"
    lens = np.asarray(w["seq_lens"], np.int64)
    B = len(lens)
    kv = int(lens.sum()) * Hkv * (2 * row_bytes + (8 if quant else 0))
    pages = int(((lens + PAGE - 1) // PAGE).sum())
    return kv + 2 * (B * T * Hq * D * 2) + B * T * Hq * 4 + 4 * (pages + B)


def algorithmic_flops(w) -> int:
    """4*D flops per (visible key, query row): QK^T and PV multiply-adds."""
    lens = np.asarray(w["seq_lens"], np.int64)
    T, Hq, D = w["T"], w["Hq"], w["D"]
    visible = sum(int(L) - T + t + 1 for L in lens for t in range(T))
    return 4 * D * Hq * visible


def to_device(w, device="cuda", copies=1):
    """Device tensors of a workload (torch).  ``copies`` > 1 makes that many
    independent copies of the cache tensors (to rotate through, so that a
    timing loop does not re-read the cache from L2)."""
    dev = torch.device(device)

    def t(a):
        return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    q = torch.from_numpy(np.ascontiguousarray(w["q"]).view(np.int16)).to(dev).view(torch.bfloat16)
    kv_caches = []
    for i in range(max(1, copies)):
        if w["kv_dtype"] == "bf16":
            k = torch.from_numpy(w["k_pages"].view(np.int16)).to(dev).view(torch.bfloat16)
            v = torch.from_numpy(w["v_pages"].view(np.int16)).to(dev).view(torch.bfloat16)
        else:
            k, v = t(w["k_pages"]), t(w["v_pages"])
        kv_caches.append((k, v, t(w["k_scale"]), t(w["v_scale"])))
    B, T, Hq, D = w["q"].shape
    return {
        "q": q,
        "caches": kv_caches,
        "k_pages": kv_caches[0][0], "v_pages": kv_caches[0][1],
        "k_scale": kv_caches[0][2], "v_scale": kv_caches[0][3],
        "block_table": t(w["block_table"]),
        "seq_lens": t(w["seq_lens"]),
        "out": torch.zeros((B, T, Hq, D), dtype=torch.bfloat16, device=dev),
        "lse": torch.zeros((B, T, Hq), dtype=torch.float32, device=dev),
    }


def token_history(seed: int, length: int, vocab: int = 151_936, copy_frac: float = 0.3,
                  seg_range=(8, 64)) -> np.ndarray:
    """Synthetic token stream for lookup-augmented drafting: uniform tokens in
    [0, vocab), with about ``copy_frac`` of the stream made of segments copied
    verbatim from earlier in the stream (a long-context assistant quoting what
    it was given), lengths uniform in ``seg_range``.  int32 [length]."""
    rng = np.random.Generator(np.random.PCG64(seed))
    x = rng.integers(0, vocab, length, dtype=np.int64).astype(np.int32)
    pos = seg_range[1] * 2
    while pos < length:
        if rng.random() < copy_frac:
            n = int(rng.integers(seg_range[0], seg_range[1] + 1))
            n = min(n, length - pos)
            src = int(rng.integers(0, pos - n)) if pos - n > 0 else 0
            x[pos:pos + n] = x[src:src + n]
            pos += n
        else:
            pos += int(rng.integers(seg_range[0], seg_range[1] + 1))
    return x
