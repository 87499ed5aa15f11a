"""CPU oracle for verify attention (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` import this package.  The C source ``verify_attn_oracle.c`` is the
plain fp64 definition of the verify step's causal GQA attention over a paged,
quantised KV cache, ``kv_append_oracle.c`` the definition of the KV append
with quantise-on-write that precedes it and ``lookup_draft_oracle.c`` the
lookup-augmented drafter's history scan; this module compiles them with gcc and
marshals numpy arrays into them.  It shares no code with the CUDA library.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRCS = [os.path.join(_HERE, f) for f in ("verify_attn_oracle.c", "kv_append_oracle.c", "lookup_draft_oracle.c")]
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

KV_DTYPES = {"bf16": 0, "fp8_e4m3": 1, "int8": 2, "int4": 3, "int2": 4}


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/liboracle.so`` (gcc, OpenMP)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= max(os.path.getmtime(f) for f in _SRCS)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    # -ffp-contract=off: the append oracle's binary32 arithmetic must not be fused
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off", *_SRCS, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I = ctypes.c_int
        common = [P, P, P, P, P, P, I, P, I, I, I, I, I, I]
        lib.oracle_verify_attn.argtypes = common + [P, P, I]
        lib.oracle_verify_attn.restype = I
        lib.oracle_verify_attn_rows.argtypes = common + [P, I, P, P, I]
        lib.oracle_verify_attn_rows.restype = I
        lib.oracle_verify_attn_partial.argtypes = common + [I, I, I, I, I, P, P]
        lib.oracle_verify_attn_partial.restype = I
        lib.oracle_decode_e4m3.argtypes = [ctypes.c_uint8]
        lib.oracle_decode_e4m3.restype = ctypes.c_double
        lib.oracle_decode_packed.argtypes = [P, ctypes.c_size_t, I]
        lib.oracle_decode_packed.restype = ctypes.c_double
        lib.oracle_decode_bf16.argtypes = [ctypes.c_uint16]
        lib.oracle_decode_bf16.restype = ctypes.c_double
        lib.oracle_max_threads.argtypes = [I]
        lib.oracle_max_threads.restype = I
        lib.oracle_kv_append.argtypes = [P, P, I, I, I, I, I, P, P, P, P, P, I, P, I, P]
        lib.oracle_kv_append.restype = I
        lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_int8_encode.argtypes = [ctypes.c_float]
        lib.oracle_int8_encode.restype = ctypes.c_int8
        lib.oracle_lookup_draft.argtypes = [P, I, I, I, I, P, P, P]
        lib.oracle_lookup_draft.restype = I
        _lib = lib
        return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def _common(w):
    """Argument tuple shared by every entry point, from a workload dict."""
    dt = w["kv_dtype"]
    raw = {"bf16": np.uint16, "fp8_e4m3": np.uint8, "int8": np.int8, "int4": np.uint8, "int2": np.uint8}[dt]
    q = _c(w["q"], np.uint16)
    k = _c(w["k_pages"], raw)
    v = _c(w["v_pages"], raw)
    ks = _c(w.get("k_scale"), np.float32)
    vs = _c(w.get("v_scale"), np.float32)
    bt = _c(w["block_table"], np.int32)
    sl = _c(w["seq_lens"], np.int32)
    B, T, Hq, D = q.shape
    Hkv = k.shape[2]
    if dt in ("int4", "int2"):
        assert k.shape[3] * 8 // {"int4": 4, "int2": 2}[dt] == D, "packed rows must hold head_dim codes"
    keep = (q, k, v, ks, vs, bt, sl)
    args = [_ptr(q), _ptr(k), _ptr(v), _ptr(ks), _ptr(vs), _ptr(bt), bt.shape[1],
            _ptr(sl), B, T, Hq, Hkv, D, KV_DTYPES[dt]]
    return keep, args, (B, T, Hq, D)


def verify_attn(w, nthreads: int = 0):
    """Full oracle output: (out float64 [B,T,Hq,D], lse float64 [B,T,Hq])."""
    lib = _load()
    keep, args, (B, T, Hq, D) = _common(w)
    out = np.empty((B, T, Hq, D), np.float64)
    lse = np.empty((B, T, Hq), np.float64)
    rc = lib.oracle_verify_attn(*args, _ptr(out), _ptr(lse), nthreads)
    if rc != 0:
        raise ValueError("oracle_verify_attn rejected its arguments")
    del keep
    return out, lse


def verify_attn_rows(w, rows, nthreads: int = 0):
    """Oracle output for selected (b, t, h) triples: (out [n, D], lse [n])."""
    lib = _load()
    keep, args, (B, T, Hq, D) = _common(w)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1, 3))
    n = rows.shape[0]
    out = np.empty((n, D), np.float64)
    lse = np.empty((n,), np.float64)
    rc = lib.oracle_verify_attn_rows(*args, _ptr(rows), n, _ptr(out), _ptr(lse), nthreads)
    if rc != 0:
        raise ValueError("oracle_verify_attn_rows rejected its arguments")
    del keep
    return out, lse


def verify_attn_partial(w, b, t, h, key_begin, key_end):
    """One split's normalised partial (out [D], lse) over keys [key_begin, key_end)."""
    lib = _load()
    keep, args, (B, T, Hq, D) = _common(w)
    out = np.empty((D,), np.float64)
    lse = np.empty((1,), np.float64)
    rc = lib.oracle_verify_attn_partial(*args, b, t, h, key_begin, key_end, _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError("oracle_verify_attn_partial rejected its arguments")
    del keep
    return out, float(lse[0])


def decode_e4m3(code: int) -> float:
    return _load().oracle_decode_e4m3(code)


def decode_packed(data, idx: int, bits: int) -> float:
    """Element idx of a packed byte array of `bits`-bit codes (4 or 2)."""
    a = np.ascontiguousarray(data, np.uint8)
    return _load().oracle_decode_packed(_ptr(a), int(idx), int(bits))


def decode_bf16(bits: int) -> float:
    return _load().oracle_decode_bf16(bits)


def max_threads(nthreads: int = 0) -> int:
    return _load().oracle_max_threads(nthreads)


def e4m3_encode(y: float) -> int:
    """Round-to-nearest-even e4m3 code of a binary32 value (|y| <= 448)."""
    return int(_load().oracle_e4m3_encode(float(y)))


def int8_encode(y: float) -> int:
    return int(_load().oracle_int8_encode(float(y)))


def kv_append(k_new, v_new, k_pages, v_pages, k_scale, v_scale, block_table, seq_lens, kv_dtype,
              num_pages: int = 0):
    """Append new K/V rows (bf16 bits, [B, T, Hkv, D]) into copies of the given
    cache arrays; returns (k_pages, v_pages, k_scale, v_scale, skipped)."""
    lib = _load()
    k_new = _c(k_new, np.uint16)
    v_new = _c(v_new, np.uint16)
    B, T, Hkv, D = k_new.shape
    kp = np.array(k_pages, copy=True, order="C")
    vp = np.array(v_pages, copy=True, order="C")
    ks = None if k_scale is None else np.array(k_scale, dtype=np.float32, copy=True, order="C")
    vs = None if v_scale is None else np.array(v_scale, dtype=np.float32, copy=True, order="C")
    bt = _c(block_table, np.int32)
    sl = _c(seq_lens, np.int32)
    skipped = ctypes.c_int(0)
    rc = lib.oracle_kv_append(_ptr(k_new), _ptr(v_new), B, T, Hkv, D, KV_DTYPES[kv_dtype], _ptr(kp), _ptr(vp),
                              _ptr(ks), _ptr(vs), _ptr(bt), bt.shape[1], _ptr(sl), int(num_pages),
                              ctypes.byref(skipped))
    if rc != 0:
        raise ValueError("oracle_kv_append rejected its arguments")
    return kp, vp, ks, vs, skipped.value


def lookup_draft(history, min_match: int, max_match: int, num_draft: int):
    """Lookup-augmented draft of one token history (int32 [L]): returns
    (draft [num_draft] with -1 past the proposal, draft_len, match_end, match_len)."""
    lib = _load()
    x = _c(history, np.int32)
    draft = np.empty(num_draft, np.int32)
    e = ctypes.c_int32(0)
    n = ctypes.c_int32(0)
    length = lib.oracle_lookup_draft(_ptr(x), int(x.size), int(min_match), int(max_match), int(num_draft),
                                     _ptr(draft), ctypes.byref(e), ctypes.byref(n))
    return draft, int(length), int(e.value), int(n.value)
