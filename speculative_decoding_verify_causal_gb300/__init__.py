"""GB300-native speculative-decoding verify attention.

Thin ctypes binding over ``libverify_attn.so`` (built in-tree by
``speculative_decoding_verify_causal_gb300.build``).  The functions carry the
C ABI's names and do argument marshalling only: every step of the attention
runs in the library's CUDA kernels.  PyTorch supplies device memory and
streams.  There is no CPU fallback: importing this package without the built
library raises.

Layouts (see ``include/verify_attn.h``):
  q bf16 [B, T, Hq, D]; k_pages / v_pages [num_pages, 16, Hkv, D] of
  bf16 / fp8-e4m3 (uint8 storage) / int8; k_scale / v_scale fp32
  [num_pages, 16, Hkv]; block_table int32 [B, stride]; seq_lens int32 [B];
  out bf16 [B, T, Hq, D]; lse fp32 [B, T, Hq].
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libverify_attn.so")

VA_BF16, VA_FP8_E4M3, VA_INT8, VA_INT4, VA_INT2 = 0, 1, 2, 3, 4
KV_DTYPE_CODES = {"bf16": VA_BF16, "fp8_e4m3": VA_FP8_E4M3, "int8": VA_INT8, "int4": VA_INT4, "int2": VA_INT2}
VA_PATH_AUTO, VA_PATH_WARP, VA_PATH_MMA = 0, 1, 2
PATH_CODES = {"auto": VA_PATH_AUTO, "warp": VA_PATH_WARP, "mma": VA_PATH_MMA}
PAGE_SIZE = 16

STATUS_NAMES = {
    0: "VA_OK", -1: "VA_ERR_INVALID_ARGUMENT", -2: "VA_ERR_UNSUPPORTED",
    -3: "VA_ERR_PLAN_MISMATCH", -4: "VA_ERR_NO_PLAN", -5: "VA_ERR_CUDA",
    -6: "VA_ERR_OUT_OF_MEMORY", -7: "VA_ERR_NO_DEVICE", -8: "VA_ERR_SCRATCH_TOO_SMALL",
}


class VerifyAttnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        msg = f"{what}: {STATUS_NAMES.get(status, status)} ({verify_attn_status_string(status)})"
        if status == -5:
            lib = _load()
            msg += f" [cuda error {lib.verify_attn_last_cuda_error()}: " \
                   f"{lib.verify_attn_last_cuda_error_string().decode()}]"
        super().__init__(msg)


class _Options(ctypes.Structure):
    _fields_ = [("block_table_stride", ctypes.c_int), ("tokens_per_split", ctypes.c_int),
                ("path", ctypes.c_int), ("num_pages", ctypes.c_int)]


class PlanInfo(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "num_seqs", "T", "num_q_heads", "num_kv_heads", "head_dim", "kv_dtype", "path",
        "rows_per_group", "num_row_groups", "tokens_per_split", "num_items",
        "num_split_groups", "max_splits", "num_sms")] + [("workspace_bytes", ctypes.c_longlong)]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


_lib = None
_lib_lock = threading.Lock()


def _load():
    global _lib
    with _lib_lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                f"{LIB_PATH} is not built: run `python -m speculative_decoding_verify_causal_gb300.build` "
                "(the package has no CPU fallback)")
        lib = ctypes.CDLL(LIB_PATH)
        P, I = ctypes.c_void_p, ctypes.c_int
        lib.verify_attn_plan.argtypes = [P, I, I, I, I, I, I, I, ctypes.POINTER(P)]
        lib.verify_attn_plan_ex.argtypes = [P, I, I, I, I, I, I, I, ctypes.POINTER(_Options), ctypes.POINTER(P)]
        lib.verify_attn.argtypes = [P] * 7 + [I, P, P, P]
        lib.verify_attn_with_plan.argtypes = [P] + [P] * 7 + [I, P, P, P]
        lib.verify_attn_plan_destroy.argtypes = [P]
        lib.verify_attn_plan_destroy.restype = None
        lib.verify_attn_status_string.argtypes = [I]
        lib.verify_attn_status_string.restype = ctypes.c_char_p
        lib.verify_attn_plan_get_info.argtypes = [P, ctypes.POINTER(PlanInfo)]
        lib.verify_attn_plan_describe.argtypes = [P, I, I, I, I, I, I, I, ctypes.POINTER(_Options),
                                                  ctypes.POINTER(PlanInfo), P, I]
        lib.verify_attn_plan_device_flags.argtypes = [P, I, ctypes.POINTER(I), P]
        lib.verify_attn_plan_set_events.argtypes = [P, P, P]
        lib.verify_attn_plan_set_events.restype = I
        lib.verify_attn_last_cuda_error.argtypes = []
        lib.verify_attn_last_cuda_error.restype = I
        lib.verify_attn_last_cuda_error_string.argtypes = []
        lib.verify_attn_last_cuda_error_string.restype = ctypes.c_char_p
        lib.verify_attn_noalloc.argtypes = [P, I, I, I, I, I, I] + [P] * 6 + [I, I, P, P, P, P]
        lib.verify_attn_noalloc_flags.argtypes = [I, ctypes.POINTER(I), P]
        lib.verify_attn_noalloc_flags.restype = I
        lib.verify_attn_noalloc.restype = I
        lib.verify_attn_kv_append.argtypes = [P, P, I, I, I, I, I, P, P, P, P, P, I, P, I, P, P]
        lib.verify_attn_kv_append.restype = I
        lib.verify_attn_lookup_draft.argtypes = [P, I, P, I, I, I, I, P, P, P, P, P]
        lib.verify_attn_lookup_draft.restype = I
        lib.verify_attn_accept_workspace_bytes.argtypes = [I, I]
        lib.verify_attn_accept_workspace_bytes.restype = ctypes.c_size_t
        lib.verify_attn_accept.argtypes = [P, P, P, P, I, I, I, ctypes.c_uint64, P, P, P, P]
        lib.verify_attn_accept.restype = I
        lib.verify_attn_validate_host.argtypes = [P, I, I, P, I, I, ctypes.POINTER(I), ctypes.POINTER(I)]
        lib.verify_attn_validate_host.restype = I
        for f in ("verify_attn_plan", "verify_attn_plan_ex", "verify_attn", "verify_attn_with_plan",
                  "verify_attn_plan_get_info", "verify_attn_plan_describe", "verify_attn_plan_device_flags"):
            getattr(lib, f).restype = I
        _lib = lib
        return lib


def library():
    """The loaded ctypes library (raises if it is not built)."""
    return _load()


def verify_attn_status_string(status: int) -> str:
    return _load().verify_attn_status_string(int(status)).decode()


def _check(rc, what):
    if rc != 0:
        raise VerifyAttnError(rc, what)


def _dtype_code(kv_dtype):
    return KV_DTYPE_CODES[kv_dtype] if isinstance(kv_dtype, str) else int(kv_dtype)


def _options(block_table_stride=0, tokens_per_split=0, path="auto", num_pages=0):
    return _Options(int(block_table_stride), int(tokens_per_split),
                    PATH_CODES[path] if isinstance(path, str) else int(path), int(num_pages))


def _host_lens(seq_lens):
    try:
        import torch
        if isinstance(seq_lens, torch.Tensor):
            seq_lens = seq_lens.detach().cpu().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(seq_lens, dtype=np.int32).reshape(-1))


class Plan:
    """Owning handle of a ``va_plan`` (freed on ``destroy()`` or collection)."""

    def __init__(self, handle, seq_lens, T, kv_dtype):
        self._h = ctypes.c_void_p(handle)
        self.seq_lens = seq_lens
        self.T = T
        self.kv_dtype = kv_dtype

    @property
    def handle(self):
        return self._h

    def info(self) -> dict:
        return verify_attn_plan_get_info(self)

    def destroy(self):
        if self._h and self._h.value:
            _load().verify_attn_plan_destroy(self._h)
            self._h = ctypes.c_void_p(0)

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass


def verify_attn_plan(seq_lens, T, num_q_heads, num_kv_heads, head_dim, kv_dtype, num_sms=0,
                     **options) -> Plan:
    """Plan one batch shape from the host ``seq_lens`` (lengths include the T
    verify tokens).  Keyword options: block_table_stride, tokens_per_split,
    path ("auto" | "warp" | "mma"), num_pages (enables device bound checks).
    The new plan also becomes this thread's current plan for ``verify_attn``."""
    lib = _load()
    lens = _host_lens(seq_lens)
    out = ctypes.c_void_p()
    opts = _options(**options)
    rc = lib.verify_attn_plan_ex(lens.ctypes.data_as(ctypes.c_void_p), len(lens), int(T), int(num_q_heads),
                                 int(num_kv_heads), int(head_dim), _dtype_code(kv_dtype), int(num_sms),
                                 ctypes.byref(opts), ctypes.byref(out))
    _check(rc, "verify_attn_plan")
    return Plan(out.value, lens, int(T), _dtype_code(kv_dtype))


def verify_attn_plan_destroy(plan: Plan):
    plan.destroy()


def verify_attn_validate_host(seq_lens, T, block_table, num_pages):
    """Host check of the paging inputs (no GPU needed).  Returns None when
    they are valid, else (sequence, block index or -1) of the first fault."""
    lens = _host_lens(seq_lens)
    try:
        import torch
        if isinstance(block_table, torch.Tensor):
            block_table = block_table.detach().cpu().numpy()
    except ImportError:  # pragma: no cover
        pass
    bt = np.ascontiguousarray(np.asarray(block_table, dtype=np.int32))
    if bt.ndim != 2 or bt.shape[0] != len(lens):
        raise ValueError("block_table must be [num_seqs, stride]")
    bad_seq, bad_block = ctypes.c_int(-1), ctypes.c_int(-1)
    rc = _load().verify_attn_validate_host(lens.ctypes.data_as(ctypes.c_void_p), len(lens), int(T),
                                           bt.ctypes.data_as(ctypes.c_void_p), bt.shape[1], int(num_pages),
                                           ctypes.byref(bad_seq), ctypes.byref(bad_block))
    if rc == 0:
        return None
    if bad_seq.value < 0:
        _check(rc, "verify_attn_validate_host")
    return bad_seq.value, bad_block.value


def verify_attn_plan_get_info(plan: Plan) -> dict:
    info = PlanInfo()
    _check(_load().verify_attn_plan_get_info(plan.handle, ctypes.byref(info)), "verify_attn_plan_get_info")
    return info.as_dict()


def verify_attn_plan_describe(seq_lens, T, num_q_heads, num_kv_heads, head_dim, kv_dtype, num_sms,
                              max_items=None, **options):
    """Host-only planning (no GPU needed): (info dict, items int32 [n, 5])
    with items = (seq, kv_head, row_group, key_begin, key_end)."""
    lib = _load()
    lens = _host_lens(seq_lens)
    opts = _options(**options)
    info = PlanInfo()
    rc = lib.verify_attn_plan_describe(lens.ctypes.data_as(ctypes.c_void_p), len(lens), int(T),
                                       int(num_q_heads), int(num_kv_heads), int(head_dim),
                                       _dtype_code(kv_dtype), int(num_sms), ctypes.byref(opts),
                                       ctypes.byref(info), None, 0)
    _check(rc, "verify_attn_plan_describe")
    n = info.num_items if max_items is None else min(int(max_items), info.num_items)
    items = np.zeros((max(n, 1), 5), np.int32)
    rc = lib.verify_attn_plan_describe(lens.ctypes.data_as(ctypes.c_void_p), len(lens), int(T),
                                       int(num_q_heads), int(num_kv_heads), int(head_dim),
                                       _dtype_code(kv_dtype), int(num_sms), ctypes.byref(opts),
                                       ctypes.byref(info), items.ctypes.data_as(ctypes.c_void_p), n)
    _check(rc, "verify_attn_plan_describe")
    return info.as_dict(), items[:n]


def _dev_ptr(t, name, dtypes, allow_none=False):
    import torch
    if t is None:
        if allow_none:
            return None
        raise ValueError(f"{name} is required")
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype not in dtypes:
        raise ValueError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _kv_dtypes(code):
    import torch
    if code == VA_BF16:
        return (torch.bfloat16, torch.int16, torch.uint16) if hasattr(torch, "uint16") else (torch.bfloat16, torch.int16)
    if code == VA_FP8_E4M3:
        return (torch.uint8, torch.float8_e4m3fn)
    if code in (VA_INT4, VA_INT2):  # packed bytes
        return (torch.uint8, torch.int8)
    return (torch.int8,)


def _marshal(kv_code, q, k_pages, v_pages, k_scale, v_scale, block_table, seq_lens, out, lse, stream):
    import torch
    q16 = (torch.bfloat16, torch.int16)
    kvd = _kv_dtypes(kv_code)
    args = [
        _dev_ptr(q, "q", q16),
        _dev_ptr(k_pages, "k_pages", kvd),
        _dev_ptr(v_pages, "v_pages", kvd),
        _dev_ptr(k_scale, "k_scale", (torch.float32,), allow_none=kv_code == VA_BF16),
        _dev_ptr(v_scale, "v_scale", (torch.float32,), allow_none=kv_code == VA_BF16),
        _dev_ptr(block_table, "block_table", (torch.int32,)),
        _dev_ptr(seq_lens, "seq_lens", (torch.int32,)),
    ]
    tail = [_dev_ptr(out, "out", q16), _dev_ptr(lse, "lse", (torch.float32,), allow_none=True)]
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    s = ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))
    return args, tail, s


def verify_attn_with_plan(plan: Plan, q, k_pages, v_pages, k_scale, v_scale, block_table, seq_lens, T,
                          out, lse=None, stream=None):
    """Enqueue verify attention with an explicit plan on ``stream`` (default:
    torch's current stream).  Writes ``out`` (and ``lse`` if given)."""
    args, tail, s = _marshal(plan.kv_dtype, q, k_pages, v_pages, k_scale, v_scale, block_table,
                             seq_lens, out, lse, stream)
    _check(_load().verify_attn_with_plan(plan.handle, *args, int(T), *tail, s), "verify_attn_with_plan")


def verify_attn(q, k_pages, v_pages, k_scale, v_scale, block_table, seq_lens, T, out, lse=None,
                stream=None, kv_dtype=None):
    """Enqueue verify attention with this thread's current plan.  ``kv_dtype``
    only selects the accepted tensor dtypes for marshalling (inferred from
    ``k_pages`` when omitted: a byte cache whose rows are D / 2 or D / 4 bytes
    long is the 4-bit or 2-bit one)."""
    import torch
    if kv_dtype is None:
        kv_code = {torch.int8: VA_INT8, torch.uint8: VA_FP8_E4M3,
                   torch.float8_e4m3fn: VA_FP8_E4M3}.get(k_pages.dtype, VA_BF16)
        if kv_code != VA_BF16 and k_pages.dim() == 4:
            D = q.shape[-1]
            kv_code = {D // 2: VA_INT4, D // 4: VA_INT2}.get(k_pages.shape[-1], kv_code)
    else:
        kv_code = _dtype_code(kv_dtype)
    args, tail, s = _marshal(kv_code, q, k_pages, v_pages, k_scale, v_scale, block_table, seq_lens,
                             out, lse, stream)
    _check(_load().verify_attn(*args, int(T), *tail, s), "verify_attn")


def verify_attn_plan_device_flags(plan: Plan, clear=True, stream=None) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    flags = ctypes.c_int(0)
    _check(_load().verify_attn_plan_device_flags(plan.handle, int(bool(clear)), ctypes.byref(flags),
                                                 ctypes.c_void_p(stream.cuda_stream)),
           "verify_attn_plan_device_flags")
    return flags.value


def verify_attn_plan_set_events(plan: Plan, ev_before=None, ev_after=None):
    """Record two torch.cuda.Event objects around the partial-attention
    kernel of every later call with ``plan`` (None, None stops)."""
    b = ctypes.c_void_p(ev_before.cuda_event) if ev_before is not None else None
    a = ctypes.c_void_p(ev_after.cuda_event) if ev_after is not None else None
    _check(_load().verify_attn_plan_set_events(plan.handle, b, a), "verify_attn_plan_set_events")


def verify_attn_noalloc(seq_lens_host, T, num_q_heads, num_kv_heads, head_dim, kv_dtype, q, k_pages,
                        v_pages, k_scale, v_scale, block_table, seq_lens, out, lse=None,
                        block_table_stride=0, num_pages=0, stream=None):
    """Verify attention that allocates no device memory: plans from the host
    ``seq_lens_host`` on every call and keeps its scratch in the library's
    static device array (see ``include/verify_attn.h``).  For callers that
    cannot call cudaMalloc.  Calls share that array, so order them on one
    stream; not for CUDA-graph capture.  ``num_pages`` > 0 checks every
    block-table entry (bad ones are skipped and flagged, see
    ``verify_attn_noalloc_flags``)."""
    lens = _host_lens(seq_lens_host)
    code = _dtype_code(kv_dtype)
    args, tail, s = _marshal(code, q, k_pages, v_pages, k_scale, v_scale, block_table, seq_lens, out, lse,
                             stream)
    rc = _load().verify_attn_noalloc(lens.ctypes.data_as(ctypes.c_void_p), len(lens), int(T), int(num_q_heads),
                                     int(num_kv_heads), int(head_dim), code, *args[:6],
                                     int(block_table_stride), int(num_pages), args[6], *tail, s)
    _check(rc, "verify_attn_noalloc")


def verify_attn_noalloc_flags(clear=True, stream=None):
    """Flag word of the last verify_attn_noalloc call on the current device
    (same bits as verify_attn_plan_device_flags); clears it by default."""
    import torch
    stream = stream or torch.cuda.current_stream()
    flags = ctypes.c_int(0)
    _check(_load().verify_attn_noalloc_flags(int(bool(clear)), ctypes.byref(flags),
                                             ctypes.c_void_p(stream.cuda_stream)), "verify_attn_noalloc_flags")
    return flags.value


def verify_attn_kv_append(k_new, v_new, k_pages, v_pages, k_scale, v_scale, block_table, seq_lens, T,
                          kv_dtype, num_pages=0, flags=None, stream=None):
    """KV append with quantise-on-write: store the T new tokens' K and V rows
    (bf16 ``[B, T, Hkv, D]``) at positions ``seq_lens[b] - T + t`` of the paged
    cache, quantised per (token, kv head) for fp8 / int8 caches (definition in
    ``include/verify_attn.h``).  ``flags`` is an optional int32 device tensor
    into which bit 0 is ORed for a skipped row."""
    import torch
    code = _dtype_code(kv_dtype)
    B, T_, Hkv, D = k_new.shape
    if int(T) != T_ or tuple(v_new.shape) != tuple(k_new.shape):
        raise ValueError("k_new and v_new must both be [B, T, Hkv, D] with the given T")
    q16 = (torch.bfloat16, torch.int16)
    kvd = _kv_dtypes(code)
    ptrs = [_dev_ptr(k_new, "k_new", q16), _dev_ptr(v_new, "v_new", q16)]
    cache = [_dev_ptr(k_pages, "k_pages", kvd), _dev_ptr(v_pages, "v_pages", kvd),
             _dev_ptr(k_scale, "k_scale", (torch.float32,), allow_none=code == VA_BF16),
             _dev_ptr(v_scale, "v_scale", (torch.float32,), allow_none=code == VA_BF16)]
    bt = _dev_ptr(block_table, "block_table", (torch.int32,))
    sl = _dev_ptr(seq_lens, "seq_lens", (torch.int32,))
    fl = _dev_ptr(flags, "flags", (torch.int32,), allow_none=True)
    if stream is None:
        stream = torch.cuda.current_stream(k_new.device)
    st = ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))
    rc = _load().verify_attn_kv_append(*ptrs, int(B), int(T), int(Hkv), int(D), code, *cache, bt,
                                       int(block_table.shape[1]), sl, int(num_pages), fl, st)
    _check(rc, "verify_attn_kv_append")


def verify_attn_lookup_draft(tokens, lens, num_draft, min_match=6, max_match=12, match_end=None,
                            match_len=None, stream=None):
    """Lookup-augmented drafting over token histories ``tokens`` (int32 CUDA
    tensor ``[num_seqs, stride]``, the first ``lens[b]`` entries valid): the
    most recent earlier occurrence of each history's last tokens (longest
    match first, ``min_match``..``max_match``) and up to ``num_draft`` tokens
    that followed it.  Returns (draft int32 ``[num_seqs, num_draft]``, -1 past
    the proposal, draft_len int32 ``[num_seqs]``); ``match_end`` /
    ``match_len`` (int32 ``[num_seqs]``) are filled when given."""
    import torch
    if tokens.dim() != 2:
        raise ValueError("tokens must be [num_seqs, stride]")
    B, stride = tokens.shape
    i32 = (torch.int32,)
    tp = _dev_ptr(tokens, "tokens", i32)
    lp = _dev_ptr(lens, "lens", i32)
    draft = torch.empty((B, int(num_draft)), dtype=torch.int32, device=tokens.device)
    dlen = torch.empty((B,), dtype=torch.int32, device=tokens.device)
    me = _dev_ptr(match_end, "match_end", i32, allow_none=True)
    ml = _dev_ptr(match_len, "match_len", i32, allow_none=True)
    if stream is None:
        stream = torch.cuda.current_stream(tokens.device)
    st = ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))
    rc = _load().verify_attn_lookup_draft(tp, int(stride), lp, int(B), int(min_match), int(max_match),
                                          int(num_draft), ctypes.c_void_p(draft.data_ptr()),
                                          ctypes.c_void_p(dlen.data_ptr()), me, ml, st)
    _check(rc, "verify_attn_lookup_draft")
    return draft, dlen


def verify_attn_accept(target_logits, draft_tokens, temperature, seed, draft_logits=None, stream=None):
    """Speculative acceptance (rejection sampler) after the verify pass:
    ``target_logits`` fp32 ``[B, T+1, V]``, ``draft_tokens`` int32 ``[B, T]``,
    ``temperature`` fp32 ``[B]`` (<= 0: greedy), ``draft_logits`` fp32
    ``[B, T, V]`` or None (a point-mass proposal, as for lookup drafts), all
    CUDA tensors; ``seed`` picks the Philox stream.  Returns (out_tokens int32
    ``[B, T+1]`` with -1 after the emitted token, num_accepted int32 ``[B]``)."""
    import torch
    if target_logits.dim() != 3 or draft_tokens.dim() != 2:
        raise ValueError("target_logits must be [B, T+1, V] and draft_tokens [B, T]")
    B, T1, V = target_logits.shape
    T = T1 - 1
    if tuple(draft_tokens.shape) != (B, T):
        raise ValueError("draft_tokens must be [B, T]")
    if draft_logits is not None and tuple(draft_logits.shape) != (B, T, V):
        raise ValueError("draft_logits must be [B, T, V]")
    f32, i32 = (torch.float32,), (torch.int32,)
    zp = _dev_ptr(target_logits, "target_logits", f32)
    wp = _dev_ptr(draft_logits, "draft_logits", f32, allow_none=True)
    dp = _dev_ptr(draft_tokens, "draft_tokens", i32)
    tp = _dev_ptr(temperature, "temperature", f32)
    lib = _load()
    ws = torch.empty(max(16, int(lib.verify_attn_accept_workspace_bytes(int(B), int(T)))), dtype=torch.uint8,
                     device=target_logits.device)
    out = torch.empty((B, T1), dtype=torch.int32, device=target_logits.device)
    nacc = torch.empty((B,), dtype=torch.int32, device=target_logits.device)
    if stream is None:
        stream = torch.cuda.current_stream(target_logits.device)
    st = ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))
    rc = lib.verify_attn_accept(zp, wp, dp, tp, int(B), int(T), int(V), int(seed) & 0xFFFFFFFFFFFFFFFF,
                                ctypes.c_void_p(ws.data_ptr()), ctypes.c_void_p(out.data_ptr()),
                                ctypes.c_void_p(nacc.data_ptr()), st)
    _check(rc, "verify_attn_accept")
    return out, nacc


__all__ = [
    "verify_attn_accept",
    "verify_attn_lookup_draft",
    "verify_attn_kv_append",
    "verify_attn_noalloc",
    "verify_attn_noalloc_flags",
    "verify_attn_plan_set_events",
    "verify_attn_plan", "verify_attn", "verify_attn_with_plan", "verify_attn_plan_destroy",
    "verify_attn_status_string", "verify_attn_plan_get_info", "verify_attn_plan_describe",
    "verify_attn_plan_device_flags", "verify_attn_validate_host", "Plan", "VerifyAttnError", "library",
    "LIB_PATH",
]
