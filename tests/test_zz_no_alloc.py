"""The allocation-free entry point, verify_attn_noalloc.

It serves callers that cannot call cudaMalloc: a runtime whose memory pool
owns all device memory, a path that must not take the allocator's locks, a
process that fixes its device footprint at start-up.  It keeps its scratch in
the library's static device array.  These tests call it through the C ABI
twice in a row, with different shapes, and check each result against the
fp64 oracle and against the regular planned entry point under the parity
tolerance; they also check the page bound check with its flag word and the
rejection of a work list that cannot fit.  The file is named to run last, so
that a failure here leaves every other test already run."""
import ctypes

import numpy as np
import pytest

import oracle
from speculative_decoding_verify_causal_gb300 import workloads as wl

from parity import compare

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from speculative_decoding_verify_causal_gb300 import build
    build.build()


def _planned(va, w, d):
    plan = va.verify_attn_plan(w["seq_lens"], w["T"], w["Hq"], w["Hkv"], w["D"], w["kv_dtype"])
    try:
        va.verify_attn_with_plan(plan, d["q"], d["k_pages"], d["v_pages"], d["k_scale"], d["v_scale"],
                                 d["block_table"], d["seq_lens"], w["T"], d["out"], d["lse"])
        torch.cuda.synchronize()
    finally:
        plan.destroy()
    return d["out"].float().cpu().numpy(), d["lse"].cpu().numpy()


def _noalloc_rc(va, w, d, out, lse, num_pages=0):
    lib = va.library()
    P = ctypes.c_void_p
    lens = np.ascontiguousarray(w["seq_lens"], np.int32)
    ptr = lambda t: P(0) if t is None else P(t.data_ptr())  # noqa: E731
    return lib.verify_attn_noalloc(lens.ctypes.data_as(P), len(lens), w["T"], w["Hq"], w["Hkv"], w["D"],
                                   va.KV_DTYPE_CODES[w["kv_dtype"]], ptr(d["q"]), ptr(d["k_pages"]),
                                   ptr(d["v_pages"]), ptr(d["k_scale"]), ptr(d["v_scale"]),
                                   ptr(d["block_table"]), 0, num_pages, ptr(d["seq_lens"]), ptr(out), ptr(lse),
                                   P(torch.cuda.current_stream().cuda_stream))


def _noalloc_via_abi(va, w, d, out, lse, num_pages=0):
    rc = _noalloc_rc(va, w, d, out, lse, num_pages)
    assert rc == 0, va.verify_attn_status_string(rc)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), lse.cpu().numpy()


def test_noalloc_matches_oracle_and_planned_entry_on_two_calls_in_a_row():
    import speculative_decoding_verify_causal_gb300 as va
    cases = [
        wl.make_workload(301, [2500, 40, 777], 5, 24, 4, 256, "fp8_e4m3"),   # split + unsplit rows
        wl.make_workload(302, [25016], 16, 24, 4, 256, "int8"),             # long context, many splits
        wl.make_workload(303, [9001, 123], 1, 8, 4, 128, "int4"),           # two packed rows, 4-bit cache
    ]
    for i, w in enumerate(cases):
        d = wl.to_device(w)
        plan_out, plan_lse = _planned(va, w, d)
        out = torch.full_like(d["out"], float("nan"))
        lse = torch.full_like(d["lse"], float("nan"))
        got_out, got_lse = _noalloc_via_abi(va, w, d, out, lse)
        ref_out, ref_lse = oracle.verify_attn(w)
        compare(got_out, got_lse, ref_out, ref_lse, f"noalloc call {i + 1} vs oracle")
        compare(got_out, got_lse, plan_out, plan_lse, f"noalloc call {i + 1} vs planned entry")
        assert va.verify_attn_noalloc_flags() == 0


def test_noalloc_bad_page_is_skipped_and_flagged():
    """With the pool size given, a block-table entry past it is skipped and
    flagged.  The entry used lies inside the allocation (the pool is allocated
    larger than the size given), so the access is in bounds either way."""
    import speculative_decoding_verify_causal_gb300 as va
    w = wl.make_workload(95, [100], 2, 4, 1, 64, "int8", extra_pages=10)
    d = wl.to_device(w)
    pages_used = set(int(x) for x in w["block_table"][0, :7])
    spare = max(set(range(w["num_pages"])) - pages_used)  # allocated, not used by the sequence
    d["block_table"][0, 3] = spare
    out = torch.zeros_like(d["out"])
    lse = torch.zeros_like(d["lse"])
    got_out, _ = _noalloc_via_abi(va, w, d, out, lse, num_pages=spare)  # spare >= num_pages: flagged
    assert va.verify_attn_noalloc_flags() & 1
    assert va.verify_attn_noalloc_flags() == 0  # cleared by the read above
    assert np.isfinite(got_out).all()
    # the same call without the bound check reads the spare page and does not flag
    _noalloc_via_abi(va, w, d, out, lse, num_pages=0)
    assert va.verify_attn_noalloc_flags() == 0


def test_noalloc_rejects_work_lists_beyond_its_scratch():
    """8192 sequences x 9 kv heads = 73,728 work items even unsplit: more than
    the entry point can stage, so it returns VA_ERR_SCRATCH_TOO_SMALL before
    any CUDA call.  Every buffer passed is a real allocation of the size the
    arguments describe (zero-filled: page 0 everywhere), so the call would stay
    in bounds even if the check failed."""
    import speculative_decoding_verify_causal_gb300 as va
    lib = va.library()
    B, T, Hq, Hkv, D = 8192, 1, 9, 9, 64
    lens = np.full(B, 1, np.int32)
    dev = torch.device("cuda")
    q = torch.zeros((B, T, Hq, D), dtype=torch.bfloat16, device=dev)
    kp = torch.zeros((B, 16, Hkv, D), dtype=torch.bfloat16, device=dev)
    vp = torch.zeros_like(kp)
    bt = torch.zeros((B, 1), dtype=torch.int32, device=dev)
    sl = torch.ones(B, dtype=torch.int32, device=dev)
    out = torch.zeros_like(q)
    lse = torch.zeros((B, T, Hq), dtype=torch.float32, device=dev)
    P = ctypes.c_void_p
    rc = lib.verify_attn_noalloc(lens.ctypes.data_as(P), B, T, Hq, Hkv, D, 0, P(q.data_ptr()), P(kp.data_ptr()),
                                 P(vp.data_ptr()), P(0), P(0), P(bt.data_ptr()), 0, 0, P(sl.data_ptr()),
                                 P(out.data_ptr()), P(lse.data_ptr()), P(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    assert rc == -8, va.verify_attn_status_string(rc)
