"""The allocation-free entry point, verify_attn_noalloc, for callers that
cannot call cudaMalloc (a runtime whose pool owns all device memory, a path
that must not take allocator locks, a fixed device footprint).  It keeps its
scratch in the library's static device array; this test calls it through the
C ABI twice in a row, with different shapes, and checks each result against
the regular planned entry point under the parity tolerance.  The file is named
to run last, so that a failure here leaves every other test already run."""
import ctypes

import numpy as np
import pytest

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


def _noalloc_via_abi(va, w, d, out, lse):
    lib = va.library()
    P = ctypes.c_void_p
    lens = np.ascontiguousarray(w["seq_lens"], np.int32)
    ptr = lambda t: P(0) if t is None else P(t.data_ptr())  # noqa: E731
    rc = lib.verify_attn_noalloc(lens.ctypes.data_as(P), len(lens), w["T"], w["Hq"], w["Hkv"], w["D"],
                                 va.KV_DTYPE_CODES[w["kv_dtype"]], ptr(d["q"]), ptr(d["k_pages"]),
                                 ptr(d["v_pages"]), ptr(d["k_scale"]), ptr(d["v_scale"]),
                                 ptr(d["block_table"]), 0, ptr(d["seq_lens"]), ptr(out), ptr(lse),
                                 P(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, va.verify_attn_status_string(rc)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), lse.cpu().numpy()


def test_noalloc_matches_planned_entry_on_two_calls_in_a_row():
    import speculative_decoding_verify_causal_gb300 as va
    cases = [
        wl.make_workload(301, [2500, 40, 777], 5, 24, 4, 256, "fp8_e4m3"),   # split + unsplit rows
        wl.make_workload(302, [25016], 16, 24, 4, 256, "int8"),             # long context, many splits
    ]
    for i, w in enumerate(cases):
        d = wl.to_device(w)
        ref_out, ref_lse = _planned(va, w, d)
        out = torch.full_like(d["out"], float("nan"))
        lse = torch.full_like(d["lse"], float("nan"))
        got_out, got_lse = _noalloc_via_abi(va, w, d, out, lse)
        compare(got_out, got_lse, ref_out, ref_lse, f"noalloc call {i + 1}")


def test_noalloc_rejects_work_lists_beyond_its_scratch():
    import speculative_decoding_verify_causal_gb300 as va
    lib = va.library()
    # 4096 sequences x 8 kv heads x 4 row groups = 131072 work items even
    # unsplit: more than the entry point can stage, so it is rejected with
    # VA_ERR_SCRATCH_TOO_SMALL before anything is copied or launched (the
    # dummy pointers are never dereferenced)
    lens = np.full(4096, 64, np.int32)
    P = ctypes.c_void_p
    rc = lib.verify_attn_noalloc(lens.ctypes.data_as(P), len(lens), 64, 8, 8, 64, 0, *([P(1)] * 6), 0,
                                 P(1), P(1), P(0), P(0))
    assert rc == -8, va.verify_attn_status_string(rc)
