"""Shared parity helpers: run the CUDA path through the C ABI and compare it
with the fp64 oracle under the stated tolerance.

Tolerance (bf16 output, unit-scale inputs): per element
|gpu - ref| <= max(1e-2, one bf16 ulp of ref) -- half an ulp of bf16 rounding
alone exceeds 1e-2 once |ref| >= 4 --, mean |gpu - ref| <= 1e-3, and
|lse_gpu - lse_ref| <= 1e-4 * |lse_ref| + 1e-6.

For value rows drawn at another scale (standard deviation v_std instead of
1) the output scales with them, so the two absolute bounds scale too:
max(1e-2 * v_std, one bf16 ulp of ref) per element and 1e-3 * v_std for the
mean; the log-sum-exp bound is already relative.  The mean bound never goes
below half the mean bf16 ulp of the reference: rounding the exact result to
bf16 alone costs a quarter ulp on average, which at |out| ~ 30 (one-hot
attention over values of scale 30) already equals 1e-3 * v_std.  At unit
scale that floor is about 1e-4 and changes nothing."""
import math

import numpy as np

MAX_ABS = 1e-2
MEAN_ABS = 1e-3
LSE_REL = 1e-4
LSE_ABS = 1e-6


def bf16_ulp(x):
    ax = np.abs(np.asarray(x, np.float64))
    e = np.floor(np.log2(np.maximum(ax, 2.0 ** -126)))
    return np.exp2(e - 7)


def compare(out_gpu, lse_gpu, out_ref, lse_ref, what="", v_std=1.0):
    """Raise AssertionError with a summary if the tolerance is broken.
    Returns a dict of the error statistics; ``ulp_allowance_used`` counts the
    elements above the absolute bound that only the one-ulp allowance let
    through."""
    o = np.asarray(out_gpu, np.float64)
    r = np.asarray(out_ref, np.float64)
    err = np.abs(o - r)
    max_abs = MAX_ABS * v_std
    allow = np.maximum(max_abs, bf16_ulp(r))
    bad = err > allow
    lerr = np.abs(np.asarray(lse_gpu, np.float64) - np.asarray(lse_ref, np.float64))
    lallow = LSE_REL * np.abs(lse_ref) + LSE_ABS
    lbad = ~(lerr <= lallow)
    stats = {
        "max_abs": float(err.max()) if err.size else 0.0,
        "mean_abs": float(err.mean()) if err.size else 0.0,
        "ulp_allowance_used": int(((err > max_abs) & ~bad).sum()),
        "elements": int(err.size),
        "mean_half_ulp": float(0.5 * bf16_ulp(r).mean()) if err.size else 0.0,
        "lse_max_rel": float((lerr / np.maximum(np.abs(lse_ref), 1e-30)).max()) if lerr.size else 0.0,
        "n_bad": int(bad.sum()),
        "n_lse_bad": int(lbad.sum()),
    }
    msg = f"{what}: {stats}"
    assert not np.isnan(o).any(), f"{what}: NaN in output"
    assert stats["n_bad"] == 0, msg
    assert stats["mean_abs"] <= max(MEAN_ABS * v_std, stats["mean_half_ulp"]), msg
    assert stats["n_lse_bad"] == 0, msg
    return stats


# bits of the plan's device flag word (verify_attn_plan_device_flags)
FLAG_NAMES = {1: "bad block-table entry skipped", 2: "device seq_lens differs from the plan",
              4: "a pipeline wait timed out"}


def flag_names(flags):
    return [n for b, n in FLAG_NAMES.items() if flags & b] + ([f"unknown bits {flags & ~7:#x}"] if flags & ~7 else [])


def run_gpu(w, plan_opts=None, dev=None, stream=None):
    """Plan + one verify call through the C ABI; returns (out f32 numpy, lse numpy, plan info)."""
    import torch
    import speculative_decoding_verify_causal_gb300 as va
    from speculative_decoding_verify_causal_gb300 import workloads as wl
    d = wl.to_device(w) if dev is None else dev
    plan = va.verify_attn_plan(w["seq_lens"], w["T"], w["Hq"], w["Hkv"], w["D"], w["kv_dtype"],
                               **(plan_opts or {}))
    try:
        va.verify_attn_with_plan(plan, d["q"], d["k_pages"], d["v_pages"], d["k_scale"], d["v_scale"],
                                 d["block_table"], d["seq_lens"], w["T"], d["out"], d["lse"], stream=stream)
        torch.cuda.synchronize()
        info = plan.info()
        flags = va.verify_attn_plan_device_flags(plan)
    finally:
        plan.destroy()
    assert flags == 0, f"device flags {flags}: {flag_names(flags)}"
    return d["out"].float().cpu().numpy(), d["lse"].cpu().numpy(), info
