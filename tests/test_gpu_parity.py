"""GPU parity: the CUDA path (called through the C ABI) against the fp64 CPU
oracle, element by element, on the same seeded inputs: the full output of all
five named configurations (the large ones in the plan the benchmark uses),
shape sweeps, split and page-permutation invariance, non-unit K/V scales, and
sampled rows at long contexts of the other head widths and cache types."""
import ctypes

import numpy as np
import pytest

import oracle
from speculative_decoding_verify_causal_gb300 import workloads as wl

from parity import compare, run_gpu

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from speculative_decoding_verify_causal_gb300 import build
    build.build()


_cache = {}


def config(name):
    if name not in _cache:
        _cache[name] = wl.config_workload(name)
    return _cache[name]


# ------------------------------------------------------------ named configs
@pytest.mark.parametrize("name", ["tiny", "mtp4"])
@pytest.mark.parametrize("path", ["auto", "warp", "mma"])
def test_small_configs_full_output(name, path):
    w = config(name)
    out, lse, info = run_gpu(w, {"path": path})
    ref_out, ref_lse = oracle.verify_attn(w)
    compare(out, lse, ref_out, ref_lse, f"{name}/{path} {info}")


def _sample_rows(w, n_extra=12, seed=0):
    B, T, Hq = w["q"].shape[:3]
    G = Hq // w["Hkv"]
    rows = {(0, 0, 0), (B - 1, T - 1, Hq - 1), (0, T - 1, 0), (B - 1, 0, Hq - 1)}
    for g in range(w["Hkv"]):  # needle-aligned heads (query 0 of each group)
        rows.add((0, 0, g * G))
    rng = np.random.default_rng(seed)
    for _ in range(n_extra):
        rows.add((int(rng.integers(B)), int(rng.integers(T)), int(rng.integers(Hq))))
    return sorted(rows)


@pytest.mark.parametrize("name", ["lookup16", "batched", "maxctx"])
def test_full_size_configs_full_output(name):
    """Every (b, t, h) row of the full-size configurations against the oracle,
    in the plan the benchmark uses: max-abs and the one-ulp allowance per
    element, mean-abs over the whole output, the LSE bound on every row.  The
    count of elements that needed the ulp allowance is printed and bounded
    (it should stay a tiny fraction: only outputs of magnitude >= 2 can use it)."""
    w = config(name)
    out, lse, info = run_gpu(w)
    ref_out, ref_lse = oracle.verify_attn(w)
    stats = compare(out, lse, ref_out, ref_lse, f"{name} {info}")
    print(f"{name}: {stats}")
    assert stats["ulp_allowance_used"] <= 1e-3 * stats["elements"], stats
    assert np.isfinite(out).all() and np.isfinite(lse).all()


def test_112k_context_full_output():
    """A 112k context ("I pushed Qwen3.8-27B to 381 tps for a single request
    on a RTX 3090" measures single-user decode there): 112,000 + 16 tokens,
    the maxctx shapes, needles at the same depth fractions; every output row
    against the oracle in the default plan."""
    w = wl.config_workload("maxctx", ctx=112000)
    out, lse, info = run_gpu(w)
    ref_out, ref_lse = oracle.verify_attn(w)
    stats = compare(out, lse, ref_out, ref_lse, f"maxctx/ctx112000 {info}")
    print(f"maxctx/ctx112000: {stats}")
    assert stats["ulp_allowance_used"] <= 1e-3 * stats["elements"], stats


# ------------------------------------------------------------ non-unit scales
SCALED = [(k, v, dt, T, G) for (k, v) in ((1e-3, 1e-3), (30.0, 30.0), (1.0, 1e-4), (1.0, 30.0), (30.0, 1e-4))
          for dt in ("int8", "fp8_e4m3", "int4", "int2") for (T, G) in ((16, 6), (1, 4))]


@pytest.mark.parametrize("k_std,v_std,dt,T,G", SCALED)
def test_non_unit_scales(k_std, v_std, dt, T, G):
    """K and V rows drawn at standard deviations far from 1 (tiny scales push
    the folded value scale toward fp16's subnormal range, large key scales make
    the softmax nearly one-hot).  The output bounds scale with v_std; the LSE
    bound is relative.  Both kernels (T=16, G=6 -> tensor cores; T=1, G=4 ->
    CUDA cores), with a split so the combine runs."""
    w = wl.make_workload(4100 + int(1000 * T + G), [3000 + T, 1200 + T], T, G * 2, 2, 256, dt,
                         k_std=k_std, v_std=v_std)
    out, lse, info = run_gpu(w, {"tokens_per_split": 512})
    ref_out, ref_lse = oracle.verify_attn(w)
    stats = compare(out, lse, ref_out, ref_lse, f"k_std {k_std} v_std {v_std} {dt} {info}", v_std=v_std)
    print(f"k_std {k_std} v_std {v_std} {dt} T{T} G{G}: {stats}")


# ------------------------------------------------------------ 4-bit / 2-bit caches
PACKED = [(T, G, D, dt) for dt in ("int4", "int2") for (T, G) in ((1, 4), (5, 4), (16, 6), (8, 8))
          for D in (64, 128, 256)]


@pytest.mark.parametrize("path", ["warp", "mma"])
@pytest.mark.parametrize("T,G,D,dt", PACKED)
def test_packed_cache_shapes(T, G, D, dt, path):
    """The 4-bit / 2-bit caches (the int8 rule with codes +-7 / +-1, packed
    low bits first) in both kernels, every head width: the shortest possible
    sequence, one page + T, ragged tails and a split sequence."""
    lens = [T, 16 + T, 203, 1200 + T]
    w = wl.make_workload(5000 + 97 * T + 13 * G + D + len(dt), lens, T, G * 2, 2, D, dt, extra_pages=2)
    out, lse, info = run_gpu(w, {"tokens_per_split": 128, "path": path})
    ref_out, ref_lse = oracle.verify_attn(w)
    compare(out, lse, ref_out, ref_lse, f"T{T} G{G} D{D} {dt} {path} {info}")


# ------------------------------------------------------------ wide shapes
@pytest.mark.parametrize("path", ["auto", "warp"])
@pytest.mark.parametrize("T,G,D,dt", [(24, 8, 128, "int8"), (16, 15, 256, "fp8_e4m3"), (32, 5, 64, "bf16")])
def test_more_rows_than_one_mma_tile(T, G, D, dt, path):
    """Packed rows per kv head above the tensor-core tile's 128 (192, 240,
    160): several row groups per kv head, each re-reading the cache, with a
    split so that the combine merges every group."""
    w = wl.make_workload(9100 + T * G + D, [T + 3, 700 + T, 2000 + T], T, G * 2, 2, D, dt)
    out, lse, info = run_gpu(w, {"path": path, "tokens_per_split": 256})
    assert info["num_row_groups"] > 1
    ref_out, ref_lse = oracle.verify_attn(w)
    compare(out, lse, ref_out, ref_lse, f"T{T} G{G} D{D} {dt} {path} {info}")


@pytest.mark.parametrize("T,G", [(1, 1), (1, 4), (5, 6)])
def test_wide_batch_many_heads(T, G):
    """256 sequences of 1 to 2,000 cached tokens (several shorter than one
    page) with 8 kv heads, D = 128, int8, in the default plan: the packed-row
    crossover picks the CUDA-core kernel at one row and tensor cores above."""
    rng = np.random.default_rng(77 + T + G)
    lens = [int(x) + T for x in rng.integers(1, 2000, 256)]
    w = wl.make_workload(9300 + T + G, lens, T, G * 8, 8, 128, "int8")
    out, lse, info = run_gpu(w)
    assert info["path"] == (1 if T * G <= 2 else 2)
    ref_out, ref_lse = oracle.verify_attn(w)
    compare(out, lse, ref_out, ref_lse, f"B256 T{T} G{G} {info}")


# ------------------------------------------------------------ CUDA-core kernel: every instantiation
WARP_ROWS = [(D, dt, T, G) for D in (64, 128, 256) for dt in ("bf16", "fp8_e4m3", "int8", "int4", "int2")
             for (T, G) in ((1, 1), (2, 1), (1, 3), (2, 2))]


@pytest.mark.parametrize("D,dt,T,G", WARP_ROWS)
def test_warp_kernel_every_variant(D, dt, T, G):
    """The CUDA-core kernel at 1, 2, 3 and 4 packed rows per kv head (its
    one-, two- and four-row variants) for every cache type and head width:
    a sequence shorter than one key batch, one ending mid-batch and
    mid-page, and two split into items of a few 32-key tiles (several
    batches per warp, the last item ragged), all against the oracle."""
    lens = [T, 37 + T, 300 + T, 2100 + T]
    w = wl.make_workload(8000 + D + 10 * T + G + len(dt), lens, T, G * 2, 2, D, dt, extra_pages=3)
    out, lse, info = run_gpu(w, {"path": "warp", "tokens_per_split": 96})
    assert info["path"] == 1 and info["rows_per_group"] == T * G
    ref_out, ref_lse = oracle.verify_attn(w)
    compare(out, lse, ref_out, ref_lse, f"warp D{D} {dt} T{T} G{G} {info}")


@pytest.mark.parametrize("dt", ["int4", "int2"])
def test_maxctx_packed_full_output(dt):
    """262144 + 16 cached tokens (24 q / 4 kv heads, D = 256, needles at
    10/50/90/99 % depth) in a 4-bit / 2-bit cache: every output row against
    the oracle, in the default plan (tensor cores, one split per SM)."""
    w = wl.config_workload("maxctx", kv_dtype=dt)
    out, lse, info = run_gpu(w)
    assert info["path"] == 2 and info["max_splits"] > 1
    ref_out, ref_lse = oracle.verify_attn(w)
    stats = compare(out, lse, ref_out, ref_lse, f"maxctx {dt} {info}")
    print(f"maxctx/{dt}: {stats}")
    assert stats["ulp_allowance_used"] <= 1e-3 * stats["elements"], stats


# ------------------------------------------------------------ long contexts, other dtypes / widths
@pytest.mark.parametrize("D,dt,L,T,G", [(128, "bf16", 20_000, 8, 6), (64, "fp8_e4m3", 30_000, 5, 8),
                                        (256, "bf16", 12_000, 16, 6), (128, "int8", 40_000, 16, 4)])
def test_long_context_other_shapes_sampled_rows(D, dt, L, T, G):
    """The tensor-core path well past one split per SM in the other head
    widths and cache types (sampled rows against the oracle, all outputs finite)."""
    w = wl.make_workload(7000 + D + L, [L], T, G * 2, 2, D, dt)
    out, lse, info = run_gpu(w)
    assert info["path"] == 2 and info["max_splits"] > 1
    rows = _sample_rows(w, n_extra=10)
    ref_o, ref_l = oracle.verify_attn_rows(w, rows)
    got_o = np.stack([out[b, t, h] for b, t, h in rows])
    got_l = np.array([lse[b, t, h] for b, t, h in rows])
    compare(got_o, got_l, ref_o, ref_l, f"D{D} {dt} L{L} {info}")
    assert np.isfinite(out).all() and np.isfinite(lse).all()


# ------------------------------------------------------------ shape sweep
SWEEP = []
for T in (1, 5, 8, 16):
    for G in (1, 4, 6, 8):
        for i, D in enumerate((64, 128, 256)):
            dt = ("bf16", "fp8_e4m3", "int8")[(T + G + i) % 3]
            SWEEP.append((T, G, D, dt))


@pytest.mark.parametrize("path", ["warp", "mma"])
@pytest.mark.parametrize("T,G,D,dt", SWEEP)
def test_shape_sweep(T, G, D, dt, path):
    Hkv = 2
    lens = [T, 16 + T, 203, 77 + T]  # shortest possible, < 1 page + T, ragged tails
    w = wl.make_workload(1000 + T * 31 + G * 7 + D, lens, T, G * Hkv, Hkv, D, dt, extra_pages=2)
    out, lse, info = run_gpu(w, {"tokens_per_split": 64, "path": path})
    ref_out, ref_lse = oracle.verify_attn(w)
    compare(out, lse, ref_out, ref_lse, f"T{T} G{G} D{D} {dt} {info}")


@pytest.mark.parametrize("path", ["warp", "mma"])
@pytest.mark.parametrize("dt", ["bf16", "fp8_e4m3", "int8"])
@pytest.mark.parametrize("split", [32, 64, 100, 512, 0])
def test_split_count_invariance(dt, split, path):
    w = wl.make_workload(77, [1234, 517], 8, 12, 2, 128, dt)
    out, lse, info = run_gpu(w, {"tokens_per_split": split, "path": path})
    ref_out, ref_lse = oracle.verify_attn(w)
    compare(out, lse, ref_out, ref_lse, f"split {split} {info}")


@pytest.mark.parametrize("path", ["warp", "mma"])
def test_page_permutation_bitwise_for_fixed_plan(path):
    w = wl.make_workload(91, [700, 333], 5, 24, 4, 256, "int8", extra_pages=5)
    out1, lse1, _ = run_gpu(w, {"tokens_per_split": 128, "path": path})
    perm = np.random.default_rng(4).permutation(w["num_pages"])
    w2 = dict(w)
    for key in ("k_pages", "v_pages", "k_scale", "v_scale"):
        a = np.empty_like(w[key])
        a[perm] = w[key]
        w2[key] = a
    w2["block_table"] = perm[w["block_table"]].astype(np.int32)
    out2, lse2, _ = run_gpu(w2, {"tokens_per_split": 128, "path": path})
    assert np.array_equal(out1, out2) and np.array_equal(lse1, lse2)


def test_block_table_stride_and_side_stream():
    w = wl.make_workload(93, [150, 90], 4, 8, 2, 64, "fp8_e4m3", bt_stride=40)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        out, lse, info = run_gpu(w, {"block_table_stride": 40}, stream=s)
    ref_out, ref_lse = oracle.verify_attn(w)
    compare(out, lse, ref_out, ref_lse, "stride40")


# ------------------------------------------------------------ checks and errors
@pytest.mark.parametrize("path", ["warp", "mma"])
def test_bad_page_is_skipped_and_flagged(path):
    """A block-table entry at or above the planned pool size is skipped and
    flagged.  The entry used still lies inside the allocation (the pool is
    allocated larger than the size given to the planner), so the access is
    in bounds whether or not the check works."""
    import speculative_decoding_verify_causal_gb300 as va
    w = wl.make_workload(95, [100], 2, 4, 1, 64, "int8", extra_pages=10)
    n_used = 7  # pages 0..6 hold the sequence after renumbering below
    # renumber so that the sequence uses pages 0..6 and pages 7..16 are spare
    order = w["block_table"][0, :n_used]
    w["k_pages"][:n_used] = w["k_pages"][order]
    w["v_pages"][:n_used] = w["v_pages"][order]
    w["k_scale"][:n_used] = w["k_scale"][order]
    w["v_scale"][:n_used] = w["v_scale"][order]
    w["block_table"][0, :n_used] = np.arange(n_used)
    d = wl.to_device(w)
    d["block_table"][0, 3] = 12  # allocated, but >= num_pages given below
    plan = va.verify_attn_plan(w["seq_lens"], 2, 4, 1, 64, "int8", num_pages=10, path=path)
    try:
        va.verify_attn_with_plan(plan, d["q"], d["k_pages"], d["v_pages"], d["k_scale"], d["v_scale"],
                                 d["block_table"], d["seq_lens"], 2, d["out"], d["lse"])
        flags = va.verify_attn_plan_device_flags(plan)
        assert flags & 1
        assert va.verify_attn_plan_device_flags(plan) == 0  # cleared
        assert torch.isfinite(d["out"].float()).all()
        # the skipped page's 16 keys are absent: compare with the oracle on a
        # cache where those keys cannot win (their K rows pushed to -inf score
        # is not expressible, so check against a direct computation instead)
        out = d["out"].float().cpu().numpy()
        keep = [j for j in range(100) if j // 16 != 3]
        ref = _masked_reference(w, keep)
        assert np.abs(out - ref).max() < 2e-2
    finally:
        plan.destroy()


def _masked_reference(w, keep):
    """Oracle output when only the key positions in `keep` exist: the oracle's
    partials over the kept contiguous key ranges, merged by log-sum-exp (the
    merge is pinned by the oracle tests)."""
    import math
    ranges = []
    for j in keep:
        if ranges and ranges[-1][1] == j:
            ranges[-1][1] = j + 1
        else:
            ranges.append([j, j + 1])
    T, Hq, D = w["T"], w["Hq"], w["D"]
    out = np.zeros((1, T, Hq, D))
    for t in range(T):
        for h in range(Hq):
            parts = [oracle.verify_attn_partial(w, 0, t, h, a, b) for a, b in ranges]
            lses = np.array([pl for _, pl in parts])
            m = lses.max()
            tot = m + math.log(np.exp(lses - m).sum())
            out[0, t, h] = sum(np.exp(pl - tot) * po for po, pl in parts if np.isfinite(pl))
    return out


def test_seq_len_mismatch_is_flagged():
    import speculative_decoding_verify_causal_gb300 as va
    w = wl.make_workload(97, [100], 2, 4, 1, 64, "bf16")
    d = wl.to_device(w)
    d["seq_lens"][0] = 99
    plan = va.verify_attn_plan(w["seq_lens"], 2, 4, 1, 64, "bf16")
    try:
        va.verify_attn_with_plan(plan, d["q"], d["k_pages"], d["v_pages"], None, None,
                                 d["block_table"], d["seq_lens"], 2, d["out"], d["lse"])
        assert va.verify_attn_plan_device_flags(plan) & 2
    finally:
        plan.destroy()


def test_error_codes_through_the_abi():
    import speculative_decoding_verify_causal_gb300 as va
    lib = va.library()
    w = wl.make_workload(99, [64], 4, 8, 2, 64, "int8")
    d = wl.to_device(w)
    plan = va.verify_attn_plan(w["seq_lens"], 4, 8, 2, 64, "int8")
    P = ctypes.c_void_p
    ptrs = [P(d[k].data_ptr()) for k in ("q", "k_pages", "v_pages", "k_scale", "v_scale", "block_table",
                                         "seq_lens")]
    outp, lsep = P(d["out"].data_ptr()), P(d["lse"].data_ptr())
    try:
        assert lib.verify_attn_with_plan(plan.handle, *ptrs, 5, outp, lsep, P(0)) == -3  # T mismatch
        bad = list(ptrs)
        bad[3] = P(0)  # quantised cache without k_scale
        assert lib.verify_attn_with_plan(plan.handle, *bad, 4, outp, lsep, P(0)) == -1
        assert lib.verify_attn_with_plan(plan.handle, *ptrs, 4, P(0), lsep, P(0)) == -1
        # the 11-argument form uses the thread's current plan
        assert lib.verify_attn(*ptrs, 4, outp, P(0), P(0)) == 0
        torch.cuda.synchronize()
        ref_out, _ = oracle.verify_attn(w)
        compare(d["out"].float().cpu().numpy(), np.zeros_like(ref_out[..., 0]),
                ref_out, np.zeros_like(ref_out[..., 0]), "current-plan form")
    finally:
        plan.destroy()
    assert lib.verify_attn(*ptrs, 4, outp, lsep, P(0)) == -4  # destroyed -> no current plan
