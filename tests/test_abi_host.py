"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every function include/verify_attn.h declares, and the split planner's work
lists are valid and chosen from the live lengths only."""
import ctypes
import os
import re

import numpy as np
import pytest

import speculative_decoding_verify_causal_gb300 as va
from speculative_decoding_verify_causal_gb300 import build as vbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    vbuild.build()


def declared_functions():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if not f.endswith(".h"):
            continue
        src = open(os.path.join(ROOT, "include", f)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\**\s*([a-z_0-9]+)\s*\(", src, flags=re.M):
            names.add(m.group(1))
    return sorted(names)


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("verify_attn_plan", "verify_attn", "verify_attn_with_plan", "verify_attn_plan_destroy",
              "verify_attn_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(va.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings():
    for code in range(-8, 1):
        s = va.verify_attn_status_string(code)
        assert s and s != "unknown status"
    assert va.verify_attn_status_string(-99) == "unknown status"


def _check_cover(lens, T, Hq, Hkv, items, info):
    G = Hq // Hkv
    R = G * T
    rg_n = info["num_row_groups"]
    assert info["rows_per_group"] * rg_n >= R
    seen = {}
    for b, kvh, rg, k0, k1 in items:
        assert 0 <= b < len(lens) and 0 <= kvh < Hkv and 0 <= rg < rg_n
        assert 0 <= k0 < k1 <= lens[b]
        seen.setdefault((b, kvh, rg), []).append((k0, k1))
    assert len(seen) == len(lens) * Hkv * rg_n
    for (b, kvh, rg), ranges in seen.items():
        ranges.sort()
        assert ranges[0][0] == 0 and ranges[-1][1] == lens[b]
        for (a0, a1), (b0, b1) in zip(ranges, ranges[1:]):
            assert a1 == b0  # contiguous, no overlap
        n = len(ranges)
        assert n <= info["max_splits"]


@pytest.mark.parametrize("lens,T,Hq,Hkv,D,dt", [
    ([261], 5, 4, 1, 64, "bf16"),
    ([1541], 5, 24, 4, 256, "fp8_e4m3"),
    ([25016], 16, 24, 4, 256, "int8"),
    ([262160], 16, 24, 4, 256, "int8"),
    (list(np.random.default_rng(3).integers(1000, 8001, 64) + 5), 5, 24, 4, 256, "fp8_e4m3"),
    ([1, 2, 3, 17, 33], 1, 8, 8, 128, "bf16"),
    ([262160], 16, 24, 4, 256, "int4"),
    ([3005, 705, 17], 5, 24, 4, 64, "int2"),
])
@pytest.mark.parametrize("path", ["warp", "mma", "auto"])
def test_planner_covers_every_key_once(lens, T, Hq, Hkv, D, dt, path):
    lens = [int(x) for x in lens]
    T = min(T, min(lens))
    info, items = va.verify_attn_plan_describe(lens, T, Hq, Hkv, D, dt, num_sms=148, path=path)
    assert info["num_items"] == len(items) > 0
    _check_cover(lens, T, Hq, Hkv, items, info)


def test_planner_fills_the_chip_for_one_long_sequence():
    # 25k tokens, 4 kv heads: the split must give at least one item per SM
    info, items = va.verify_attn_plan_describe([25016], 16, 24, 4, 256, "int8", num_sms=148, path="warp")
    assert info["num_items"] >= 148
    assert info["max_splits"] > 1


def test_planner_picks_the_kernel_by_packed_row_count():
    # CUDA cores for one or two packed rows per kv head, tcgen05 from three
    # rows on (the crossover measured on GB300); either kernel on request
    big, _ = va.verify_attn_plan_describe([25016], 16, 24, 4, 256, "int8", num_sms=148)
    two, _ = va.verify_attn_plan_describe([25016], 1, 8, 4, 256, "int8", num_sms=148)
    one, _ = va.verify_attn_plan_describe([261], 1, 1, 1, 64, "bf16", num_sms=148)
    three, _ = va.verify_attn_plan_describe([25016], 3, 4, 4, 256, "int8", num_sms=148)
    forced, _ = va.verify_attn_plan_describe([25016], 1, 8, 4, 256, "int8", num_sms=148, path="mma")
    assert big["path"] == 2 and three["path"] == 2 and forced["path"] == 2
    assert two["path"] == 1 and one["path"] == 1
    assert two["rows_per_group"] == 2 and two["num_row_groups"] == 1
    wide, _ = va.verify_attn_plan_describe([2000], 16, 24, 4, 256, "int8", num_sms=148, path="warp")
    assert wide["rows_per_group"] == 4 and wide["num_row_groups"] == 24  # 4 rows per CUDA-core item
    assert big["rows_per_group"] == 96 and big["num_row_groups"] == 1
    # one CTA per SM for the tensor-core kernel: about one wave of items
    assert 148 * 0.75 <= big["num_items"] <= 148


def test_planner_uses_live_lengths_only():
    # The block-table stride (the declared maximum context) must not change
    # the split geometry.
    a = va.verify_attn_plan_describe([3000, 700], 5, 24, 4, 256, "fp8_e4m3", num_sms=148)
    b = va.verify_attn_plan_describe([3000, 700], 5, 24, 4, 256, "fp8_e4m3", num_sms=148,
                                     block_table_stride=16384)
    assert a[0] == b[0] and np.array_equal(a[1], b[1])


def test_planner_forced_split_length():
    info, items = va.verify_attn_plan_describe([1000], 4, 8, 2, 64, "bf16", num_sms=148, path="warp",
                                               tokens_per_split=100)
    # rounded up to the 32-key tile: 128-token splits -> 8 splits per kv-head / row group
    assert info["tokens_per_split"] == 128
    assert info["max_splits"] == 8
    _check_cover([1000], 4, 8, 2, items, info)


@pytest.mark.parametrize("kw,code", [
    (dict(seq_lens=[4], T=5), va.VerifyAttnError),                      # L < T
    (dict(Hq=6, Hkv=4), va.VerifyAttnError),                            # Hq % Hkv
    (dict(D=96), va.VerifyAttnError),                                   # unsupported head_dim
    (dict(dt=5), va.VerifyAttnError),                                   # unknown cache type
    (dict(block_table_stride=1, seq_lens=[100]), va.VerifyAttnError),   # stride < pages
])
def test_planner_rejects_bad_arguments(kw, code):
    args = dict(seq_lens=[64], T=4, Hq=8, Hkv=2, D=64, dt="bf16")
    extra = {}
    for k, v in kw.items():
        if k in args:
            args[k] = v
        else:
            extra[k] = v
    with pytest.raises(code):
        va.verify_attn_plan_describe(args["seq_lens"], args["T"], args["Hq"], args["Hkv"], args["D"],
                                     args["dt"], num_sms=148, **extra)


def test_verify_attn_without_plan_reports_no_plan():
    lib = va.library()
    rc = lib.verify_attn(*([ctypes.c_void_p(0)] * 7), 5, ctypes.c_void_p(0), ctypes.c_void_p(0),
                         ctypes.c_void_p(0))
    assert rc == -4  # VA_ERR_NO_PLAN


def test_destroy_null_is_noop():
    va.library().verify_attn_plan_destroy(ctypes.c_void_p(0))


@pytest.mark.parametrize("B,T", [(1, 1), (1, 16), (64, 5), (3, 7)])
def test_accept_workspace_size(B, T):
    """Host only: one 32-byte statistics record per (sequence, position) plus
    one 16-byte race slot per sequence; 0 for arguments the call rejects."""
    lib = va.library()
    assert lib.verify_attn_accept_workspace_bytes(B, T) == 32 * B * (T + 1) + 16 * B
    assert lib.verify_attn_accept_workspace_bytes(0, T) == 0
    assert lib.verify_attn_accept_workspace_bytes(B, 0) == 0


def test_validate_host_paging_inputs():
    # host-only check of seq_lens and the block-table entries in use
    rng = np.random.default_rng(5)
    lens = np.array([40, 16, 5, 33], np.int32)
    bt = rng.integers(0, 50, size=(4, 3)).astype(np.int32)
    assert va.verify_attn_validate_host(lens, 5, bt, 50) is None
    bt_unused = bt.copy()
    bt_unused[1, 1:] = -7           # sequence 1 uses one page: later entries are not read
    bt_unused[2, 1:] = 999
    assert va.verify_attn_validate_host(lens, 5, bt_unused, 50) is None
    bad = bt.copy()
    bad[3, 2] = 50                  # == num_pages: outside the pool
    assert va.verify_attn_validate_host(lens, 5, bad, 50) == (3, 2)
    bad = bt.copy()
    bad[0, 1] = -1
    assert va.verify_attn_validate_host(lens, 5, bad, 50) == (0, 1)
    assert va.verify_attn_validate_host(np.array([40, 16, 4, 33], np.int32), 5, bt, 50) == (2, -1)  # L < T
    assert va.verify_attn_validate_host(np.array([40, 16, 5, 49], np.int32), 5, bt, 50) == (3, -1)  # > 16 * stride
    with pytest.raises(va.VerifyAttnError):
        va.verify_attn_validate_host(lens, 5, bt, 0)


def test_planner_random_shapes_cover_every_key_and_respect_kernel_limits():
    # randomised shapes through the host planner: every (sequence, kv head,
    # row group) key range covered exactly once, item starts on the kernel's
    # split tile, tensor-core items no longer than the page ids it stages,
    # CUDA-core items no wider than its 4-row variant, and the path the
    # packed-row crossover names
    rng = np.random.default_rng(2026)
    for _ in range(150):
        B = int(rng.integers(1, 40))
        T = int(rng.integers(1, 17))
        Hkv = int(rng.choice([1, 2, 4, 8]))
        G = int(rng.integers(1, 9))
        D = int(rng.choice([64, 128, 256]))
        dt = str(rng.choice(["bf16", "fp8_e4m3", "int8", "int4", "int2"]))
        lens = [int(x) + T for x in rng.integers(0, int(rng.choice([50, 2000, 70000])), B)]
        path = str(rng.choice(["auto", "warp", "mma"]))
        sms = int(rng.choice([16, 148, 152]))
        info, items = va.verify_attn_plan_describe(lens, T, G * Hkv, Hkv, D, dt, num_sms=sms, path=path)
        assert info["num_items"] == len(items) > 0
        _check_cover(lens, T, G * Hkv, Hkv, items, info)
        want = {"warp": 1, "mma": 2}.get(path, 1 if G * T <= 2 else 2)
        assert info["path"] == want
        tile = 64 if want == 2 else 32
        assert all(k0 % tile == 0 for _, _, _, k0, _ in items)
        if want == 2:
            assert max(k1 - k0 for _, _, _, k0, k1 in items) <= 16384
        else:
            assert info["rows_per_group"] <= 4
