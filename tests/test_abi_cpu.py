"""The C ABI on a host without a GPU: the library builds, loads and exports every
function include/dp_gemm.h declares; the planner, workspace sizing, status strings
and argument checks work without touching a device."""
import ctypes
import os
import re

import pytest

import fp32_dense_projection_gb300 as dp
from fp32_dense_projection_gb300 import build as dpbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dp_gemm.h")


@pytest.fixture(scope="module")
def L():
    dpbuild.build()
    return dp.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([A-Za-z_][A-Za-z0-9_]*)\s*\(", src, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "while", "sizeof")))


def test_header_declares_the_six_ops():
    names = declared_functions()
    for n in ("dp_gemm_fwd", "dp_gemm_dgrad", "dp_gemm_wgrad", "router_fwd", "router_dgrad", "router_wgrad",
              "dp_workspace_size", "dp_plan_query", "dp_status_string"):
        assert n in names


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert len(names) >= 18
    missing = [n for n in names if not hasattr(L, n)]
    assert not missing, missing


def test_status_strings(L):
    for s in range(8):
        assert dp.status_string(s) and "unknown" not in dp.status_string(s)
    assert "unknown" in dp.status_string(99)
    assert L.dp_version() >= 100


SM = 152


def check_simt_plan(op, T, N, K, p):
    assert op.startswith("router")
    assert p["block_m"] == 64 and p["block_n"] in (32, 64) and p["block_k"] == 4096 // p["block_n"]
    assert 1 <= p["splits"] <= 8 and p["workspace_bytes"] == 0 and not p["cta_pair"] and not p["swap_ab"]
    view = {"router_fwd": (T, N, K, 0, 0), "router_dgrad": (T, K, N, 0, 1), "router_wgrad": (N, K, T, 1, 1)}[op]
    assert (p["gemm_m"], p["gemm_n"], p["gemm_k"], p["a_mn_major"], p["b_mn_major"]) == view
    assert p["tiles_m"] == -(-p["gemm_m"] // 64) and p["tiles_n"] == -(-p["gemm_n"] // p["block_n"])
    assert p["units"] == p["grid"] == p["tiles_m"] * p["tiles_n"] * p["splits"]
    assert p["k_blocks"] == -(-p["gemm_k"] // p["block_k"]) and p["splits"] <= p["k_blocks"]
    assert dp.plan(op, T, N, K, sm_count=SM) == p


@pytest.mark.parametrize("op", list(dp.OP_NAMES))
@pytest.mark.parametrize("T,N,K", [(64, 1024, 4096), (16384, 12288, 4096), (16231, 12288, 4096),
                                   (65537, 64, 4096), (1025, 48, 5120), (1024, 256, 4096), (1, 8, 8)])
def test_plan_is_valid(op, T, N, K):
    p = dp.plan(op, T, N, K, out_f32=False, sm_count=SM)
    if p["program"] == 1:  # the router's SIMT FP32 program
        check_simt_plan(op, T, N, K, p)
        return
    pair = bool(p["cta_pair"])
    x3 = op in ("router_fwd", "router_wgrad")  # FP32 A split in the kernel, 32-wide blocks
    assert p["block_m"] == (256 if pair else 128)
    assert p["block_k"] == (32 if x3 else 64)
    assert p["block_n"] in ((128, 256) if pair else (64, 128, 256))
    slots = SM // 2 if pair else SM
    ctas_per_tile = 2 if pair else 1
    assert 1 <= p["grid"] <= SM and p["grid"] % ctas_per_tile == 0
    assert p["grid"] // ctas_per_tile <= p["units"]
    tiles = p["tiles_m"] * p["tiles_n"]
    assert p["units"] == p["full_units"] + (tiles - p["full_units"]) * p["splits"]
    assert 0 <= p["full_units"] <= tiles
    # either no tile is split, every tile is, or only the last partial wave's tiles are
    assert p["full_units"] in (0, tiles) or (p["full_units"] % slots == 0 and tiles - p["full_units"] < slots)
    assert 1 <= p["splits"] <= max(1, p["k_blocks"])
    assert p["tiles_m"] * p["block_m"] >= p["gemm_m"] and p["tiles_n"] * p["block_n"] >= p["gemm_n"]
    bk = p["block_k"]
    assert p["k_blocks"] * bk >= p["gemm_k"] > (p["k_blocks"] - 1) * bk
    if op == "router_wgrad":  # always transposed: dW^T = X^T dY
        assert p["swap_ab"] == 1 and (p["gemm_m"], p["gemm_n"], p["gemm_k"]) == (K, N, T)
        assert p["a_mn_major"] == 1 and p["b_mn_major"] == 1
    elif op.endswith("wgrad"):
        if p["swap_ab"]:
            assert (p["gemm_m"], p["gemm_n"], p["gemm_k"]) == (K, N, T)
        else:
            assert (p["gemm_m"], p["gemm_n"], p["gemm_k"]) == (N, K, T)
        assert p["a_mn_major"] == 1 and p["b_mn_major"] == 1
    elif op.endswith("dgrad"):
        # the router contracts the concatenated [lo | hi | hi] x [hi; lo; hi] operands
        assert (p["gemm_m"], p["gemm_n"], p["gemm_k"]) == (T, K, (3 if op == "router_dgrad" else 1) * N)
        assert p["a_mn_major"] == 0 and p["b_mn_major"] == 1
    else:
        assert (p["gemm_m"], p["gemm_n"], p["gemm_k"]) == (T, N, K)
        assert p["a_mn_major"] == 0 and p["b_mn_major"] == 0
    assert not p["swap_ab"] or op.endswith("wgrad")
    if op.startswith("router"):  # the pre-split bf16 operands live in the workspace
        assert p["workspace_bytes"] > 0
    # blocks per ring stage: 1 or 2, two only on an even ring depth, one for BF16x3
    assert p["blocks_per_stage"] in (1, 2) and p["stages"] % p["blocks_per_stage"] == 0
    assert not x3 or p["blocks_per_stage"] == 1
    # pure function: same answer twice, and the workspace query agrees
    assert dp.plan(op, T, N, K, sm_count=SM) == p
    assert dp.workspace_size(op, T, N, K, sm_count=SM) == p["workspace_bytes"]


def test_split_partition_covers_every_block_once():
    # The kernel gives split s the k-blocks [floor(s*nb/S), floor((s+1)*nb/S)).
    for nb in (1, 2, 17, 253, 254, 256, 1025):
        for S in range(1, min(nb, 40) + 1):
            bounds = [s * nb // S for s in range(S + 1)]
            assert bounds[0] == 0 and bounds[-1] == nb
            assert all(bounds[i + 1] > bounds[i] for i in range(S))  # no empty split while S <= nb


def test_wide_projection_keeps_whole_k_in_full_waves():
    # The pages' deterministic dgrad keeps whole K per output tile at 4096 -> 12288; here every
    # tile of the full waves keeps whole K and only the last partial wave may be split.
    for op in ("fwd", "dgrad", "wgrad"):
        for T in (16384, 16231):
            p = dp.plan(op, T, 12288, 4096, sm_count=SM)
            tiles = p["tiles_m"] * p["tiles_n"]
            slots = SM // 2 if p["cta_pair"] else SM
            assert p["full_units"] >= tiles - slots, (op, T, p)


def test_thin_wgrad_spreads_over_the_sms():
    for (K, N) in ((4096, 64), (4096, 128), (5120, 48), (5120, 64)):
        p = dp.plan("wgrad", 65537, N, K, sm_count=SM)
        assert p["units"] >= SM * 0.6, p
        assert p["splits"] > 1


def test_plan_depends_on_sm_count_only_through_argument():
    a = dp.plan("wgrad", 65537, 64, 4096, sm_count=148)
    b = dp.plan("wgrad", 65537, 64, 4096, sm_count=152)
    assert a["grid"] <= 148 and b["grid"] <= 152
    for sm in (2, 3, 148, 152):  # odd SM counts still give whole CTA pairs
        p = dp.plan("fwd", 16384, 12288, 4096, sm_count=sm)
        assert p["grid"] <= sm and (not p["cta_pair"] or p["grid"] % 2 == 0)


def test_plan_overrides_are_read_per_call(monkeypatch):
    monkeypatch.setenv("DP_FORCE_SWAP", "1")
    assert dp.plan("wgrad", 16173, 64, 4096, sm_count=SM)["swap_ab"] == 1
    monkeypatch.setenv("DP_FORCE_SWAP", "0")
    assert dp.plan("wgrad", 16173, 64, 4096, sm_count=SM)["swap_ab"] == 0
    monkeypatch.setenv("DP_FORCE_PAIR", "0")
    assert dp.plan("fwd", 16384, 12288, 4096, sm_count=SM)["cta_pair"] == 0
    monkeypatch.setenv("DP_FORCE_PAIR", "1")
    assert dp.plan("fwd", 16384, 12288, 4096, sm_count=SM)["cta_pair"] == 1
    for sm in (2, 3, 148, 152):  # odd SM counts still give whole CTA pairs
        p = dp.plan("fwd", 16384, 12288, 4096, sm_count=sm)
        assert p["grid"] <= sm and p["grid"] % 2 == 0
    assert dp.plan("fwd", 16384, 12288, 4096, sm_count=SM)["cta_pair"] == 1


def test_raster_groups_the_larger_operand():
    # thin wgrad 4096 -> 512 not swapped: B (X, 4096 columns) is larger than A (dY, 512):
    # row tiles fastest, so the row tiles sharing an X column block run together
    import os
    os.environ["DP_FORCE_SWAP"] = "0"
    try:
        p = dp.plan("wgrad", 65537, 512, 4096, sm_count=SM)
    finally:
        del os.environ["DP_FORCE_SWAP"]
    assert p["raster_rows"] == 1
    # B fits in L2: groups along the dimension whose operand is larger (here columns)
    assert dp.plan("fwd", 16384, 1024, 4096, sm_count=SM)["raster_rows"] == 0


@pytest.mark.parametrize("op,group", [("fwd", 16), ("dgrad", 16), ("wgrad", 8)])
def test_raster_row_groups_keep_a_in_l2_when_b_is_large(monkeypatch, op, group):
    # 4096 -> 12288 at T = 16384: B (W, or X for the weight gradient) is more than half the
    # L2, so groups of row tiles, as many as keep their A slabs within ~104 MB
    p = dp.plan(op, 16384, 12288, 4096, sm_count=SM)
    assert p["raster_rows"] == 1 and p["raster_group"] == group
    assert p["raster_group"] * p["block_m"] * p["gemm_k"] * 2 <= 104e6
    monkeypatch.setenv("DP_FORCE_RASTER_M", "0")
    monkeypatch.setenv("DP_FORCE_GROUP", "4")
    q = dp.plan(op, 16384, 12288, 4096, sm_count=SM)
    assert q["raster_rows"] == 0 and q["raster_group"] == 4


def test_empty_tokens_need_no_workspace():
    for op in dp.OP_NAMES:
        assert dp.workspace_size(op, 0, 64, 128, sm_count=SM) == 0


@pytest.mark.parametrize("T,N,K,want", [(-1, 8, 8, 1), (8, 0, 8, 1), (8, 12, 8, 3), (8, 8, 20, 3),
                                        (2**31, 8, 8, 3)])
def test_size_checks(L, T, N, K, want):
    info = dp.PlanInfo()
    assert L.dp_plan_query(0, T, N, K, 0, SM, ctypes.byref(info)) == want


def test_argument_checks_before_any_device_call(L):
    P = ctypes.c_void_p
    good = P(1 << 20)           # never dereferenced: every call below fails its checks first
    odd = P((1 << 20) + 8)
    # null operand
    assert L.dp_gemm_fwd(None, good, good, 64, 64, 64, 0, 1, None, 0, None) == 1
    # misaligned operand
    assert L.dp_gemm_fwd(odd, good, good, 64, 64, 64, 0, 1, None, 0, None) == 2
    # N not a multiple of 8
    assert L.dp_gemm_dgrad(good, good, good, 64, 60, 64, 0, 1, None, 0, None) == 3
    # leading dimension shorter than the row
    assert L.dp_gemm_wgrad_ex(good, 32, good, 64, good, 64, 64, 64, 64, 0, 1, None, 0, None) == 1
    # leading dimension that breaks the 16-byte row alignment
    assert L.dp_gemm_fwd_ex(good, 68, good, 64, good, 64, 64, 64, 64, 0, 1, None, 0, None) == 2
    # bad output dtype
    assert L.dp_gemm_fwd(good, good, good, 64, 64, 64, 7, 1, None, 0, None) == 1
    # router rows of fp32 must be 16-byte multiples too (ld 66 floats = 264 B is fine, 65 is not)
    assert L.router_fwd_ex(good, 65, good, 64, good, 64, 8, 64, 64, 1, None, 0, None) == 2


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    monkeypatch.setattr(dp, "_lib", None)
    monkeypatch.setattr(dp, "LIB_PATH", str(tmp_path / "absent.so"))
    with pytest.raises(RuntimeError, match="missing"):
        dp.lib()


def test_workspace_only_when_needed():
    # the workspace holds split partials (one 128 x block_n FP32 tile per split of each
    # split tile and CTA) and the router's bf16 operand copies; plain unsplit plans need none
    for op in dp.OP_NAMES:
        for T, N, K in ((64, 1024, 4096), (1024, 256, 4096), (65537, 64, 4096), (16384, 12288, 4096)):
            p = dp.plan(op, T, N, K, sm_count=SM)
            n = dp.workspace_size(op, T, N, K, sm_count=SM)
            tiles = p["tiles_m"] * p["tiles_n"]
            partials = (tiles - p["full_units"]) * (2 if p["cta_pair"] else 1) * p["splits"] * 128 * p["block_n"] * 4
            if p["program"] == 1:  # the router's SIMT program sums its splits in the cluster
                assert n == 0
            elif op.startswith("router"):
                assert n > partials
            elif p["splits"] > 1:
                assert n >= partials > 0
            else:
                assert n == 0


def longest_accumulation(p) -> int:
    """Most contraction elements one accumulator of the plan sums (x3 for BF16x3)."""
    if p["program"] == 1:  # the router's SIMT program accumulates with FP32 FMAs (round to nearest)
        return 0
    if p["stream_k"]:  # a piece never spans more than one slot's share of the blocks
        slots = p["grid"] // (2 if p["cta_pair"] else 1)
        per = -(-p["tiles"] * p["k_blocks"] // slots)
        return min(per, p["k_blocks"]) * p["block_k"]
    split_tiles = p["tiles"] - p["full_units"]
    per = p["k_blocks"] if p["full_units"] > 0 else 0
    if split_tiles > 0:
        per = max(per, -(-p["k_blocks"] // p["splits"]))
    return per * p["block_k"]


# The contraction view of each op: (rows, columns, contraction) of D = A B^T
LONG_SHAPES = [  # (T, N, K) whose contraction exceeds 16384 in some op, with few and with many tiles
    (16385, 64, 4096), (65537, 512, 4096), (200000, 256, 4096), (65536, 16384, 16384), (40000, 24576, 8192),
    (64, 32768, 1024), (1024, 65536, 4096), (8192, 20480, 20480), (3, 17000, 8), (20000, 8, 17000),
]


@pytest.mark.parametrize("op", list(dp.OP_NAMES))
@pytest.mark.parametrize("T", [1025, 16173, 16384, 65537, 200000])
def test_accumulation_length_is_bounded(op, T):
    # no TMEM accumulator takes more than 16384 MMA accumulations per element: 16384
    # contraction elements, or 16384 / 3 for the three BF16x3 terms of the router's
    # forward and weight gradient (its input gradient contracts over 3N elements)
    terms = 3 if op in ("router_fwd", "router_wgrad") else 1
    for N, K in ((64, 4096), (512, 4096), (256, 4096), (12288, 4096)):
        p = dp.plan(op, T, N, K, sm_count=SM)
        assert longest_accumulation(p) * terms <= 16384, (op, T, N, K, p)


@pytest.mark.parametrize("op", list(dp.OP_NAMES))
@pytest.mark.parametrize("T,N,K", LONG_SHAPES)
@pytest.mark.parametrize("out_f32", [False, True])
def test_accumulation_bound_holds_for_every_shape(op, T, N, K, out_f32):
    # including shapes with far more than 4096 output tiles, which split the contraction
    # all the same (their partials take a workspace the size of a few outputs)
    terms = 3 if op in ("router_fwd", "router_wgrad") else 1
    for sm in (SM, 148, 8):
        p = dp.plan(op, T, N, K, out_f32=out_f32, sm_count=sm)
        assert longest_accumulation(p) * terms <= 16384, (op, T, N, K, sm, p)
        if longest_accumulation(p) > 0 and p["k_blocks"] * p["block_k"] * terms > 16384 and p["program"] == 0:
            assert p["splits"] > 1 and p["workspace_bytes"] > 0


@pytest.mark.parametrize("env", [{"DP_FORCE_BN": "64"}, {"DP_FORCE_PAIR": "1"}, {"DP_FORCE_PAIR": "0"},
                                 {"DP_FORCE_SWAP": "1"}, {"DP_FORCE_SWAP": "0"}, {"DP_FORCE_STREAM_K": "1"},
                                 {"DP_FORCE_SPLITS": "2"}, {"DP_FORCE_TAIL_SPLITS": "3"}, {"DP_FORCE_KPS": "2"}])
def test_forced_plans_keep_the_accumulation_bound(monkeypatch, env):
    for k, v in env.items():
        monkeypatch.setenv(k, v)
    for op in dp.OP_NAMES:
        terms = 3 if op in ("router_fwd", "router_wgrad") else 1
        for T, N, K in LONG_SHAPES[:6]:
            try:
                p = dp.plan(op, T, N, K, sm_count=SM)
            except dp.DPError:
                continue  # an override no plan of this shape admits
            assert longest_accumulation(p) * terms <= 16384, (env, op, T, N, K, p)


def test_tuning_overrides_need_the_tuning_switch(tmp_path):
    # without DP_TUNING the library reads no DP_FORCE_* variable: the planner's own plan
    import subprocess
    import sys
    code = ("import fp32_dense_projection_gb300 as dp;"
            "p = dp.plan('fwd', 16384, 12288, 4096, sm_count=152);"
            "print(p['block_n'], p['cta_pair'], p['blocks_per_stage'])")
    env = {k: v for k, v in os.environ.items() if k != "DP_TUNING"}
    env.update({"DP_FORCE_BN": "64", "DP_FORCE_PAIR": "0", "DP_FORCE_KPS": "1", "PYTHONPATH": ROOT})
    plain = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, check=True)
    env["DP_TUNING"] = "1"
    tuned = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, check=True)
    assert tuned.stdout.split() == ["64", "0", "1"]
    p = dp.plan("fwd", 16384, 12288, 4096, sm_count=152)  # (this process: no override set)
    assert plain.stdout.split() == [str(p["block_n"]), str(p["cta_pair"]), str(p["blocks_per_stage"])]
    assert plain.stdout != tuned.stdout


@pytest.mark.parametrize("op", ["fwd", "dgrad", "wgrad"])
@pytest.mark.parametrize("kn", [False, True])
@pytest.mark.parametrize("B,T,N,K", [(1, 1000, 128, 512), (16, 2048, 128, 512), (128, 64, 512, 128), (4, 65537, 64, 256)])
def test_batched_plan_is_valid(op, kn, B, T, N, K):
    p = dp.plan_batched(op, B, T, N, K, weight_kn=kn, sm_count=SM)
    tiles = B * p["tiles_m"] * p["tiles_n"]
    assert p["batch"] == B and p["tiles"] == tiles and p["weight_kn"] == int(kn)
    assert p["units"] == p["full_units"] + (tiles - p["full_units"]) * p["splits"]
    assert 1 <= p["grid"] <= SM
    # [K][N] weights flip the majorness of W's view; the weight gradient's view does not change
    if op == "fwd":
        assert (p["a_mn_major"], p["b_mn_major"]) == (0, int(kn))
    elif op == "dgrad":
        assert (p["a_mn_major"], p["b_mn_major"]) == (0, int(not kn))
    else:
        assert (p["a_mn_major"], p["b_mn_major"]) == (1, 1)
    if B == 1:  # one problem: the plan of the single-problem call (for the [N][K] layout)
        single = dp.plan(op, T, N, K, sm_count=SM)
        if not kn:
            assert p == single
    assert dp.workspace_size_batched(op, B, T, N, K, weight_kn=kn, sm_count=SM) == p["workspace_bytes"]


def test_batched_argument_checks(L):
    P = ctypes.c_void_p
    good = P(1 << 20)
    # bad weight layout flag
    assert L.dp_gemm_fwd_batched(good, 0, 0, good, 0, 0, 2, good, 0, 0, 4, 64, 64, 64, 0, 1, None, 0, None) == 1
    # batch stride breaking the 16-byte alignment (bf16: a multiple of 8 elements)
    assert L.dp_gemm_fwd_batched(good, 0, 12, good, 0, 0, 0, good, 0, 0, 4, 64, 64, 64, 0, 1, None, 0, None) == 2
    # negative batch count
    assert L.dp_gemm_wgrad_batched(good, 0, 0, good, 0, 0, good, 0, 0, 0, -1, 64, 64, 64, 0, 1, None, 0, None) == 1
    # router ops have no batched form
    info = dp.PlanInfo()
    assert L.dp_plan_query_batched(3, 2, 64, 64, 64, 0, 0, SM, ctypes.byref(info)) == 1


# ------------------------------------------------------------------ backward pass

@pytest.mark.parametrize("T,N,K", [(1024, 1024, 4096), (4031, 1024, 4096), (1024, 12288, 4096),
                                   (16384, 12288, 4096), (64, 1024, 4096), (1000, 384, 640), (65537, 64, 4096),
                                   (0, 64, 128)])
@pytest.mark.parametrize("dx32,dw32", [(False, False), (True, False), (False, True)])
def test_bwd_plan_is_consistent(T, N, K, dx32, dw32):
    b = dp.plan_bwd(T, N, K, dx32, dw32, sm_count=SM)
    d, w = b["dgrad"], b["wgrad"]
    if b["fused"]:
        # one tile shape, whole K in every tile of both problems, no workspace, one CTA
        # (or pair) per unit up to one per SM
        per = 2 if d["cta_pair"] else 1
        assert (d["cta_pair"], d["block_n"]) == (w["cta_pair"], w["block_n"])
        for p in (d, w):
            assert p["splits"] == 1 and p["full_units"] == p["units"] == p["tiles"]
        assert b["workspace_bytes"] == 0
        assert b["grid"] == min(d["units"] + w["units"], SM // per) * per
        assert b["model_us"] < b["separate_us"]
    else:
        # the single-op plans, run one after the other with one workspace
        assert d == dp.plan("dgrad", T, N, K, dx32, sm_count=SM)
        assert w == dp.plan("wgrad", T, N, K, dw32, sm_count=SM)
        assert b["workspace_bytes"] == (0 if T == 0 else max(d["workspace_bytes"], w["workspace_bytes"]))
        assert b["grid"] == 0 and b["model_us"] == b["separate_us"]
    assert dp.workspace_size_bwd(T, N, K, dx32, dw32, sm_count=SM) == b["workspace_bytes"]


def test_bwd_co_schedules_small_and_mid_sizes_only():
    assert dp.plan_bwd(1024, 1024, 4096, sm_count=SM)["fused"]
    assert dp.plan_bwd(4031, 1024, 4096, sm_count=SM)["fused"]
    assert not dp.plan_bwd(16384, 12288, 4096, sm_count=SM)["fused"]
    assert not dp.plan_bwd(0, 1024, 4096, sm_count=SM)["fused"]


def test_bwd_overrides(monkeypatch):
    monkeypatch.setenv("DP_FORCE_FUSE", "1")
    assert dp.plan_bwd(16384, 12288, 4096, sm_count=SM)["fused"]
    # beyond the accumulation bound the weight gradient must split: two launches
    assert not dp.plan_bwd(40000, 1024, 1024, sm_count=SM)["fused"]
    for order, first in (("2", 1), ("3", 0)):
        monkeypatch.setenv("DP_FORCE_FUSE", order)
        assert dp.plan_bwd(1000, 384, 640, sm_count=SM)["wgrad_first"] == first
    monkeypatch.setenv("DP_FORCE_FUSE", "1")
    monkeypatch.setenv("DP_FORCE_PAIR", "0")
    monkeypatch.setenv("DP_FORCE_BN", "128")
    b = dp.plan_bwd(1000, 384, 640, sm_count=SM)
    assert b["fused"] and (b["dgrad"]["cta_pair"], b["dgrad"]["block_n"]) == (0, 128)
    monkeypatch.setenv("DP_FORCE_FUSE", "0")
    assert not dp.plan_bwd(1024, 1024, 4096, sm_count=SM)["fused"]


def test_bwd_argument_checks(L):
    P = ctypes.c_void_p
    good = P(1 << 20)   # never dereferenced: every call below fails its checks first
    odd = P((1 << 20) + 8)
    args = lambda dY=good, X=good, W=good, dX=good, dW=good, odx=0, odw=0, N=64: (
        dY, 0, X, 0, W, 0, dX, 0, odx, dW, 0, odw, 64, N, 64, 1, None, 0, None)
    assert L.dp_gemm_bwd(*args(W=None)) == 1
    assert L.dp_gemm_bwd(*args(dW=None)) == 1
    assert L.dp_gemm_bwd(*args(X=odd)) == 2
    assert L.dp_gemm_bwd(*args(odw=5)) == 1
    assert L.dp_gemm_bwd(*args(N=60)) == 3
    info = dp.BwdPlanInfo()
    assert L.dp_plan_query_bwd(64, 64, 64, 2, 0, SM, ctypes.byref(info)) == 1


# ------------------------------------------------------------ router SIMT program

def test_router_program_choice():
    # the SIMT FP32 program for the router's input gradient at a few dozen tokens (one
    # launch, no workspace); the BF16x3 tensor-core program elsewhere
    for T in (1, 64):
        p = dp.plan("router_dgrad", T, 256, 4096, sm_count=SM)
        assert p["program"] == 1 and p["workspace_bytes"] == 0 and p["block_m"] == 64
        assert p["units"] == p["tiles_m"] * p["tiles_n"] * p["splits"] and 1 <= p["splits"] <= 8
    for op in ("router_fwd", "router_wgrad"):
        assert dp.plan(op, 64, 256, 4096, sm_count=SM)["program"] == 0
    for op in ("router_fwd", "router_dgrad", "router_wgrad"):
        assert dp.plan(op, 1024, 256, 4096, sm_count=SM)["program"] == 0
    for op in ("fwd", "dgrad", "wgrad"):
        assert dp.plan(op, 64, 256, 4096, sm_count=SM)["program"] == 0


def test_router_program_overrides(monkeypatch):
    monkeypatch.setenv("DP_FORCE_FFMA", "1")
    monkeypatch.setenv("DP_FORCE_BN", "32")
    monkeypatch.setenv("DP_FORCE_SPLITS", "3")
    p = dp.plan("router_wgrad", 1000, 256, 4096, sm_count=SM)
    assert (p["program"], p["block_n"], p["splits"]) == (1, 32, 3)
    # its view: the plain contraction (weight gradient over the tokens, unswapped)
    assert (p["gemm_m"], p["gemm_n"], p["gemm_k"], p["swap_ab"]) == (256, 4096, 1000, 0)
    assert p["k_blocks"] == -(-1000 // p["block_k"]) and p["block_k"] == 4096 // 32
    monkeypatch.setenv("DP_FORCE_FFMA", "0")
    monkeypatch.delenv("DP_FORCE_BN")
    monkeypatch.delenv("DP_FORCE_SPLITS")
    assert dp.plan("router_dgrad", 64, 256, 4096, sm_count=SM)["program"] == 0


# ------------------------------------------------------------------ stream-K plans

@pytest.mark.parametrize("op,T,N,K", [("wgrad", 16173, 64, 4096), ("wgrad", 1025, 128, 4096), ("fwd", 1000, 136, 4096)])
def test_stream_k_plan(monkeypatch, op, T, N, K):
    # forced: every slot of the grid, splits = the most pieces one tile is cut into,
    # units = all pieces, a partial slot per piece in the workspace
    monkeypatch.setenv("DP_FORCE_STREAM_K", "1")
    p = dp.plan(op, T, N, K, sm_count=SM)
    per = 2 if p["cta_pair"] else 1
    slots = SM // per
    tiles = p["tiles_m"] * p["tiles_n"]
    assert p["stream_k"] == 1 and p["grid"] == slots * per and p["full_units"] == 0 and tiles <= slots
    W = tiles * p["k_blocks"]
    counts = [0] * tiles
    for c in range(slots):
        b, e = c * W // slots, (c + 1) * W // slots
        for t in range(b // p["k_blocks"], (e - 1) // p["k_blocks"] + 1):
            counts[t] += 1
    assert p["splits"] == max(counts) >= 2 and p["units"] == sum(counts)
    assert p["workspace_bytes"] >= tiles * per * p["splits"] * 128 * p["block_n"] * 4
    # the planner's own choice for these shapes is not stream-K (measured slower on GB300)
    monkeypatch.delenv("DP_FORCE_STREAM_K")
    assert dp.plan(op, T, N, K, sm_count=SM)["stream_k"] == 0


# ------------------------------------------------------- non-deterministic plans

@pytest.mark.parametrize("op", list(dp.OP_NAMES))
@pytest.mark.parametrize("T,N,K", [(64, 1024, 4096), (1024, 256, 4096), (65537, 64, 4096), (16384, 12288, 4096)])
def test_non_deterministic_plans(op, T, N, K):
    for f32 in (False, True):
        det = dp.plan(op, T, N, K, out_f32=f32, sm_count=SM)
        nd = dp.plan(op, T, N, K, out_f32=f32, sm_count=SM, deterministic=False)
        assert det["atomic"] == 0
        out32 = f32 or op.startswith("router")
        if not out32:  # BF16 outputs: the deterministic plan, whatever the flag
            assert nd == det
            continue
        # atomic sums only for split tiles, and never more workspace than the ordered sums
        assert nd["atomic"] == 0 or nd["splits"] > 1
        assert nd["workspace_bytes"] <= det["workspace_bytes"]
        if nd["atomic"] and not op.startswith("router"):
            assert nd["workspace_bytes"] == 0


def test_atomic_override(monkeypatch):
    monkeypatch.setenv("DP_FORCE_ATOMIC", "1")
    monkeypatch.setenv("DP_FORCE_SPLITS", "3")
    assert dp.plan("dgrad", 200, 512, 2048, out_f32=True, sm_count=SM, deterministic=False)["atomic"] == 1
    # deterministic calls and BF16 outputs never take it
    assert dp.plan("dgrad", 200, 512, 2048, out_f32=True, sm_count=SM)["atomic"] == 0
    assert dp.plan("dgrad", 200, 512, 2048, out_f32=False, sm_count=SM, deterministic=False)["atomic"] == 0
    monkeypatch.setenv("DP_FORCE_ATOMIC", "0")
    assert dp.plan("dgrad", 200, 512, 2048, out_f32=True, sm_count=SM, deterministic=False)["atomic"] == 0


@pytest.mark.parametrize("op,T,N,K,kps", [
    ("fwd", 64, 1024, 4096, 2), ("dgrad", 64, 1024, 4096, 2),      # short, latency-bound units
    ("wgrad", 1025, 64, 4096, 2),
    ("fwd", 16384, 12288, 4096, 2), ("dgrad", 16384, 12288, 4096, 2),  # many waves of L2-fed units
    ("wgrad", 16384, 12288, 4096, 2),
    ("wgrad", 16173, 128, 4096, 1), ("wgrad", 65537, 64, 4096, 1),    # long DRAM streams, one wave
    ("wgrad", 65537, 512, 4096, 1), ("dgrad", 1024, 12288, 4096, 1),
    ("wgrad", 16173, 64, 4096, 2),   # a long stream in eight block slots (swapped 128 x 64 tiles)
    ("router_fwd", 1024, 256, 4096, 1), ("router_wgrad", 1024, 256, 4096, 1)])
def test_blocks_per_stage_rule(op, T, N, K, kps):
    """Two contraction blocks per ring stage except for long streams (units of >= 48
    blocks, at most three per SM) in rings of fewer than eight block slots, and the
    BF16x3 program."""
    assert dp.plan(op, T, N, K, sm_count=SM, out_f32=op.startswith("router"))["blocks_per_stage"] == kps


def test_blocks_per_stage_override(monkeypatch):
    monkeypatch.setenv("DP_FORCE_KPS", "1")
    assert dp.plan("fwd", 16384, 12288, 4096, sm_count=SM)["blocks_per_stage"] == 1
    monkeypatch.setenv("DP_FORCE_KPS", "2")
    assert dp.plan("wgrad", 16173, 128, 4096, sm_count=SM)["blocks_per_stage"] == 2
    # the BF16x3 program keeps one block per stage; the co-scheduled backward takes it too
    assert dp.plan("router_fwd", 1024, 256, 4096, sm_count=SM, out_f32=True)["blocks_per_stage"] == 1
    b = dp.plan_bwd(1024, 1024, 4096, sm_count=SM)
    assert b["fused"] == 1 and b["blocks_per_stage"] == 2
    monkeypatch.setenv("DP_FORCE_KPS", "1")
    assert dp.plan_bwd(1024, 1024, 4096, sm_count=SM)["blocks_per_stage"] == 1


@pytest.mark.parametrize("T,N,K,swap", [(16173, 64, 4096, 1), (16173, 48, 5120, 1), (16173, 128, 4096, 0),
                                        (1025, 64, 4096, 0), (65537, 64, 4096, 0)])
def test_thin_stream_orientation(T, N, K, swap):
    """N <= 64 over a long contraction takes the swapped 128 x 64 tiles, whose ring has
    eight block slots, where that plan keeps one wave; short contractions and
    plans that would need a second wave keep N as the tile rows."""
    p = dp.plan("wgrad", T, N, K, sm_count=SM)
    assert p["swap_ab"] == swap
    if swap:
        assert p["block_n"] == 64 and p["cta_pair"] == 0 and p["units"] <= SM and p["blocks_per_stage"] == 2


def test_test_helpers_cover_every_tile_and_block():
    # the GPU tests' samplers: raster_tile visits every tile of a plan exactly once,
    # stratified_points puts its points in every block and inside the matrix
    import numpy as np
    from gpu_common import raster_tile, stratified_points
    for op, T, N, K in (("fwd", 16384, 12288, 4096), ("dgrad", 16231, 12288, 4096), ("wgrad", 16384, 12288, 4096),
                        ("wgrad", 65537, 64, 4096), ("fwd", 300, 200, 64)):
        p = dp.plan(op, T, N, K, sm_count=SM)
        seen = {raster_tile(p, t) for t in range(p["tiles"])}
        assert len(seen) == p["tiles"] == p["tiles_m"] * p["tiles_n"]
        assert all(0 <= tm < p["tiles_m"] and 0 <= tn < p["tiles_n"] for tm, tn in seen)
    rng = np.random.default_rng(0)
    for R, C in ((16231, 4096), (64, 4096), (130, 129)):
        r, c = stratified_points((R, C), rng)
        assert r.min() >= 0 and c.min() >= 0 and r.max() < R and c.max() < C
        blocks = set(zip((r // 128).tolist(), (c // 128).tolist()))
        assert len(blocks) == (-(-R // 128)) * (-(-C // 128))
        assert r.size == 8 * len(blocks)
