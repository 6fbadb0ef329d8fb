"""Parity of the CUDA library with the CPU oracle, through the C-ABI (GPU only).

Every case draws seeded inputs from ``workloads.py``, runs the library through
``tpgemm_gemm`` / ``tpgemm_gemm_path`` and compares element by element with
the oracle on the same 16-bit patterns. The bar (the synchronous gemm page,
"TVM TIRx 同步 GEMM 深度解析", validates D = A.B within a tolerance; the bound
used here is): bit-exact (by value) when every input is integer-valued, else
|D - D_ref| <= 2^-10 * sum_k |a b| + 1e-6 elementwise.

Coverage follows the page's test section: the single-atom demo, tilings x
(dtype, beta) including ragged and 8-wide K tails, all four transpose combos
x both dtypes, plus the in-place form (C position = D), beta = 0 ignoring C,
guard bands around D, and the five workloads at their full sizes (every
element against the oracle's whole output).
"""
import dataclasses
import re
import itertools
import os
import sys

import numpy as np
import pytest
import torch

import oracle
import tile_primitive_tensor_gb300 as tp
import workloads as wl

pytestmark = pytest.mark.gpu

AUTO, TC, MMA = tp.TPGEMM_PATH_AUTO, tp.TPGEMM_PATH_TCGEN05, tp.TPGEMM_PATH_MMA_SYNC
GUARD = 4096  # floats of NaN canary on each side of D


@pytest.fixture(scope="module", autouse=True)
def _setup():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tile_primitive_tensor_gb300 import build as tpbuild
    tpbuild.build()
    oracle.build()
    yield
    assert tp.tpgemm_last_device_error() == tp.TPGEMM_OK, tp.tpgemm_last_error_detail()


def device_inputs(w, c_fill=None):
    A, B, C = wl.make_inputs(w, c_fill=c_fill)
    return (A, B, C), (A.cuda(), B.cuda(), None if C is None else C.cuda())


def run_gpu(w, Ad, Bd, Cd, path, D=None):
    """Run the library; returns D on the host. D is carved from a canary buffer."""
    n = w.M * w.N
    if D is None:
        buf = torch.full((n + 2 * GUARD,), float("nan"), dtype=torch.float32, device="cuda")
        D = buf[GUARD:GUARD + n].view(w.M, w.N)
    else:
        buf = None
    st = tp.tpgemm_gemm_path(D, Ad, Bd, Cd, w.M, w.N, w.K, w.transA, w.transB,
                             w.dtype, w.beta, None, path)
    assert st == tp.TPGEMM_OK, tp.tpgemm_last_error_detail()
    torch.cuda.synchronize()
    if buf is not None:
        h = buf.cpu().numpy()
        assert np.isnan(h[:GUARD]).all() and np.isnan(h[GUARD + n:]).all(), "write outside D"
    return D.cpu().numpy()


def oracle_full(w, A, B, C):
    return oracle.gemm(wl.bits(A), wl.bits(B), None if C is None else C.numpy(), w.M, w.N, w.K,
                       w.transA, w.transB, w.dtype, w.beta)


def check_full(w, path, c_fill=None):
    (A, B, C), (Ad, Bd, Cd) = device_inputs(w, c_fill=c_fill)
    D = run_gpu(w, Ad, Bd, Cd, path)
    Dref, S = oracle_full(w, A, B, C if w.beta else None)
    ok, msg = oracle.compare(D, Dref, S, exact=w.integer_valued)
    assert ok, f"{w.name} path={path}: {msg}"
    return D


# --------------------------------------------------------------- the atom
@pytest.mark.parametrize("path", [AUTO, MMA, TC])
def test_single_atom_bit_exact(path):
    w = wl.WORKLOADS[0]
    D = check_full(w, path)
    here = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
    sys.path.insert(0, here)
    import make_golden
    g = make_golden.read_case(os.path.join(here, f"{w.name}.txt"))
    assert np.array_equal(D, g["D_f32bits"])


@pytest.mark.parametrize("path", [MMA, TC])
def test_golden_ragged_fixture(path):
    here = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
    sys.path.insert(0, here)
    import make_golden
    w = make_golden.CASES[1][0]
    g = make_golden.read_case(os.path.join(here, f"{w.name}.txt"))
    (A, B, C), (Ad, Bd, Cd) = device_inputs(w)
    D = run_gpu(w, Ad, Bd, Cd, path)
    _, S = oracle_full(w, A, B, C)
    ok, msg = oracle.compare(D, g["D_f32bits"], S)
    assert ok, msg


# ------------------------------------------------------- tilings x modes
TILED_M = [16, 64, 144, 256]
TILED_N = [8, 16, 264]
TILED_K = [8, 24, 72]
MODES = [(wl.F16, 0.0), (wl.F16, 1.0), (wl.BF16, 0.0), (wl.BF16, 1.0)]


@pytest.mark.parametrize("path", [MMA, TC])
@pytest.mark.parametrize("dtype,beta", MODES)
def test_tiled_grid(path, dtype, beta):
    base = wl.BY_NAME["gemm_256_bf16_transB_beta1"]
    for i, (M, N, K) in enumerate(itertools.product(TILED_M, TILED_N, TILED_K)):
        w = base.with_shape(M, N, K, seed=5000 + i)
        w = dataclasses.replace(w, dtype=dtype, beta=beta, transB=False,
                                c_dist=("normal", 0.0, 1.0) if beta else None)
        check_full(w, path)


@pytest.mark.parametrize("path", [MMA, TC])
@pytest.mark.parametrize("dtype", [wl.F16, wl.BF16])
@pytest.mark.parametrize("tA,tB", list(itertools.product([False, True], repeat=2)))
def test_transpose_combos(path, dtype, tA, tB):
    base = wl.BY_NAME["gemm_256_bf16_transB_beta1"]
    w = base.with_shape(272, 392, 200, seed=6000 + 2 * tA + tB)
    w = dataclasses.replace(w, dtype=dtype, transA=tA, transB=tB)
    check_full(w, path)


@pytest.mark.parametrize("dtype", [wl.F16, wl.BF16])
@pytest.mark.parametrize("tA,tB", list(itertools.product([False, True], repeat=2)))
def test_transpose_combos_single_cta(dtype, tA, tB, tune):
    # The one-CTA-per-tile tcgen05 path (the default uses CTA pairs here).
    tune.setenv("TPGEMM_TC_PAIR", "0")
    base = wl.BY_NAME["gemm_256_bf16_transB_beta1"]
    w = base.with_shape(272, 392, 200, seed=6050 + 2 * tA + tB)
    w = dataclasses.replace(w, dtype=dtype, transA=tA, transB=tB)
    check_full(w, TC)


@pytest.mark.parametrize("tA,tB", list(itertools.product([False, True], repeat=2)))
def test_transpose_combos_swapped_orientation(tA, tB):
    # Small M with wide N runs the tcgen05 kernel in its swapped orientation.
    base = wl.BY_NAME["skinny_144x16392x4104_f16_beta1"]
    w = base.with_shape(48, 1544, 264, seed=6100 + 2 * tA + tB)
    w = dataclasses.replace(w, transA=tA, transB=tB)
    check_full(w, TC)


def test_multi_tile_waves_tc():
    # More tiles than SMs (several persistent waves), ragged in M, N and K.
    base = wl.BY_NAME["gemm_8192_bf16_transB_beta1"]
    w = base.with_shape(2320, 2600, 520, seed=6200)
    check_full(w, TC)


@pytest.mark.parametrize("case", ["normal_kmajor", "normal_mnmajor", "swapped"])
def test_single_cta_plans(case, tune):
    # With the CTA pair off every CTA is its own cluster and loads the whole Q
    # tile itself (no plan shares a tile between CTAs), including a P-tile
    # count that is odd.
    tune.setenv("TPGEMM_TC_PAIR", "0")
    if case == "swapped":
        w = dataclasses.replace(wl.BY_NAME["skinny_144x16392x4104_f16_beta1"].with_shape(
            128, 1416, 520, seed=6272))
    else:
        w = dataclasses.replace(wl.BY_NAME["gemm_8192_bf16_transB_beta1"].with_shape(
            656, 536, 392, seed=6282), transB=(case == "normal_kmajor"))
    st, text = tp.tpgemm_describe_plan(w.M, w.N, w.K, w.transA, w.transB, w.dtype, w.beta)
    assert st == tp.TPGEMM_OK and " cluster=1 pair=0 " in text, text
    check_full(w, TC)


def test_small_m_mn_major_q_runs_unclustered():
    # Small M with A stored [K, M]: the only Q tile is MN-contiguous and 144
    # wide, too narrow to split between a pair, so the plan runs one CTA per
    # cluster (earlier builds shared that tile between CTAs by multicast).
    w = dataclasses.replace(wl.BY_NAME["skinny_144x16392x4104_f16_beta1"].with_shape(
        144, 2064, 264, seed=6290), transA=True)
    st, text = tp.tpgemm_describe_plan(w.M, w.N, w.K, w.transA, w.transB, w.dtype, w.beta)
    assert st == tp.TPGEMM_OK and " cluster=1 " in text, text
    check_full(w, TC)


@pytest.mark.parametrize("case", ["normal_kmajor", "normal_mnmajor", "normal_odd_tiles",
                                  "swapped", "swapped_transA"])
@pytest.mark.parametrize("dtype", [wl.F16, wl.BF16])
def test_cta_pair_mma(case, dtype, tune):
    # CTA-pair MMA (cta_group::2, M = 256 per pair): each CTA loads its own 128
    # P rows and half of the Q tile; the pair's leader issues the MMA.
    tune.setenv("TPGEMM_TC_PAIR", "1")
    tune.setenv("TPGEMM_TC_BN", "128")
    base = wl.BY_NAME["gemm_8192_bf16_transB_beta1"]
    if case == "normal_kmajor":
        w = base.with_shape(512, 384, 328, seed=6300)
    elif case == "normal_mnmajor":
        w = dataclasses.replace(base.with_shape(512, 384, 328, seed=6301), transB=False)
    elif case == "normal_odd_tiles":
        w = dataclasses.replace(base.with_shape(656, 264, 200, seed=6302), transA=True)
    elif case == "swapped":
        w = base.with_shape(128, 1000, 264, seed=6303)
    else:
        w = dataclasses.replace(base.with_shape(128, 1000, 264, seed=6304), transA=True,
                                transB=False)
    w = dataclasses.replace(w, dtype=dtype)
    st, text = tp.tpgemm_describe_plan(w.M, w.N, w.K, w.transA, w.transB, w.dtype, w.beta, TC)
    assert "pair=1" in text, text
    check_full(w, TC)


@pytest.mark.parametrize("bn,tB", [(256, True), (256, False), (224, False), (224, True),
                                   (160, False)])
def test_cta_pair_full_width(bn, tB, tune):
    # Pair tiles up to 256 x 256 (two 256-column accumulators per CTA), with
    # MN-contiguous Q halves that are not whole 64-row atoms (224, 160).
    tune.setenv("TPGEMM_TC_PAIR", "1")
    tune.setenv("TPGEMM_TC_BN", str(bn))
    base = wl.BY_NAME["gemm_8192_bf16_transB_beta1"]
    w = dataclasses.replace(base.with_shape(768, 1056, 456, seed=6310 + bn), transB=tB)
    st, text = tp.tpgemm_describe_plan(w.M, w.N, w.K, w.transA, w.transB, w.dtype, w.beta, TC)
    assert "pair=1" in text, text
    check_full(w, TC)


@pytest.mark.parametrize("M,N,pair", [(2048, 2560, "1"), (2320, 2600, "1"), (2320, 2328, "0")])
@pytest.mark.parametrize("tB", [False, True])
def test_tail_wave_split(M, N, pair, tB, tune):
    # More work items than clusters, so the last wave's tiles are split along
    # N into 2 or 4 narrower units (the plan text shows "units=full+rem x split").
    tune.setenv("TPGEMM_TC_PAIR", pair)
    tune.setenv("TPGEMM_TC_BN", "256")
    tune.setenv("TPGEMM_TC_SK", "0")  # the tail split, not stream-K
    base = wl.BY_NAME["gemm_8192_bf16_transB_beta1"]
    w = dataclasses.replace(base.with_shape(M, N, 136, seed=6330 + M), transB=tB)
    st, text = tp.tpgemm_describe_plan(w.M, w.N, w.K, w.transA, w.transB, w.dtype, w.beta, TC)
    assert "x1 " not in text.split("units=")[1][:12], text
    check_full(w, TC)


@pytest.mark.parametrize("pair", ["0", "1"])
@pytest.mark.parametrize("tA,tB", list(itertools.product([False, True], repeat=2)))
def test_swapped_orientation_large(tA, tB, pair, tune):
    # P = B^T, Q = A for a problem with many tiles along both, D written back
    # transposed by the epilogue (the orientation used for B stored [K, N]).
    tune.setenv("TPGEMM_TC_ORIENT", "swap")
    tune.setenv("TPGEMM_TC_PAIR", pair)
    base = wl.BY_NAME["gemm_4096_f16"]
    w = dataclasses.replace(base.with_shape(784, 1320, 264, seed=6340 + 2 * tA + tB),
                            transA=tA, transB=tB, beta=1.0, c_dist=("normal", 0.0, 1.0))
    st, text = tp.tpgemm_describe_plan(w.M, w.N, w.K, w.transA, w.transB, w.dtype, w.beta, TC)
    assert "orientation=swapped" in text, text
    check_full(w, TC)


@pytest.mark.parametrize("pair", ["0", "1"])
def test_normal_orientation_mn_contiguous_q(pair, tune):
    # A [M,K] and B [K,N] default to the swapped orientation; the normal one,
    # with an MN-contiguous Q operand, stays correct when forced.
    tune.setenv("TPGEMM_TC_ORIENT", "normal")
    tune.setenv("TPGEMM_TC_PAIR", pair)
    base = wl.BY_NAME["gemm_4096_f16"]
    w = dataclasses.replace(base.with_shape(784, 1320, 264, seed=6350), beta=1.0,
                            c_dist=("normal", 0.0, 1.0))
    st, text = tp.tpgemm_describe_plan(w.M, w.N, w.K, w.transA, w.transB, w.dtype, w.beta, TC)
    assert "orientation=normal" in text and "q_major=mn" in text, text
    check_full(w, TC)


@pytest.mark.parametrize("case", [
    ("swap_small", 144, 4104, 1160, False, False, 1.0, "1"),
    ("swap_small_transA", 144, 4104, 1160, True, False, 0.0, "1"),
    ("normal_chain", 1024, 1024, 2048, False, True, 1.0, "1"),
    ("normal_chain_beta0", 1024, 1024, 2048, True, True, 0.0, "1"),
    ("swapped_large", 1024, 1024, 2048, False, False, 1.0, "1"),
    ("one_cta", 1024, 1024, 2048, False, True, 1.0, "0"),
    ("ragged_odd_k", 1040, 1000, 2056, False, True, 1.0, "1"),  # partial edge tiles, 33 K blocks
    ("ragged_nn_beta0", 1008, 1304, 1096, False, False, 0.0, "1"),
], ids=lambda c: c[0])
def test_stream_k(case, tune):
    # Each leftover work item split into two K halves on two clusters: the
    # first zeroes the tile's D region at kernel start, both add into it with
    # TMA reductions (the first with beta.C).
    name, M, N, K, tA, tB, beta, pair = case
    tune.setenv("TPGEMM_TC_PAIR", pair)
    tune.setenv("TPGEMM_TC_SK", "1")
    base = wl.BY_NAME["gemm_256_bf16_transB_beta1"]
    w = dataclasses.replace(base.with_shape(M, N, K, seed=6370 + M + K), transA=tA, transB=tB,
                            beta=beta, c_dist=("normal", 0.0, 1.0) if beta else None)
    st, text = tp.tpgemm_describe_plan(w.M, w.N, w.K, w.transA, w.transB, w.dtype, w.beta, TC)
    assert "stream_k=1" in text, text
    rem = int(re.search(r"units=(\d+)\+(\d+)x", text).group(2))
    assert f"sk_clusters={2 * rem}" in text, text
    D1 = check_full(w, TC)
    # Deterministic: a second launch (next epoch) gives the same bits.
    (A, B, C), (Ad, Bd, Cd) = device_inputs(w)
    D2 = run_gpu(w, Ad, Bd, Cd, TC)
    assert np.array_equal(D1.view(np.uint32), D2.view(np.uint32))


@pytest.mark.parametrize("case", [
    # name, workload, M, N, K, tA, tB, beta, pair, extra overrides
    ("pair_kmajor_ragged_k", "gemm_4096_f16_int", 1024, 1024, 1032, False, True, 1.0, "1", {}),
    ("pair_swapped_beta0", "gemm_4096_f16_int", 1024, 1040, 2056, False, False, 0.0, "1", {}),
    ("one_cta_rotated", "gemm_4096_f16_int", 1024, 1024, 1096, False, True, 1.0, "0",
     {"TPGEMM_TC_KROTATE": "3", "TPGEMM_TC_SK": "0"}),
    ("pair_n_split_tail", "gemm_4096_f16_int", 1040, 1000, 1032, True, True, 1.0, "1",
     {"TPGEMM_TC_SK": "0"}),
    ("pair_fp8", "gemm_4096_e4m3_int_transB", 1024, 1280, 1040, False, True, 0.0, "1", {}),
    ("pair_random_bf16", "gemm_256_bf16_transB_beta1", 1024, 1024, 1032, False, True, 1.0, "1", {}),
], ids=lambda c: c[0])
@pytest.mark.parametrize("krev", ["0", "1"])
def test_k_direction(case, krev, tune):
    # With k_reverse a cluster's second, fourth, ... unit walks its K blocks
    # backwards. Six clusters give each one several units, so both directions
    # run in one launch. Integer-valued inputs make every order of the sum give
    # the same value, so those results must equal the oracle's exactly.
    name, base_name, M, N, K, tA, tB, beta, pair, extra = case
    tune.setenv("TPGEMM_TC_PAIR", pair)
    tune.setenv("TPGEMM_TC_MAX_CLUSTERS", "6")
    tune.setenv("TPGEMM_TC_KREV", krev)
    for k, v in extra.items():
        tune.setenv(k, v)
    base = wl.BY_NAME[base_name]
    w = dataclasses.replace(base.with_shape(M, N, K, seed=6410 + M + K), transA=tA, transB=tB,
                            beta=beta,
                            c_dist=(("int", -3, 3) if base.integer_valued else
                                    ("normal", 0.0, 1.0)) if beta else None)
    st, text = tp.tpgemm_describe_plan(w.M, w.N, w.K, w.transA, w.transB, w.dtype, w.beta, TC)
    assert f"k_reverse={krev}" in text, text
    if "TPGEMM_TC_KROTATE" in extra:
        assert f"k_rotate={extra['TPGEMM_TC_KROTATE']}" in text, text
    units = re.search(r"units=(\d+)\+(\d+)x(\d+)", text)
    whole = int(units.group(1))
    grid = int(re.search(r"grid=(\d+)", text).group(1))
    assert whole >= 2 * (grid // (2 if pair == "1" else 1)), text  # a second wave exists
    check_full(w, TC)


@pytest.mark.parametrize("case", [
    # name, workload, M, N, K, tA, tB, beta, extra overrides
    ("whole_units_beta1", "gemm_4096_f16_int", 1024, 1024, 1032, False, True, 1.0,
     {"TPGEMM_TC_MAX_CLUSTERS": "6"}),
    ("swapped_beta0", "gemm_4096_f16_int", 1024, 1040, 2056, False, False, 0.0,
     {"TPGEMM_TC_MAX_CLUSTERS": "6"}),
    ("stream_k_halves_beta1", "gemm_4096_f16_int", 1040, 1000, 2056, False, True, 1.0,
     {"TPGEMM_TC_SK": "1"}),
    ("stream_k_halves_beta0", "gemm_4096_f16_int", 1008, 1304, 1096, False, False, 0.0,
     {"TPGEMM_TC_SK": "1"}),
    ("n_split_tail_ragged", "gemm_4096_f16_int", 1040, 1000, 1032, True, True, 1.0,
     {"TPGEMM_TC_SK": "0", "TPGEMM_TC_MAX_CLUSTERS": "6"}),
    ("odd_chunks_one_cta", "gemm_4096_f16_int", 1024, 1000, 1032, False, True, 1.0,
     {"TPGEMM_TC_PAIR": "0", "TPGEMM_TC_BN": "224", "TPGEMM_TC_MAX_CLUSTERS": "6"}),
    ("fp8", "gemm_4096_e4m3_int_transB", 1024, 1280, 1040, False, True, 1.0,
     {"TPGEMM_TC_MAX_CLUSTERS": "6"}),
], ids=lambda c: c[0])
@pytest.mark.parametrize("help_", ["0", "1"])
def test_last_segment_helpers(case, help_, tune):
    # In a one-group plan warps 6..9 take the odd 32-column chunks of each
    # CTA's last segment, staged through the TMA ring; with C they load it
    # there themselves. Integer-valued inputs: the result must equal the
    # oracle's exactly, with the helpers and without.
    name, base_name, M, N, K, tA, tB, beta, extra = case
    for k, v in extra.items():
        tune.setenv(k, v)
    tune.setenv("TPGEMM_TC_EPI_HELP", help_)
    base = wl.BY_NAME[base_name]
    w = dataclasses.replace(base.with_shape(M, N, K, seed=6470 + M + K), transA=tA, transB=tB,
                            beta=beta, c_dist=("int", -3, 3) if beta else None)
    st, text = tp.tpgemm_describe_plan(w.M, w.N, w.K, w.transA, w.transB, w.dtype, w.beta, TC)
    assert "epi_groups=1" in text and f"epi_help={help_}" in text, text
    if extra.get("TPGEMM_TC_SK") == "1":
        assert "stream_k=1" in text, text
    D1 = check_full(w, TC)
    assert f"epi_help={help_}" in tp.tpgemm_last_plan()[1]
    # A second launch (stream-K: the next flag epoch) gives the same bits.
    (A, B, C), (Ad, Bd, Cd) = device_inputs(w)
    D2 = run_gpu(w, Ad, Bd, Cd, TC)
    assert np.array_equal(D1.view(np.uint32), D2.view(np.uint32))


@pytest.mark.parametrize("case", [
    ("skinny_swap_pair", 144, 2072, 520, False, False, 1.0, {"TPGEMM_TC_PAIR": "1"}),
    ("normal_beta1_one_buf", 1024, 1024, 2048, False, True, 1.0, {}),
    ("normal_beta0_one_buf", 1024, 1024, 520, True, True, 0.0, {}),
    ("swapped_beta0", 784, 1320, 264, False, False, 0.0, {"TPGEMM_TC_ORIENT": "swap"}),
    ("odd_bufs_reload", 1024, 1024, 264, False, True, 1.0, {"TPGEMM_TC_EPI_BUFS": "3"}),
    ("tail_split", 2048, 2560, 136, False, True, 1.0, {"TPGEMM_TC_BN": "256", "TPGEMM_TC_SK": "0"}),
    ("stream_k", 1024, 1024, 2048, False, True, 1.0, {"TPGEMM_TC_SK": "1"}),
    ("one_cta", 784, 1320, 264, False, True, 1.0, {"TPGEMM_TC_PAIR": "0"}),
], ids=lambda c: c[0])
def test_epilogue_groups(case, tune):
    # One or two epilogue warpgroups: the second splits each lane quadrant's
    # 32-column chunks (and its staging tiles) with the first. The K order is
    # the same, so both give the same bits; each is checked against the oracle.
    name, M, N, K, tA, tB, beta, env = case
    for k, v in env.items():
        tune.setenv(k, v)
    base = wl.BY_NAME["gemm_256_bf16_transB_beta1"]
    w = dataclasses.replace(base.with_shape(M, N, K, seed=6390 + M + K), transA=tA, transB=tB,
                            beta=beta, c_dist=("normal", 0.0, 1.0) if beta else None)
    out = []
    for g in ("1", "2"):
        tune.setenv("TPGEMM_TC_EPI_GROUPS", g)
        st, text = tp.tpgemm_describe_plan(w.M, w.N, w.K, w.transA, w.transB, w.dtype, w.beta, TC)
        assert f"epi_groups={g}" in text, text
        out.append(check_full(w, TC))
    assert np.array_equal(out[0].view(np.uint32), out[1].view(np.uint32))


def test_cta_pair_skinny_m144(tune):
    tune.setenv("TPGEMM_TC_PAIR", "1")
    w = wl.BY_NAME["skinny_144x16392x4104_f16_beta1"].with_shape(144, 2072, 520, seed=6320)
    st, text = tp.tpgemm_describe_plan(w.M, w.N, w.K, w.transA, w.transB, w.dtype, w.beta, TC)
    assert "pair=1" in text, text
    check_full(w, TC)


@pytest.mark.parametrize("pair", ["0", "1"])
@pytest.mark.parametrize("bn", [32, 128, 160, 192, 224, 256])
@pytest.mark.parametrize("tB", [False, True])
def test_every_tile_width(bn, tB, pair, tune):
    # Each accumulator width the planner may choose, with B K- or MN-contiguous,
    # on one CTA per tile and on CTA pairs.
    tune.setenv("TPGEMM_TC_BN", str(bn))
    tune.setenv("TPGEMM_TC_PAIR", pair)
    base = wl.BY_NAME["gemm_4096_f16"]
    w = dataclasses.replace(base.with_shape(400, 1000, 264, seed=6250 + bn), transB=tB,
                            beta=1.0, c_dist=("normal", 0.0, 1.0))
    check_full(w, TC)


def test_integer_bit_exact_tc_multi_tile():
    base = wl.WORKLOAD_4096_INT
    w = base.with_shape(400, 520, 1032, seed=6300)
    check_full(w, TC)
    check_full(w, MMA)


# ------------------------------------------------------------ edge cases
@pytest.mark.parametrize("path", [MMA, TC])
def test_beta_zero_never_reads_c(path):
    w = wl.BY_NAME["gemm_4096_f16"].with_shape(144, 264, 72, seed=6400)
    (A, B, _), (Ad, Bd, _) = device_inputs(w)
    Cnan = torch.full((w.M, w.N), float("nan"), device="cuda")
    D = run_gpu(w, Ad, Bd, Cnan, path)
    Dref, S = oracle_full(w, A, B, None)
    ok, msg = oracle.compare(D, Dref, S)
    assert ok, msg


@pytest.mark.parametrize("path", [MMA, TC])
def test_in_place_d_equals_c(path):
    w = wl.BY_NAME["gemm_256_bf16_transB_beta1"].with_shape(272, 392, 200, seed=6500)
    (A, B, C), (Ad, Bd, Cd) = device_inputs(w)
    D = run_gpu(w, Ad, Bd, Cd, path, D=Cd)
    Dref, S = oracle_full(w, A, B, C)
    ok, msg = oracle.compare(D, Dref, S)
    assert ok, msg


@pytest.mark.parametrize("bp", ["112", "80"])
def test_stream_k_half_quadrant(bp, tune):
    # P tiles of 112 or 80 rows: one lane quadrant holds 16 of the tile's rows
    # and reduces (and zero-fills) through the half-width D map.
    tune.setenv("TPGEMM_TC_BP", bp)
    tune.setenv("TPGEMM_TC_SK", "1")
    base = wl.BY_NAME["skinny_144x16392x4104_f16_beta1"]
    w = base.with_shape(144, 4104, 1160, seed=6380 + int(bp))
    st, text = tp.tpgemm_describe_plan(w.M, w.N, w.K, w.transA, w.transB, w.dtype, w.beta, TC)
    assert f"tile={bp}x" in text and "stream_k=1" in text, text
    check_full(w, TC)


def test_graph_capture_replays_take_no_stream_k():
    # A launch captured into a CUDA graph keeps its stream-K flag epoch, and a
    # replay would find the flags already at that value; so a call on a
    # capturing stream plans the split along N. Outside the capture the same
    # shape runs stream-K. Three replays each match the oracle.
    w = wl.BY_NAME["gemm_256_bf16_transB_beta1"].with_shape(1024, 1024, 2048, seed=6520)
    (A, B, C), (Ad, Bd, Cd) = device_inputs(w)
    D = torch.empty(w.M, w.N, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        st = tp.tpgemm_gemm_path(D, Ad, Bd, Cd, w.M, w.N, w.K, w.transA, w.transB, w.dtype,
                                 w.beta, None, TC)
        assert st == tp.TPGEMM_OK, tp.tpgemm_last_error_detail()
    torch.cuda.synchronize()
    assert "stream_k=1" in tp.tpgemm_last_plan()[1]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        st = tp.tpgemm_gemm_path(D, Ad, Bd, Cd, w.M, w.N, w.K, w.transA, w.transB, w.dtype,
                                 w.beta, None, TC)
    assert st == tp.TPGEMM_OK, tp.tpgemm_last_error_detail()
    assert "stream_k=0" in tp.tpgemm_last_plan()[1], tp.tpgemm_last_plan()[1]
    Dref, S = oracle_full(w, A, B, C)
    for _ in range(3):
        D.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        ok, msg = oracle.compare(D.cpu().numpy(), Dref, S)
        assert ok, msg
    assert tp.tpgemm_last_device_error() == tp.TPGEMM_OK


def test_in_place_takes_the_n_split_not_stream_k():
    # 1024^2 x 2048 (16 pair tiles, one partial wave) would split each tile
    # into two K halves whose first zeroes D at kernel start; in place (D ==
    # C) that would erase C, so the call takes the split along N and the
    # result still matches the oracle. The same shape out of place runs
    # stream-K.
    w = wl.BY_NAME["gemm_256_bf16_transB_beta1"].with_shape(1024, 1024, 2048, seed=6510)
    st, text = tp.tpgemm_describe_plan(w.M, w.N, w.K, w.transA, w.transB, w.dtype, w.beta, TC)
    assert "stream_k=1" in text, text
    (A, B, C), (Ad, Bd, Cd) = device_inputs(w)
    D = run_gpu(w, Ad, Bd, Cd, TC, D=Cd)
    st, plan = tp.tpgemm_last_plan()
    assert "stream_k=0" in plan, plan
    Dref, S = oracle_full(w, A, B, C)
    ok, msg = oracle.compare(D, Dref, S)
    assert ok, msg


@pytest.mark.parametrize("path", [MMA, TC])
def test_identity_bit_exact_real_data(path):
    # A = I  =>  D = fp32(B) exactly, for any real B (the oracle pin, now on the GPU).
    n, N = 208, 136
    for dtype in (wl.F16, wl.BF16):
        td = wl.torch_dtype(dtype)
        g = torch.Generator().manual_seed(77)
        Bh = torch.randn(n, N, generator=g).to(td)
        I = torch.eye(n).to(td)
        D = torch.empty(n, N, device="cuda")
        st = tp.tpgemm_gemm_path(D, I.cuda(), Bh.cuda(), None, n, N, n, 0, 0, dtype, 0.0, None,
                                 path)
        assert st == tp.TPGEMM_OK, tp.tpgemm_last_error_detail()
        assert torch.equal(D.cpu(), Bh.float())


def test_rejects_misaligned_device_pointers():
    A = torch.zeros(64 * 64 + 8, dtype=torch.float16, device="cuda")
    B = torch.zeros(64 * 64, dtype=torch.float16, device="cuda")
    D = torch.zeros(64 * 64, dtype=torch.float32, device="cuda")
    st = tp.tpgemm_gemm(D, A.data_ptr() + 2, B, None, 64, 64, 64, 0, 0, 0, 0.0, None)
    assert st == tp.TPGEMM_ERR_ALIGN


# -------------------------------------------- the five workloads, full size
@pytest.mark.parametrize("name", [w.name for w in wl.WORKLOADS] + ["gemm_4096_f16_int"])
def test_workload_full_size(name):
    # The five workloads at their full sizes, through tpgemm_gemm as the
    # benchmark calls it, against the oracle's whole output element by
    # element: bit-exact (by value) for the integer-valued ones, within the
    # bound otherwise. (8192^3 takes the oracle about half a minute on 16 cores.)
    w = wl.BY_NAME[name]
    (A, B, C), (Ad, Bd, Cd) = device_inputs(w)
    D = torch.empty(w.M, w.N, device="cuda")
    st = tp.tpgemm_gemm(D, Ad, Bd, Cd, w.M, w.N, w.K, w.transA, w.transB, w.dtype, w.beta, None)
    assert st == tp.TPGEMM_OK, tp.tpgemm_last_error_detail()
    torch.cuda.synchronize()
    Dh = D.cpu().numpy()
    del D, Ad, Bd, Cd
    Dref, S = oracle_full(w, A, B, C if w.beta else None)
    ok, msg = oracle.compare(Dh, Dref, S, exact=w.integer_valued)
    assert ok, f"{name}: {msg}"


# ------------------------------------------------------ host-buffer entry point
@pytest.mark.parametrize("M,N,K,tA,tB,beta", [
    (16, 8, 16, False, False, 0.0),       # one block, mma.sync
    (528, 392, 200, True, False, 1.0),    # 4 blocks of 144 (last 96), A column blocks
    (2320, 1000, 264, False, True, 1.0),  # edges of 512, 5 blocks of 256 and one of 16 between
    (4096, 520, 136, True, True, 0.0),    # edges of 512, 6 blocks of 512, A column blocks
])
def test_gemm_host_buffers(M, N, K, tA, tB, beta):
    check_host_buffers(M, N, K, tA, tB, beta)


@pytest.mark.parametrize("edge", ["0", "256"])
@pytest.mark.parametrize("M,N,K,tA,tB,beta", [
    (2320, 1000, 264, False, True, 1.0),
    (4096, 520, 136, True, True, 0.0),
])
def test_gemm_host_buffers_edge_blocks(M, N, K, tA, tB, beta, edge, tune):
    # Equal row blocks (no edge blocks), and edges of 256 rows.
    tune.setenv("TPGEMM_HOST_EDGE", edge)
    check_host_buffers(M, N, K, tA, tB, beta)


def check_host_buffers(M, N, K, tA, tB, beta):
    base = wl.BY_NAME["gemm_256_bf16_transB_beta1"]
    w = dataclasses.replace(base.with_shape(M, N, K, seed=6400 + M), transA=tA, transB=tB,
                            beta=beta, c_dist=("normal", 0.0, 1.0) if beta else None)
    A, B, C = wl.make_inputs(w)
    Ah, Bh = A.pin_memory(), B.pin_memory()
    Ch = None if C is None else C.pin_memory()
    Dh = torch.full((M, N), float("nan")).pin_memory()
    nbytes = tp.tpgemm_gemm_host_workspace_bytes(M, N, K, w.dtype, beta)
    ws = torch.full((nbytes // 4,), float("nan"), device="cuda")
    st = tp.tpgemm_gemm_host(Dh, Ah, Bh, Ch, M, N, K, tA, tB, w.dtype, beta, ws, nbytes, None)
    assert st == tp.TPGEMM_OK, tp.tpgemm_last_error_detail()
    torch.cuda.current_stream().synchronize()
    Dref, S = oracle_full(w, A, B, C)
    ok, msg = oracle.compare(Dh.numpy(), Dref, S)
    assert ok, msg


# ------------------------------------------------------- failure detection
@pytest.mark.parametrize("producers", ["1", "4"])
@pytest.mark.parametrize("case", ["one_cta", "pair", "swapped_small"])
def test_bounded_wait_reports_timeout_and_context_survives(case, producers, tune):
    tune.setenv("TPGEMM_TC_PRODUCERS", producers)
    # A stage fill that never arrives (no TMA is issued for it) must not hang
    # the GPU: the kernel's bounded wait expires, the status word is set, every
    # role stops, in-flight copies and MMAs drain, tensor memory is freed, and
    # the next call on the same context computes the right answer.
    if case == "one_cta":
        tune.setenv("TPGEMM_TC_PAIR", "0")
        w = wl.BY_NAME["gemm_8192_bf16_transB_beta1"].with_shape(512, 512, 256, seed=6360)
    elif case == "pair":
        w = wl.BY_NAME["gemm_8192_bf16_transB_beta1"].with_shape(512, 512, 256, seed=6361)
    else:
        w = wl.BY_NAME["skinny_144x16392x4104_f16_beta1"].with_shape(144, 1032, 264, seed=6362)
    (A, B, C), (Ad, Bd, Cd) = device_inputs(w)
    D = torch.zeros(w.M, w.N, device="cuda")
    assert tp.tpgemm_last_device_error() == tp.TPGEMM_OK
    tune.setenv("TPGEMM_WAIT_TIMEOUT_MS", "200")
    st = tp.tpgemm_test_gemm_withhold_fill(D, Ad, Bd, Cd, w.M, w.N, w.K, w.transA, w.transB,
                                           w.dtype, w.beta)
    assert st == tp.TPGEMM_OK, tp.tpgemm_last_error_detail()
    assert tp.tpgemm_last_device_error() == tp.TPGEMM_ERR_TIMEOUT
    assert tp.tpgemm_last_device_error() == tp.TPGEMM_OK  # reading it cleared it
    Dh = run_gpu(w, Ad, Bd, Cd, TC)
    Dref, S = oracle_full(w, A, B, C)
    ok, msg = oracle.compare(Dh, Dref, S)
    assert ok, msg
    assert tp.tpgemm_last_device_error() == tp.TPGEMM_OK


# ------------------------------------------------------------ extreme shapes
@pytest.mark.parametrize("case", [
    ("n8_tall", 8192, 8, 64, False, True, wl.BF16, 1.0, AUTO),
    ("n8_tall_tc", 8192, 8, 64, True, True, wl.F16, 0.0, TC),
    ("long_k_tiny", 16, 8, 65536, False, True, wl.F16, 0.0, AUTO),
    ("long_k_tc", 256, 256, 16384, True, False, wl.BF16, 1.0, AUTO),
    ("m16_wide_tc", 16, 16392, 520, False, False, wl.F16, 1.0, TC),
    ("k8_tc", 1024, 1024, 8, False, True, wl.BF16, 1.0, TC),
    ("m16_n131072", 16, 131072, 64, False, False, wl.F16, 1.0, TC),
    ("m65536_n16", 65536, 16, 128, True, True, wl.BF16, 1.0, TC),
], ids=lambda c: c[0])
def test_extreme_shapes(case):
    name, M, N, K, tA, tB, dtype, beta, path = case
    base = wl.BY_NAME["gemm_256_bf16_transB_beta1"]
    w = dataclasses.replace(base.with_shape(M, N, K, seed=7000 + M + N + K), transA=tA,
                            transB=tB, dtype=dtype, beta=beta,
                            c_dist=("normal", 0.0, 1.0) if beta else None)
    check_full(w, path)


# ------------------------------------------------- P rows per tile (bp < 128)
# Single-wave plans whose tiles share the one Q tile give each CTA bp < 128 P
# rows. Lanes bp .. 127 of the accumulator then hold results nobody stores; a
# lane quadrant half inside the tile (bp = 80, 112) uses the half-width C / D
# boxes, quadrants past bp are idle, and an MN-contiguous P tile is one full
# 64-row box plus a narrower one. Every combination is checked against the
# oracle; the last tile along P is ragged.
@pytest.mark.parametrize("bp", [64, 80, 96, 112, 128])
@pytest.mark.parametrize("orient,tA,tB", [
    ("swap", False, False),   # P = B^T MN-contiguous
    ("swap", False, True),    # P = B^T K-contiguous
    ("normal", False, True),  # P = A K-contiguous
    ("normal", True, True),   # P = A MN-contiguous
])
@pytest.mark.parametrize("beta", [0.0, 1.0])
def test_p_rows_per_tile(bp, orient, tA, tB, beta, tune):
    tune.setenv("TPGEMM_TC_ORIENT", orient)
    tune.setenv("TPGEMM_TC_BP", str(bp))
    M, N = (144, 1304) if orient == "swap" else (1040, 200)
    base = wl.BY_NAME["gemm_256_bf16_transB_beta1"]
    w = dataclasses.replace(base.with_shape(M, N, 264, seed=7100 + bp + int(tA) + 2 * int(tB)),
                            transA=tA, transB=tB, dtype=wl.F16, beta=beta,
                            c_dist=("normal", 0.0, 1.0) if beta else None)
    st, text = tp.tpgemm_describe_plan(w.M, w.N, w.K, w.transA, w.transB, w.dtype, w.beta, TC)
    assert st == tp.TPGEMM_OK and f"tile={bp}x" in text and f"orientation={'swapped' if orient == 'swap' else 'normal'}" in text, text
    check_full(w, TC)


@pytest.mark.parametrize("bp", [80, 112])
@pytest.mark.parametrize("pair", ["0", "1"])
def test_p_rows_integer_bit_exact_and_in_place(bp, pair, tune):
    # Integer-valued inputs: exact. Then D = C in place over the same plan.
    tune.setenv("TPGEMM_TC_BP", str(bp))
    tune.setenv("TPGEMM_TC_PAIR", pair)
    w = wl.WORKLOAD_4096_INT.with_shape(144, 2072, 520, seed=7200 + bp)
    st, text = tp.tpgemm_describe_plan(w.M, w.N, w.K, w.transA, w.transB, w.dtype, w.beta, TC)
    assert f"tile={bp}x" in text and f"pair={pair}" in text, text
    check_full(w, TC)
    w1 = dataclasses.replace(wl.BY_NAME["skinny_144x16392x4104_f16_beta1"].with_shape(
        144, 2072, 264, seed=7250 + bp))
    (A, B, C), (Ad, Bd, Cd) = device_inputs(w1)
    D = run_gpu(w1, Ad, Bd, Cd, TC, D=Cd)
    Dref, S = oracle_full(w1, A, B, C)
    ok, msg = oracle.compare(D, Dref, S)
    assert ok, msg


@pytest.mark.parametrize("bp", [64, 112])
@pytest.mark.parametrize("name", ["skinny_144x16392x4112_e4m3_transB_beta1"])
def test_p_rows_fp8(bp, name, tune):
    tune.setenv("TPGEMM_TC_BP", str(bp))
    w = wl.BY_NAME[name].with_shape(144, 2072, 528, seed=7300 + bp)
    st, text = tp.tpgemm_describe_plan(w.M, w.N, w.K, w.transA, w.transB, w.dtype, w.beta, TC)
    assert f"tile={bp}x" in text and "kind=f8f6f4" in text, text
    check_full(w, TC)


def test_p_rows_default_skinny_plan():
    # The planner's own choice for the 144 x 16392 x 4104 shape: 112 rows, one wave.
    st, text = tp.tpgemm_describe_plan(144, 16392, 4104, 0, 0, wl.F16, 1.0, TC)
    assert st == tp.TPGEMM_OK and "tile=112x144x64" in text and "grid=148" in text, text


# ------------------------------------------------ several TMA-issuing threads
# Fill g of the ring is issued by producer g % P (warp 0, then warps 6, 7, 8).
# The K order of the MMAs does not depend on P, so every P gives the same bits;
# each is also checked against the oracle. Cases: multi-wave with a tail split
# (one epilogue group: warps 6..8 only produce), single-wave with two epilogue
# groups (warps 6..8 produce, then run their epilogue), no CTA pair, stream-K,
# fp8 and a two-stage ring (P capped at the ring depth).
@pytest.mark.parametrize("case", [
    ("multi_wave_tail", "gemm_256_bf16_transB_beta1", 2048, 2560, 264,
     {"TPGEMM_TC_BN": "256", "TPGEMM_TC_SK": "0"}),
    ("single_wave_two_groups", "skinny_144x16392x4104_f16_beta1", 144, 4104, 520, {}),
    ("no_pair", "gemm_4096_f16", 784, 1320, 264, {"TPGEMM_TC_PAIR": "0"}),
    ("stream_k", "gemm_256_bf16_transB_beta1", 1024, 1024, 2048, {"TPGEMM_TC_SK": "1"}),
    ("fp8", "gemm_4096_e4m3_int_transB", 1024, 1536, 528, {}),
    ("two_stages", "gemm_4096_f16", 512, 768, 520, {"TPGEMM_TC_STAGES": "2"}),
], ids=lambda c: c[0])
def test_producer_counts(case, tune):
    name, wname, M, N, K, env = case
    for k, v in env.items():
        tune.setenv(k, v)
    w = wl.BY_NAME[wname].with_shape(M, N, K, seed=7400 + M + K)
    out = []
    for n in ("1", "2", "3", "4"):
        tune.setenv("TPGEMM_TC_PRODUCERS", n)
        st, text = tp.tpgemm_describe_plan(w.M, w.N, w.K, w.transA, w.transB, w.dtype, w.beta, TC)
        assert st == tp.TPGEMM_OK, text
        stages = int(text.split("stages=")[1].split()[0])
        assert f"producers={min(int(n), stages)}" in text, text
        out.append(check_full(w, TC))
    for D in out[1:]:
        assert np.array_equal(out[0].view(np.uint32), D.view(np.uint32))


# ---------------------------------------- back-to-back launches on one stream
# Each launch may start while the previous one drains (programmatic dependent
# launch). Its threads wait for the previous grid before their first global
# access: after set-up (dep_early = 0) or each just before it (dep_early = 1).
# Four in-place accumulations D += A.B issued back to back read the D the
# previous launch is still writing; integer inputs make D = C0 + 4 A.B exact.
@pytest.mark.parametrize("early", ["0", "1"])
@pytest.mark.parametrize("case", [
    ("skinny_single_wave", "skinny_144x16392x4104_f16_beta1", 144, 4104, 520),
    ("multi_wave", "gemm_4096_f16", 2320, 2600, 264),
    ("fp8", "gemm_4096_e4m3_int_transB", 1024, 1536, 528),
], ids=lambda c: c[0])
def test_chained_in_place_launches(case, early, tune):
    name, wname, M, N, K = case
    tune.setenv("TPGEMM_TC_DEP_EARLY", early)
    base = wl.BY_NAME[wname].with_shape(M, N, K, seed=7500 + M)
    w = dataclasses.replace(base, a_dist=("int", -3, 3), b_dist=("int", -3, 3),
                            c_dist=("int", -8, 8), beta=1.0)
    st, text = tp.tpgemm_describe_plan(w.M, w.N, w.K, w.transA, w.transB, w.dtype, w.beta, TC)
    assert st == tp.TPGEMM_OK and f"dep_early={early}" in text, text
    (A, B, C), (Ad, Bd, Cd) = device_inputs(w)
    D = Cd.clone()
    for _ in range(4):
        st = tp.tpgemm_gemm_path(D, Ad, Bd, D, w.M, w.N, w.K, w.transA, w.transB, w.dtype,
                                 1.0, None, TC)
        assert st == tp.TPGEMM_OK, tp.tpgemm_last_error_detail()
    torch.cuda.synchronize()
    w0 = dataclasses.replace(w, beta=0.0, c_dist=None)
    AB, S = oracle_full(w0, A, B, None)
    ok, msg = oracle.compare(D.cpu().numpy(), C.numpy() + 4.0 * AB, 4.0 * S, exact=True)
    assert ok, msg



# ------------------------------------------- several host threads, own streams
def test_concurrent_host_threads_own_streams():
    # Four host threads each run a different plan (tcgen05 pair, one CTA per
    # tile, the swapped skinny plan, mma.sync) five times on their own stream.
    # The library's caches are shared under its locks and the error detail is
    # per thread; every result is checked against the oracle.
    import concurrent.futures

    base = wl.BY_NAME["gemm_256_bf16_transB_beta1"]
    shapes = [(512, 512, 256, {}), (784, 1320, 264, {}), (144, 2072, 264, {}), (64, 64, 72, {})]
    works = []
    for i, (M, N, K, _) in enumerate(shapes):
        w = dataclasses.replace(base.with_shape(M, N, K, seed=7800 + i), transB=bool(i % 2),
                                beta=1.0, c_dist=("normal", 0.0, 1.0))
        (A, B, C), (Ad, Bd, Cd) = device_inputs(w)
        Dref, S = oracle_full(w, A, B, C)
        works.append((w, Ad, Bd, Cd, Dref, S))
    torch.cuda.synchronize()

    def run(idx):
        w, Ad, Bd, Cd, Dref, S = works[idx]
        stream = torch.cuda.Stream()
        outs = []
        with torch.cuda.stream(stream):
            for _ in range(5):
                D = torch.empty(w.M, w.N, device="cuda")
                st = tp.tpgemm_gemm(D, Ad, Bd, Cd, w.M, w.N, w.K, w.transA, w.transB, w.dtype,
                                    w.beta, stream)
                assert st == tp.TPGEMM_OK, tp.tpgemm_last_error_detail()
                outs.append(D)
        stream.synchronize()
        return [oracle.compare(D.cpu().numpy(), Dref, S) for D in outs]

    with concurrent.futures.ThreadPoolExecutor(4) as ex:
        results = list(ex.map(run, range(len(works))))
    for res in results:
        for ok, msg in res:
            assert ok, msg
    assert tp.tpgemm_last_device_error() == tp.TPGEMM_OK
