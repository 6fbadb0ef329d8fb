"""The planner's rules, checked on the host (no GPU).

tpgemm_describe_plan plans a problem as tpgemm_gemm would on a 152-SM GB300
(the persistent grid is one CTA, or CTA pair, per SM or SM pair), so every rule
the kernels depend on can be checked here over a sweep of shapes, without a
launch. Each test states the rule and checks the plan string against it; the
GPU parity tests then run the plans these rules produce.
"""
import itertools
import re

import pytest

import tile_primitive_tensor_gb300 as tp
import workloads as wl
from tile_primitive_tensor_gb300 import build as tpbuild

TC = tp.TPGEMM_PATH_TCGEN05


@pytest.fixture(scope="module", autouse=True)
def _lib():
    tpbuild.build()
    tp.library()


def plan(M, N, K, tA, tB, dtype, beta):
    st, text = tp.tpgemm_describe_plan(M, N, K, tA, tB, dtype, beta, TC)
    assert st == tp.TPGEMM_OK, text
    d = dict(kv.split("=", 1) for kv in text.split() if "=" in kv)
    d["text"] = text
    full, rem, split = (int(x) for x in re.match(r"(\d+)\+(\d+)x(\d+)", d["units"]).groups())
    tiles_p, tiles_q = (int(x) for x in d["tiles"].split("x"))
    mc = int(d["cluster"])
    d.update(full=full, rem=rem, split=split, ncl=int(d["grid"]) // mc,
             num_super=(tiles_p + mc - 1) // mc * tiles_q)
    return d


# Shapes across one wave, a few waves and many; both orientations; f16, bf16,
# e4m3; beta 0 and 1.
SWEEP = [
    (M, N, K, tA, tB, dtype, beta)
    for (M, N, K), (tA, tB), dtype, beta in itertools.product(
        [(144, 16392, 4104), (1024, 1024, 2048), (2048, 2560, 1032), (4096, 4096, 4096),
         (8192, 8192, 8192), (12288, 8192, 1024), (16384, 16384, 512), (784, 1320, 528)],
        [(False, True), (False, False)],
        [wl.F16, wl.BF16, wl.E4M3],
        [0.0, 1.0])
    # fp8 takes A [M,K] and B [N,K] only, and K % 16 = 0
    if not (dtype == wl.E4M3 and (tA or not tB or K % 16))
]


def sweep_ids(c):
    M, N, K, tA, tB, dtype, beta = c
    return f"{M}x{N}x{K}-{'T' if tA else 'N'}{'T' if tB else 'N'}-d{dtype}-b{int(beta)}"


@pytest.mark.parametrize("case", SWEEP, ids=sweep_ids)
def test_k_direction_rule(case):
    # A cluster's odd units walk K backwards in 16-bit plans of at least
    # eight waves without K rotation; every other plan keeps one direction.
    p = plan(*case)
    want = (p["kind"] == "f16" and p["k_rotate"] == "0" and p["num_super"] >= 8 * p["ncl"])
    assert p["k_reverse"] == ("1" if want else "0"), p["text"]


@pytest.mark.parametrize("case", SWEEP, ids=sweep_ids)
def test_helper_and_producer_rules(case):
    # Helpers: every one-group plan here has a ring of at least 4 stages of
    # 32 KB or more, which holds a helper's half of a tile's chunks.
    # Producers: two, unless a two-group plan with more than one unit per
    # cluster (or stream-K) needs warp 6 for its epilogue.
    p = plan(*case)
    groups = int(p["epi_groups"])
    assert p["epi_help"] == ("1" if groups == 1 else "0"), p["text"]
    multi = p["stream_k"] == "1" or p["full"] + p["rem"] * p["split"] > p["ncl"]
    want = 1 if (groups == 2 and multi) else min(2, int(p["stages"]))
    assert int(p["producers"]) == want, p["text"]


@pytest.mark.parametrize("case", SWEEP, ids=sweep_ids)
def test_stream_k_rule(case):
    # The last, partial wave is split into two K halves per leftover tile when
    # twice the leftover tiles fit the grid's clusters and the tile has at
    # least 16 K blocks; otherwise it is split along N (or not at all).
    p = plan(*case)
    k_blocks = -(-case[2] // int(p["tile"].split("x")[2]))
    want = p["rem"] > 0 and 2 * p["rem"] <= p["ncl"] and k_blocks >= 16
    assert p["stream_k"] == ("1" if want else "0"), p["text"]
    if want:
        assert p["sk_clusters"] == str(2 * p["rem"]) and p["split"] == 1, p["text"]


def test_k_reverse_and_helpers_on_the_benchmark_workloads():
    for M, N, K, tA, tB, dtype, beta, want in [
        (8192, 8192, 8192, False, True, wl.BF16, 1.0,
         "epi_groups=1 epi_help=1 producers=2 dep_early=1 k_rotate=0 k_reverse=1"),
        (4096, 4096, 4096, False, False, wl.F16, 0.0,
         "epi_groups=1 epi_help=1 producers=2 dep_early=1 k_rotate=0 k_reverse=0"),
        (8192, 8192, 8192, False, True, wl.E4M3, 1.0,
         "epi_groups=1 epi_help=1 producers=2 dep_early=1 k_rotate=0 k_reverse=0"),
        (144, 16392, 4104, False, False, wl.F16, 1.0,
         "epi_groups=2 epi_help=0 producers=2 dep_early=1 k_rotate=1 k_reverse=0"),
    ]:
        assert want in plan(M, N, K, tA, tB, dtype, beta)["text"]


def test_overrides_turn_the_rules_off_and_on(tune):
    tune.setenv("TPGEMM_TC_KREV", "1")
    assert plan(4096, 4096, 4096, False, False, wl.F16, 0.0)["k_reverse"] == "1"
    tune.setenv("TPGEMM_TC_KREV", "0")
    assert plan(8192, 8192, 8192, False, True, wl.BF16, 1.0)["k_reverse"] == "0"
    tune.setenv("TPGEMM_TC_EPI_HELP", "0")
    assert plan(8192, 8192, 8192, False, True, wl.BF16, 1.0)["epi_help"] == "0"
    tune.setenv("TPGEMM_TC_PRODUCERS", "1")
    assert plan(8192, 8192, 8192, False, True, wl.BF16, 1.0)["producers"] == "1"


def test_helpers_need_the_ring_to_hold_their_chunks(tune):
    # A two-stage ring of 32 KB stages holds 64 KB: less than the eight warps'
    # 4 KB staging tiles for half of a 256-wide tile's eight chunks each
    # (8 x 4 x 4 KB = 128 KB), so the helpers stay out.
    tune.setenv("TPGEMM_TC_STAGES", "2")
    p = plan(8192, 8192, 8192, False, True, wl.BF16, 1.0)
    assert p["stages"] == "2" and p["tile"] == "128x256x64", p["text"]
    assert p["epi_help"] == "0", p["text"]
    tune.setenv("TPGEMM_TC_STAGES", "4")
    p = plan(8192, 8192, 8192, False, True, wl.BF16, 1.0)
    assert p["stages"] == "4" and p["epi_help"] == "1", p["text"]
