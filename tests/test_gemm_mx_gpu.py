"""Parity of the block-scaled fp8 (MX) multiply with the CPU oracle (GPU only).

tpgemm_gemm_mx runs tcgen05.mma kind::mxf8f6f4.block_scale on the tcgen05
kernel, the E8M0 scales packed by a pre-pass and copied into tensor memory by
tcgen05.cp. Every case draws seeded operands and scales and compares every
element with ``oracle.gemm_mx`` (the OCP Microscaling reading of the block
scaling the synchronous gemm page lists for gemm_async, section 七): bit-exact
for integer operands with scales in [1/2, 2], else |D - D_ref| <= 2^-10 * S +
1e-6. Shapes cover one tile, ragged M / N / K (a partial last scale block and
a partial last 128-element stage), both orientations (small M is swapped, so
B's scales become the MMA's A scales), both formats, beta 0 / 1, guard bands
around D, and the MX workloads at full size.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import tile_primitive_tensor_gb300 as tp
import workloads as wl

pytestmark = pytest.mark.gpu
GUARD = 4096


@pytest.fixture(scope="module", autouse=True)
def _setup():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tile_primitive_tensor_gb300 import build as tpbuild
    tpbuild.build()
    oracle.build()
    yield
    assert tp.tpgemm_last_device_error() == tp.TPGEMM_OK, tp.tpgemm_last_error_detail()


def case(M, N, K, dtype, beta, dist=("normal", 0.0, 1.0), sf=(120, 134), seed=0):
    base = wl.BY_NAME["mx_256_e4m3_transB_beta1"]
    return dataclasses.replace(base, name=f"mx_{M}x{N}x{K}_{dtype}_{beta}", M=M, N=N, K=K,
                               dtype=dtype, a_dist=dist, b_dist=dist,
                               c_dist=("normal", 0.0, 1.0) if beta else None, beta=beta,
                               seed=seed, sf_dist=sf)


def run_mx(w):
    """Run the library on workload w; returns (D host, plan text)."""
    A, B, C = wl.make_inputs(w)
    SFA, SFB = wl.make_scales(w)
    Ad, Bd = A.cuda(), B.cuda()
    Cd = None if C is None else C.cuda()
    sa, sb = SFA.cuda(), SFB.cuda()
    n = w.M * w.N
    buf = torch.full((n + 2 * GUARD,), float("nan"), device="cuda")
    D = buf[GUARD:GUARD + n].view(w.M, w.N)
    wsb = tp.tpgemm_gemm_mx_workspace_bytes(w.M, w.N, w.K)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    st = tp.tpgemm_gemm_mx(D, Ad, Bd, Cd, sa, sb, w.M, w.N, w.K, w.dtype, w.beta, ws, wsb)
    assert st == tp.TPGEMM_OK, tp.tpgemm_last_error_detail()
    torch.cuda.synchronize()
    plan = tp.tpgemm_last_plan()[1]
    h = buf.cpu().numpy()
    assert np.isnan(h[:GUARD]).all() and np.isnan(h[GUARD + n:]).all(), "write outside D"
    return h[GUARD:GUARD + n].reshape(w.M, w.N), plan, (A, B, C, SFA, SFB)


def check(w):
    D, plan, (A, B, C, SFA, SFB) = run_mx(w)
    assert "kind=mxf8f6f4" in plan, plan
    Dref, S = oracle.gemm_mx(wl.operand_bits(w, A), wl.operand_bits(w, B),
                             None if C is None else C.numpy(), SFA.numpy(), SFB.numpy(), w.M, w.N,
                             w.K, w.transA, w.transB, w.dtype, w.beta)
    ok, msg = oracle.compare(D, Dref, S, exact=w.integer_valued)
    assert ok, f"{w.name} [{plan}]: {msg}"
    return plan


def test_mx_one_tile_integer_exact():
    # One 128 x 128 tile, one 128-element stage: integer operands and scales
    # in {1/2, 1, 2} make every partial sum exact.
    check(case(128, 128, 128, wl.E4M3, 0.0, dist=("int", -3, 3), sf=(126, 128), seed=1))


@pytest.mark.parametrize("dtype", [wl.E4M3, wl.E5M2])
@pytest.mark.parametrize("beta", [0.0, 1.0])
def test_mx_multi_tile(dtype, beta):
    check(case(784, 1320, 528, dtype, beta, seed=2 + dtype + int(beta)))


@pytest.mark.parametrize("M,N,K", [
    (272, 392, 272),    # partial last scale block (K % 32 = 16) and stage (K % 128 = 16)
    (256, 136, 4112),   # a last Q tile of 8 rows, long K
    (1040, 16, 2048),   # N = 16: one narrow Q tile
    (2048, 4096, 128),  # one K stage, many tiles
])
def test_mx_ragged_normal(M, N, K):
    plan = check(case(M, N, K, wl.E4M3, 1.0, seed=M + N + K))
    assert "orientation=normal" in plan, plan


@pytest.mark.parametrize("M", [16, 64, 144, 160])
def test_mx_small_m_swapped(M):
    # All of M fits one accumulator: P = B, so B's scales are the MMA's A
    # scales and A's (up to 160 rows, two 128-row chunks) the B scales.
    plan = check(case(M, 4104 if M != 160 else 2056, 1040, wl.E5M2 if M % 32 else wl.E4M3, 1.0,
                      seed=50 + M))
    assert "orientation=swapped" in plan, plan


@pytest.mark.parametrize("bp", [64, 80, 96, 112])
@pytest.mark.parametrize("shape", [(144, 4104, 1040), (2064, 200, 528)])
def test_mx_p_rows(bp, shape, tune):
    # All of Q in one tile: each CTA streams bp < 128 rows of P, whose scales
    # are packed in tiles of bp rows (the copy's rows past bp read as 1).
    # Swapped small M, and the normal orientation with a narrow N.
    tune.setenv("TPGEMM_TC_BP", str(bp))
    plan = check(case(*shape, wl.E4M3, 1.0, seed=120 + bp + shape[0]))
    assert f"tile={bp}x" in plan, plan


def test_mx_m176_stays_normal():
    plan = check(case(176, 2048, 512, wl.E4M3, 0.0, seed=61))
    assert "orientation=normal" in plan, plan


def test_mx_integer_bit_exact_large():
    check(case(1024, 1024, 1024, wl.E4M3, 1.0, dist=("int", -3, 3), sf=(126, 128), seed=71))
    check(case(512, 768, 2048, wl.E5M2, 0.0, dist=("int", -3, 3), sf=(126, 128), seed=72))


@pytest.mark.parametrize("krev", ["0", "1"])
def test_mx_k_direction(krev, tune):
    # Each stage's scales are loaded for the K block its operands come from,
    # whichever way the unit walks K; six clusters give each one several units.
    tune.setenv("TPGEMM_TC_MAX_CLUSTERS", "6")
    tune.setenv("TPGEMM_TC_KREV", krev)
    plan = check(case(1024, 1344, 1024, wl.E4M3, 1.0, dist=("int", -3, 3), sf=(126, 128), seed=91))
    assert f"k_reverse={krev}" in plan, plan


@pytest.mark.parametrize("help_", ["0", "1"])
def test_mx_last_segment_helpers(help_, tune):
    # The helpers' share of a block-scaled tile's last segment (224 columns:
    # 7 chunks, 3 of them the helpers'), with C.
    tune.setenv("TPGEMM_TC_MAX_CLUSTERS", "6")
    tune.setenv("TPGEMM_TC_EPI_HELP", help_)
    plan = check(case(1024, 1344, 1024, wl.E4M3, 1.0, dist=("int", -3, 3), sf=(126, 128), seed=93))
    assert f"epi_help={help_}" in plan, plan


def test_mx_unit_scales_equal_plain_fp8():
    # With every scale 1 the block-scaled multiply is the plain fp8 one, and the
    # library's two paths agree within the bound (the oracle agrees bit for bit).
    w = case(512, 640, 384, wl.E4M3, 1.0, sf=(127, 127), seed=81)
    D, _, (A, B, C, _, _) = run_mx(w)
    Dp = torch.empty(w.M, w.N, device="cuda")
    st = tp.tpgemm_gemm(Dp, A.cuda(), B.cuda(), C.cuda(), w.M, w.N, w.K, 0, 1, w.dtype, 1.0)
    assert st == tp.TPGEMM_OK, tp.tpgemm_last_error_detail()
    Dref, S = oracle.gemm(wl.bits(A), wl.bits(B), C.numpy(), w.M, w.N, w.K, False, True, w.dtype,
                          1.0)
    for got in (D, Dp.cpu().numpy()):
        ok, msg = oracle.compare(got, Dref, S)
        assert ok, msg


def test_mx_back_to_back_calls_share_nothing():
    # Two different problems enqueued back to back on one stream, each with
    # its own workspace, then checked: the second launch may start while the
    # first drains (programmatic dependent launch).
    ws = [case(384, 512, 256, wl.E4M3, 1.0, seed=91), case(256, 640, 384, wl.E5M2, 0.0, seed=92)]
    outs = []
    for w in ws:
        A, B, C = wl.make_inputs(w)
        SFA, SFB = wl.make_scales(w)
        D = torch.empty(w.M, w.N, device="cuda")
        wsb = tp.tpgemm_gemm_mx_workspace_bytes(w.M, w.N, w.K)
        buf = torch.empty(wsb, dtype=torch.uint8, device="cuda")
        keep = (A.cuda(), B.cuda(), None if C is None else C.cuda(), SFA.cuda(), SFB.cuda(), buf)
        st = tp.tpgemm_gemm_mx(D, keep[0], keep[1], keep[2], keep[3], keep[4], w.M, w.N, w.K,
                               w.dtype, w.beta, buf, wsb)
        assert st == tp.TPGEMM_OK, tp.tpgemm_last_error_detail()
        outs.append((w, D, keep, (A, B, C, SFA, SFB)))
    torch.cuda.synchronize()
    for w, D, _, (A, B, C, SFA, SFB) in outs:
        Dref, S = oracle.gemm_mx(wl.operand_bits(w, A), wl.operand_bits(w, B),
                                 None if C is None else C.numpy(), SFA.numpy(), SFB.numpy(), w.M,
                                 w.N, w.K, False, True, w.dtype, w.beta)
        ok, msg = oracle.compare(D.cpu().numpy(), Dref, S)
        assert ok, msg


@pytest.mark.parametrize("name", [w.name for w in wl.MX_WORKLOADS])
def test_mx_workload_full_size(name):
    # Every element against the oracle's whole output.
    check(wl.BY_NAME[name])


def test_mx_pair_and_224_wide_tiles():
    # The default for large problems: CTA pairs (cta_group::2 block-scaled MMA,
    # each CTA holding its own A scales and all of the tile's B scales) on
    # 224-wide tiles, so Q tiles start at multiples of 224 and their scales
    # span two 128-row chunks (one replicated 128x256b copy), two scale slots
    # per accumulator half.
    plan = check(case(784, 1320, 528, wl.E4M3, 1.0, seed=101))
    assert "pair=1" in plan and "tile=128x224x128" in plan, plan


@pytest.mark.parametrize("bn", [192, 160, 128, 96])
def test_mx_tile_widths(bn, tune):
    # Narrower tiles: five 12-column slots per half at 192, eight at 160, and
    # one warpx4 Q copy (no replication) at 128 and below.
    tune.setenv("TPGEMM_TC_BN", str(bn))
    plan = check(case(784, 1320, 528, wl.E4M3, 1.0, seed=110 + bn))
    assert f"tile=128x{bn}x128" in plan, plan


def test_mx_single_cta_when_one_p_tile():
    # One 128-row P tile: no pair.
    plan = check(case(128, 64, 512, wl.E5M2, 1.0, seed=102))
    assert "pair=0" in plan and "orientation=normal" in plan, plan


@pytest.mark.parametrize("shape", [(784, 1320, 528), (144, 4104, 1040)])
def test_mx_pair_off(shape, tune):
    # The single-CTA block-scaled path on multi-tile and swapped problems.
    tune.setenv("TPGEMM_TC_PAIR", "0")
    plan = check(case(*shape, wl.E4M3, 1.0, seed=103 + shape[0]))
    assert "pair=0" in plan, plan


def test_mx_8192_plan_is_a_pair():
    w = wl.BY_NAME["mx_8192_e4m3_transB_beta1"]
    A, B, C = wl.make_inputs(w.with_shape(512, 512, 256))
    plan = check(w.with_shape(512, 512, 256, seed=104))
    assert "pair=1" in plan, plan



# ------------------------------------------------------------ fp4 (MXFP4)
FP4 = ("codes", 0, 15)


def test_mxfp4_one_tile_exact():
    # One 128 x 128 tile, one 128-element stage; every fp4 value is a multiple
    # of 1/2, so with scales in {1/2, 1, 2} the sums are exact.
    check(case(128, 128, 128, wl.E2M1, 0.0, dist=FP4, sf=(126, 128), seed=201))


@pytest.mark.parametrize("M,N,K,beta", [
    (784, 1320, 512, 1.0),   # CTA pairs, 224-wide tiles
    (144, 4104, 1024, 1.0),  # swapped small M
    (128, 64, 384, 0.0),     # one P tile, single CTA
    (1024, 1024, 4096, 0.0),
])
def test_mxfp4_shapes(M, N, K, beta):
    check(case(M, N, K, wl.E2M1, beta, dist=FP4, sf=(120, 134), seed=210 + M + K))


def test_mxfp4_integer_exact_large():
    check(case(1024, 1536, 2048, wl.E2M1, 0.0, dist=FP4, sf=(126, 128), seed=220))
