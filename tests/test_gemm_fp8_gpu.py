"""fp8 (e4m3 / e5m2) GEMM on the tcgen05 kind::f8f6f4 path, against the oracle.

Same bar as the f16 / bf16 path: bit-exact (by value) on integer-valued
inputs, else |D - D_ref| <= 2^-10 * sum_k |a b| + 1e-6 elementwise, with the
oracle decoding the very same fp8 bytes. fp8 operands are K-contiguous (A
[M,K], B [N,K]); cases cover both formats, beta 0 and 1, ragged M / N / K
tails (K a multiple of 16, not of the 128-element stage), the swapped
orientation of small M, CTA pairs and single CTAs, clusters, tail splitting,
stream-K, and the fp8 workloads at full size (sampled entries plus an fp64
product of the whole output).
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import tile_primitive_tensor_gb300 as tp
import workloads as wl

pytestmark = pytest.mark.gpu
TC = tp.TPGEMM_PATH_TCGEN05


@pytest.fixture(scope="module", autouse=True)
def _setup():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tile_primitive_tensor_gb300 import build as tpbuild
    tpbuild.build()
    oracle.build()
    yield
    assert tp.tpgemm_last_device_error() == tp.TPGEMM_OK, tp.tpgemm_last_error_detail()


def case(M, N, K, dtype, beta, dist=("normal", 0.0, 1.0), seed=0):
    base = wl.BY_NAME["gemm_8192_e4m3_transB_beta1"]
    return dataclasses.replace(base.with_shape(M, N, K, seed=seed), dtype=dtype, beta=beta,
                               a_dist=dist, b_dist=dist,
                               c_dist=("normal", 0.0, 1.0) if beta else None)


def check(w, path=tp.TPGEMM_PATH_AUTO):
    A, B, C = wl.make_inputs(w)
    Ad, Bd = A.cuda(), B.cuda()
    Cd = None if C is None else C.cuda()
    guard = 4096
    buf = torch.full((w.M * w.N + 2 * guard,), float("nan"), device="cuda")
    D = buf[guard: guard + w.M * w.N].view(w.M, w.N)
    st = tp.tpgemm_gemm_path(D, Ad, Bd, Cd, w.M, w.N, w.K, w.transA, w.transB, w.dtype, w.beta,
                             None, path)
    assert st == tp.TPGEMM_OK, tp.tpgemm_last_error_detail()
    torch.cuda.synchronize()
    h = buf.cpu().numpy()
    assert np.isnan(h[:guard]).all() and np.isnan(h[guard + w.M * w.N:]).all()
    Dh = D.cpu().numpy()
    Dref, S = oracle.gemm(wl.bits(A), wl.bits(B), None if C is None else C.numpy(), w.M, w.N,
                          w.K, w.transA, w.transB, w.dtype, w.beta)
    ok, msg = oracle.compare(Dh, Dref, S, exact=w.integer_valued)
    assert ok, f"{w.name}: {msg}"
    return Dh


FMTS = [wl.E4M3, wl.E5M2]


@pytest.mark.parametrize("dtype", FMTS, ids=["e4m3", "e5m2"])
@pytest.mark.parametrize("beta", [0.0, 1.0])
@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (272, 264, 272), (128, 128, 144),
                                   (384, 392, 400), (16, 8, 32), (48, 40, 48)])
def test_fp8_tiled(M, N, K, dtype, beta):
    check(case(M, N, K, dtype, beta, seed=7 * M + K + dtype))


@pytest.mark.parametrize("dtype", FMTS, ids=["e4m3", "e5m2"])
def test_fp8_swapped_small_m(dtype):
    w = case(144, 2072, 528, dtype, 1.0, seed=11)
    st, text = tp.tpgemm_describe_plan(w.M, w.N, w.K, 0, 1, dtype, 1.0)
    assert "orientation=swapped" in text and "kind=f8f6f4" in text, text
    check(w)


@pytest.mark.parametrize("pair", ["0", "1"])
@pytest.mark.parametrize("bn", ["128", "256"])
def test_fp8_pair_and_width(pair, bn, tune):
    tune.setenv("TPGEMM_TC_PAIR", pair)
    tune.setenv("TPGEMM_TC_BN", bn)
    check(case(784, 1320, 272, wl.E4M3, 1.0, seed=13))


def test_fp8_single_cta_shared_q(tune):
    # Every tile shares the one Q tile and each CTA loads it itself.
    tune.setenv("TPGEMM_TC_PAIR", "0")
    check(case(1024, 128, 256, wl.E5M2, 0.0, seed=17))


def test_fp8_tail_split(tune):
    tune.setenv("TPGEMM_TC_BN", "256")
    tune.setenv("TPGEMM_TC_SK", "0")  # the tail split, not stream-K
    w = case(2048, 2560, 160, wl.E4M3, 1.0, seed=19)
    st, text = tp.tpgemm_describe_plan(w.M, w.N, w.K, 0, 1, w.dtype, 1.0)
    assert "x1 " not in text.split("units=")[1][:12], text
    check(w)


def test_fp8_stream_k(tune):
    tune.setenv("TPGEMM_TC_SK", "1")
    w = case(1024, 1024, 4096, wl.E4M3, 1.0, seed=23)  # 32 K blocks of 128: enough to split
    st, text = tp.tpgemm_describe_plan(w.M, w.N, w.K, 0, 1, w.dtype, 1.0)
    assert "stream_k=1" in text, text
    check(w)


def test_fp8_integer_bit_exact():
    check(case(1024, 1024, 1024, wl.E4M3, 0.0, dist=("int", -3, 3), seed=29))
    check(case(512, 768, 2048, wl.E5M2, 1.0, dist=("int", -3, 3), seed=31))


@pytest.mark.parametrize("name", [w.name for w in wl.FP8_WORKLOADS])
def test_fp8_workload_full_size(name):
    w = wl.BY_NAME[name]
    A, B, C = wl.make_inputs(w)
    Ad, Bd = A.cuda(), B.cuda()
    Cd = None if C is None else C.cuda()
    D = torch.empty(w.M, w.N, device="cuda")
    st = tp.tpgemm_gemm(D, Ad, Bd, Cd, w.M, w.N, w.K, w.transA, w.transB, w.dtype, w.beta, None)
    assert st == tp.TPGEMM_OK, tp.tpgemm_last_error_detail()
    torch.cuda.synchronize()
    Dh = D.cpu().numpy()
    del D, Ad, Bd, Cd
    # Every element against the oracle's whole output.
    Dref, S = oracle.gemm(wl.bits(A), wl.bits(B), None if C is None else C.numpy(), w.M, w.N, w.K,
                          w.transA, w.transB, w.dtype, w.beta)
    ok, msg = oracle.compare(Dh, Dref, S, exact=w.integer_valued)
    assert ok, f"{name}: {msg}"


@pytest.mark.parametrize("M,N,K,dtype", [(4096, 16, 4096, wl.E4M3), (16, 16392, 128, wl.E5M2),
                                         (16, 8, 16, wl.E4M3), (2048, 2056, 16, wl.E5M2)])
def test_fp8_extreme_shapes(M, N, K, dtype):
    check(case(M, N, K, dtype, 1.0, seed=M + N + K))



# fp4 e2m1 without block scales (kind::f8f6f4, format 5): A [M, K/2] and B
# [N, K/2] packed two codes per byte, unpacked by the TMA into the 16-byte
# padded groups the MMA reads.
@pytest.mark.parametrize("M,N,K,beta", [(128, 128, 128, 0.0), (784, 1320, 512, 1.0),
                                        (144, 4104, 1024, 1.0), (2048, 2048, 2048, 0.0)])
def test_fp4_plain(M, N, K, beta):
    w = dataclasses.replace(wl.BY_NAME["mxfp4_4096_int_transB"], name=f"fp4_{M}x{N}x{K}",
                            M=M, N=N, K=K, beta=beta,
                            c_dist=("normal", 0.0, 1.0) if beta else None, seed=300 + M + K)
    w = wl.Workload(**{f.name: getattr(w, f.name) for f in dataclasses.fields(wl.Workload)})
    A, B, C = wl.make_inputs(w)
    D = torch.empty(M, N, device="cuda")
    st = tp.tpgemm_gemm(D, A.cuda(), B.cuda(), None if C is None else C.cuda(), M, N, K, 0, 1,
                        wl.E2M1, beta)
    assert st == tp.TPGEMM_OK, tp.tpgemm_last_error_detail()
    torch.cuda.synchronize()
    Dref, S = oracle.gemm(wl.operand_bits(w, A), wl.operand_bits(w, B),
                          None if C is None else C.numpy(), M, N, K, False, True, wl.E2M1, beta)
    # fp4 values are multiples of 1/2 up to 6: every partial sum below K = 4096
    # is a multiple of 1/4 under 2^18, exact in float32
    ok, msg = oracle.compare(D.cpu().numpy(), Dref, S, exact=C is None)
    assert ok, msg
