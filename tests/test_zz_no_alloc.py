"""The allocation-free entry point tpgemm_gemm_noalloc (GPU only).

Some callers cannot allocate device memory at call time (a fixed budget
reserved at start-up, an allocator's own reclaim path, memory held by another
framework's pool). tpgemm_gemm_noalloc serves them: its stream-K scratch is a
static device array, never cudaMalloc. This file is collected last so that a
run stopping at the first failure has already run every other test.

Each case calls the entry point twice in a row through the C ABI (the second
call sees the first call's leftovers in the shared static array) and checks
both results against tpgemm_gemm within the acceptance bound the other tests
use, |D - D_ref| <= 2^-10 * sum_k |a b| + 1e-6, doubled because both sides
round independently.
"""
import dataclasses

import pytest
import torch

import tile_primitive_tensor_gb300 as tp
import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _setup():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tile_primitive_tensor_gb300 import build as tpbuild
    tpbuild.build()
    yield
    assert tp.tpgemm_last_device_error() == tp.TPGEMM_OK, tp.tpgemm_last_error_detail()


CASES = [
    # (name, workload, M, N, K, transA, transB, beta): shapes whose plan has a
    # partial last wave, so the stream-K mode and its scratch are used.
    ("skinny_swapped", "skinny_144x16392x4104_f16_beta1", 144, 4104, 1160, False, False, 1.0),
    ("square_chain", "gemm_256_bf16_transB_beta1", 1024, 1024, 2048, False, True, 1.0),
    ("square_nn_beta0", "gemm_4096_f16", 1024, 1024, 2048, False, False, 0.0),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0])
def test_noalloc_matches_gemm_twice(case):
    name, wname, M, N, K, tA, tB, beta = case
    w = dataclasses.replace(wl.BY_NAME[wname].with_shape(M, N, K, seed=7000 + M + K),
                            transA=tA, transB=tB, beta=beta,
                            c_dist=("normal", 0.0, 1.0) if beta else None)
    A, B, C = wl.make_inputs(w)
    Ad, Bd = A.cuda(), B.cuda()
    Cd = None if C is None else C.cuda()
    ref = torch.empty(M, N, device="cuda")
    assert tp.tpgemm_gemm(ref, Ad, Bd, Cd, M, N, K, tA, tB, w.dtype, beta, None) == tp.TPGEMM_OK
    a = Ad.double().t() if tA else Ad.double()
    b = Bd.double().t() if tB else Bd.double()
    bound = 2.0 * ((a.abs() @ b.abs()) * 2.0 ** -10 + 1e-6)
    for call in range(2):
        D = torch.full((M, N), float("nan"), device="cuda")
        st = tp.tpgemm_gemm_noalloc(D, Ad, Bd, Cd, M, N, K, tA, tB, w.dtype, beta, None)
        assert st == tp.TPGEMM_OK, tp.tpgemm_last_error_detail()
        torch.cuda.synchronize()
        err = (D.double() - ref.double()).abs()
        assert bool(torch.isfinite(D).all()), f"call {call}: non-finite output"
        assert bool((err <= bound).all()), f"call {call}: max err/bound {float((err / bound).max())}"
    assert tp.tpgemm_last_device_error() == tp.TPGEMM_OK
