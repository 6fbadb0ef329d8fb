"""The allocation-free entry point tpgemm_gemm_noalloc (GPU only).

Some callers cannot allocate device memory at call time: a service that
reserves its whole device-memory budget at start-up, code running inside an
allocator's own out-of-memory or reclaim path, or a process whose device memory
is all held by another framework's pool. tpgemm_gemm_noalloc serves them: the
stream-K scratch it needs lives in a static device array, never cudaMalloc.
This file is collected last so that a run stopping at the first failure has
already run every other test.

Each case calls the entry point twice in a row through the C ABI (the second
call sees the first call's leftovers in the shared static array) and checks
both results element by element against the CPU oracle with the acceptance
bound of the other parity tests, |D - D_ref| <= 2^-10 * sum_k |a b| + 1e-6. The
shapes have a partial last wave, and the test asserts from tpgemm_last_plan()
that the stream-K mode really ran on the static array, and that the device's
free memory is the same before and after the second call.
"""
import dataclasses

import pytest
import torch

import oracle
import tile_primitive_tensor_gb300 as tp
import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _setup():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tile_primitive_tensor_gb300 import build as tpbuild
    tpbuild.build()
    oracle.build()
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
def test_noalloc_matches_oracle_twice(case):
    name, wname, M, N, K, tA, tB, beta = case
    w = dataclasses.replace(wl.BY_NAME[wname].with_shape(M, N, K, seed=7000 + M + K),
                            transA=tA, transB=tB, beta=beta,
                            c_dist=("normal", 0.0, 1.0) if beta else None)
    A, B, C = wl.make_inputs(w)
    Dref, S = oracle.gemm(wl.bits(A), wl.bits(B), None if C is None else C.numpy(), M, N, K,
                          tA, tB, w.dtype, beta)
    Ad, Bd = A.cuda(), B.cuda()
    Cd = None if C is None else C.cuda()
    for call in range(2):
        D = torch.full((M, N), float("nan"), device="cuda")
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info()[0]
        st = tp.tpgemm_gemm_noalloc(D, Ad, Bd, Cd, M, N, K, tA, tB, w.dtype, beta, None)
        assert st == tp.TPGEMM_OK, tp.tpgemm_last_error_detail()
        torch.cuda.synchronize()
        free1 = torch.cuda.mem_get_info()[0]
        st, plan = tp.tpgemm_last_plan()
        assert st == tp.TPGEMM_OK
        assert "stream_k=1" in plan and "scratch=static" in plan, plan
        if call == 1:  # the first call on a device may load the kernel's module
            assert free1 == free0, f"device free memory changed by {free0 - free1} bytes"
        ok, msg = oracle.compare(D.cpu().numpy(), Dref, S)
        assert ok, f"call {call}: {msg}"
    assert tp.tpgemm_last_device_error() == tp.TPGEMM_OK
