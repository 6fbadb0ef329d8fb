"""The debug build (libtpgemm_debug.so, -DTPGEMM_DEBUG) on the GPU.

Every computed tensor-memory column, TMA store / C-load coordinate and
stream-K flag index in the tcgen05 kernel is checked against its range; a
failed check records TPGEMM_ERR_BOUNDS and the site for
tpgemm_last_device_error and skips the access (nothing traps). These tests
run the parity cases of the main plans through the debug library (every
check must pass and the results match the oracle), then plant one bad column
(TPGEMM_DEBUG_PLANT, read by the debug build only) that the check must catch,
and check that the next call is clean.
"""
import ctypes
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import tile_primitive_tensor_gb300 as tp
import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dbg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tile_primitive_tensor_gb300 import build as tpbuild
    tpbuild.build(debug=True)
    oracle.build()
    lib = tp.debug_library()
    yield lib
    lib.tpgemm_reload_tuning()


def status(lib):
    st = int(lib.tpgemm_last_device_error())
    return st, lib.tpgemm_last_error_detail().decode()


def run(lib, w, C_override=None):
    A, B, C = wl.make_inputs(w)
    Ad, Bd = A.cuda(), B.cuda()
    Cd = None if C is None else C.cuda()
    D = torch.full((w.M, w.N), float("nan"), device="cuda")
    st = lib.tpgemm_gemm(D.data_ptr(), Ad.data_ptr(), Bd.data_ptr(),
                         None if Cd is None else Cd.data_ptr(), w.M, w.N, w.K, int(w.transA),
                         int(w.transB), w.dtype, float(w.beta), None)
    assert st == tp.TPGEMM_OK, lib.tpgemm_last_error_detail()
    torch.cuda.synchronize()
    return D.cpu().numpy(), (A, B, C)


def check(lib, w):
    D, (A, B, C) = run(lib, w)
    st, why = status(lib)
    assert st == tp.TPGEMM_OK, why
    Dref, S = oracle.gemm(wl.operand_bits(w, A), wl.operand_bits(w, B),
                          None if C is None else C.numpy(), w.M, w.N, w.K, w.transA, w.transB,
                          w.dtype, w.beta)
    ok, msg = oracle.compare(D, Dref, S, exact=w.integer_valued)
    assert ok, msg


CASES = [
    ("pair_transB", "gemm_8192_bf16_transB_beta1", 784, 1320, 520),
    ("swapped_skinny_112rows", "skinny_144x16392x4104_f16_beta1", 144, 4104, 264),
    ("nn_square", "gemm_4096_f16", 1024, 1024, 512),
    ("fp8", "gemm_8192_e4m3_transB_beta1", 512, 768, 512),
    ("fp4", "mxfp4_4096_int_transB", 256, 384, 512),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0])
def test_debug_build_parity_with_every_check_passing(dbg, case):
    name, base, M, N, K = case
    w = wl.BY_NAME[base].with_shape(M, N, K, seed=900 + M + K)
    if isinstance(w, wl.MxWorkload):  # the plain multiply of fp4 operands
        w = wl.Workload(**{f.name: getattr(w, f.name) for f in dataclasses.fields(wl.Workload)})
    check(dbg, w)


def test_debug_build_stream_k(dbg, monkeypatch):
    monkeypatch.setenv("TPGEMM_TC_SK", "1")
    dbg.tpgemm_reload_tuning()
    try:
        check(dbg, wl.BY_NAME["gemm_256_bf16_transB_beta1"].with_shape(1024, 1024, 2048, seed=950))
    finally:
        monkeypatch.delenv("TPGEMM_TC_SK")
        dbg.tpgemm_reload_tuning()


def test_debug_build_stream_k_default_swapped(dbg):
    # The default two-half split of a single partial wave in the swapped
    # orientation with beta = 0 (the layout of the 4096^3 workload): the
    # kernel-start zero-fill, the flag waits, the TMA reductions and the
    # ring-staged last epilogue, every index checked.
    w = wl.BY_NAME["gemm_4096_f16"].with_shape(1024, 1024, 2048, seed=955)
    st, text = tp.tpgemm_describe_plan(w.M, w.N, w.K, w.transA, w.transB, w.dtype, w.beta)
    assert "orientation=swapped" in text and "stream_k=1" in text, text
    check(dbg, w)


def test_debug_build_block_scaled(dbg):
    w = wl.BY_NAME["mx_8192_e4m3_transB_beta1"].with_shape(784, 1320, 528, seed=958)
    A, B, C = wl.make_inputs(w)
    SFA, SFB = wl.make_scales(w)
    t = [x.cuda() for x in (A, B, C, SFA, SFB)]
    D = torch.full((w.M, w.N), float("nan"), device="cuda")
    wsb = int(dbg.tpgemm_gemm_mx_workspace_bytes(w.M, w.N, w.K))
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    st = dbg.tpgemm_gemm_mx(D.data_ptr(), t[0].data_ptr(), t[1].data_ptr(), t[2].data_ptr(),
                            t[3].data_ptr(), t[4].data_ptr(), w.M, w.N, w.K, w.dtype,
                            float(w.beta), ws.data_ptr(), wsb, None)
    assert st == tp.TPGEMM_OK, dbg.tpgemm_last_error_detail()
    torch.cuda.synchronize()
    st, why = status(dbg)
    assert st == tp.TPGEMM_OK, why
    Dref, S = oracle.gemm_mx(wl.operand_bits(w, A), wl.operand_bits(w, B), C.numpy(),
                             SFA.numpy(), SFB.numpy(), w.M, w.N, w.K, w.transA, w.transB,
                             w.dtype, w.beta)
    ok, msg = oracle.compare(D.cpu().numpy(), Dref, S)
    assert ok, msg


def test_planted_bad_column_is_caught_and_skipped(dbg, monkeypatch):
    # The plant moves the epilogue's first tensor-memory load past the
    # allocation; the check reports it and the load is skipped.
    w = wl.BY_NAME["gemm_8192_bf16_transB_beta1"].with_shape(512, 512, 256, seed=960)
    monkeypatch.setenv("TPGEMM_DEBUG_PLANT", "1")
    dbg.tpgemm_reload_tuning()
    try:
        run(dbg, w)
        st, why = status(dbg)
        assert st == tp.TPGEMM_ERR_BOUNDS, why
        assert "epilogue tensor-memory load" in why
    finally:
        monkeypatch.delenv("TPGEMM_DEBUG_PLANT")
        dbg.tpgemm_reload_tuning()
    check(dbg, w)  # the next call is clean and correct
