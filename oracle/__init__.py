"""CPU oracle for D = A.B + beta.C (fp16/bf16 in, fp64 accumulate, fp32 out).

TEST INFRASTRUCTURE. Only the test suite, the smoke check and the benchmark's
CPU-baseline leg may import this package. The CUDA library never does, and
nothing here is shared with it: the arithmetic lives in ``oracle_gemm.c``
(plain C, compiled with gcc), this module only marshals numpy arrays.

The method it follows is the TVM TIRx synchronous ``gemm`` tile primitive
(page "TVM TIRx 同步 GEMM 深度解析", sections 语义定义, 二 What it accepts,
维度一致性 and 四 step 3): alpha = 1, beta in {0, 1}, transpose flags only set
the logical orientation, the accumulator starts from C (beta = 1) or zero.

The acceptance rule for a GPU result against this oracle is elementwise
|D - D_ref| <= 2^-10 * S + 1e-6, where S = sum_k |a(i,k) b(k,j)|, and exact
equality (by value, so -0 == +0) when every input is integer-valued.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle_gemm.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")

F16 = 0
BF16 = 1
E4M3 = 2
E5M2 = 3

TOL_REL = 2.0 ** -10
TOL_ABS = 1e-6

_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile oracle_gemm.c into _build/liboracle.so with gcc (OpenMP if available)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    base = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-ffp-contract=off", _SRC, "-lm"]
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:] + ["-o", tmp], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base + ["-o", tmp], check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        p = ctypes.c_void_p
        i64 = ctypes.c_int64
        ci = ctypes.c_int
        lib.oracle_decode_f16.argtypes = [ctypes.c_uint16]
        lib.oracle_decode_f16.restype = ctypes.c_double
        lib.oracle_decode_bf16.argtypes = [ctypes.c_uint16]
        lib.oracle_decode_bf16.restype = ctypes.c_double
        lib.oracle_decode.argtypes = [p, p, i64, ci]
        lib.oracle_decode.restype = None
        lib.oracle_num_threads.argtypes = []
        lib.oracle_num_threads.restype = ci
        lib.oracle_gemm.argtypes = [p, p, p, p, p, i64, i64, i64, ci, ci, ci, ci]
        lib.oracle_gemm.restype = ci
        lib.oracle_gemm_entries.argtypes = [p, p, p, p, i64, p, p, p, i64, i64, i64, ci, ci, ci, ci]
        lib.oracle_gemm_entries.restype = ci
        lib.oracle_gemm_rows.argtypes = [p, p, p, p, i64, i64, i64, i64, i64, ci, ci, ci, ci]
        lib.oracle_gemm_rows.restype = ci
        lib.oracle_decode_e2m1.argtypes = [ctypes.c_uint16]
        lib.oracle_decode_e2m1.restype = ctypes.c_double
        lib.oracle_decode_e8m0.argtypes = [ctypes.c_uint8]
        lib.oracle_decode_e8m0.restype = ctypes.c_double
        lib.oracle_gemm_mx.argtypes = [p, p, p, p, p, p, p, i64, i64, i64, ci, ci, ci, ci, i64]
        lib.oracle_gemm_mx.restype = ci
        _lib = lib
        return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _as_bits(x, n_expected: int):
    a = np.ascontiguousarray(x)
    if a.dtype != np.uint16:
        raise TypeError(f"operand must be raw uint16 bit patterns, got {a.dtype}")
    if a.size != n_expected:
        raise ValueError(f"operand has {a.size} elements, expected {n_expected}")
    return a


def _as_c(C, M, N, beta):
    # C is handed to the C code whenever the caller gives one; with beta = 0
    # the C code never reads it (a NaN-filled C proves that).
    if C is None:
        if beta:
            raise ValueError("beta = 1 needs C")
        return None
    c = np.ascontiguousarray(C, dtype=np.float32)
    if c.size != M * N:
        raise ValueError(f"C has {c.size} elements, expected {M * N}")
    return c


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def decode(bits, dtype: int) -> np.ndarray:
    """Exact float64 values of fp16 (dtype 0) or bf16 (dtype 1) patterns, or of fp8
    e4m3 (2) / e5m2 (3) patterns widened to 16 bits."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(b.shape, dtype=np.float64)
    _load().oracle_decode(_ptr(b), _ptr(out), b.size, int(dtype))
    return out


def gemm(A_bits, B_bits, C, M: int, N: int, K: int, transA: bool, transB: bool,
         dtype: int, beta: float):
    """Full D_ref [M, N] float32 and S [M, N] float64 (sum of |products|)."""
    _check_beta(beta)
    A = _as_bits(A_bits, M * K)
    B = _as_bits(B_bits, K * N)
    c = _as_c(C, M, N, beta)
    D = np.empty((M, N), dtype=np.float32)
    S = np.empty((M, N), dtype=np.float64)
    rc = _load().oracle_gemm(_ptr(D), _ptr(S), _ptr(A), _ptr(B), _ptr(c), M, N, K, int(bool(transA)),
                             int(bool(transB)), int(dtype), int(beta != 0.0))
    if rc != 0:
        raise RuntimeError(f"oracle_gemm failed with code {rc}")
    return D, S


def decode_e8m0(e: int) -> float:
    """Value of one E8M0 block scale: 2^(e - 127); 255 is NaN."""
    return float(_load().oracle_decode_e8m0(int(e)))


def gemm_mx(A_bits, B_bits, C, SFA, SFB, M: int, N: int, K: int, transA: bool, transB: bool,
            dtype: int, beta: float, block: int = 32):
    """Block-scaled fp8 (MX): full D_ref [M, N] float32 and S [M, N] float64.

    SFA is [M, ceil(K / block)] and SFB [N, ceil(K / block)] E8M0 bytes; each
    scales `block` consecutive K elements of a row of A / a column of B."""
    _check_beta(beta)
    A = _as_bits(A_bits, M * K)
    B = _as_bits(B_bits, K * N)
    c = _as_c(C, M, N, beta)
    kb = (K + block - 1) // block
    sfa = np.ascontiguousarray(SFA, dtype=np.uint8)
    sfb = np.ascontiguousarray(SFB, dtype=np.uint8)
    if sfa.size != M * kb or sfb.size != N * kb:
        raise ValueError(f"scales must be [M, {kb}] and [N, {kb}]")
    D = np.empty((M, N), dtype=np.float32)
    S = np.empty((M, N), dtype=np.float64)
    rc = _load().oracle_gemm_mx(_ptr(D), _ptr(S), _ptr(A), _ptr(B), _ptr(c), _ptr(sfa),
                                _ptr(sfb), M, N, K, int(bool(transA)), int(bool(transB)),
                                int(dtype), int(beta != 0.0), int(block))
    if rc != 0:
        raise RuntimeError(f"oracle_gemm_mx failed with code {rc}")
    return D, S


def gemm_entries(rows, cols, A_bits, B_bits, C, M: int, N: int, K: int, transA: bool,
                 transB: bool, dtype: int, beta: float):
    """D_ref and S at the given (row, col) positions only, computed one by one."""
    _check_beta(beta)
    A = _as_bits(A_bits, M * K)
    B = _as_bits(B_bits, K * N)
    c = _as_c(C, M, N, beta)
    r = np.ascontiguousarray(rows, dtype=np.int64)
    q = np.ascontiguousarray(cols, dtype=np.int64)
    if r.shape != q.shape:
        raise ValueError("rows and cols must have the same shape")
    D = np.empty(r.shape, dtype=np.float32)
    S = np.empty(r.shape, dtype=np.float64)
    rc = _load().oracle_gemm_entries(_ptr(D), _ptr(S), _ptr(r), _ptr(q), r.size, _ptr(A), _ptr(B),
                                     _ptr(c), M, N, K, int(bool(transA)), int(bool(transB)),
                                     int(dtype), int(beta != 0.0))
    if rc != 0:
        raise RuntimeError(f"oracle_gemm_entries failed with code {rc}")
    return D, S


def gemm_rows(row_begin: int, row_end: int, A_bits, B_bits, C, M: int, N: int, K: int,
              transA: bool, transB: bool, dtype: int, beta: float):
    """Rows [row_begin, row_end) of D_ref (no S); the bounded CPU-baseline sample."""
    _check_beta(beta)
    A = _as_bits(A_bits, M * K)
    B = _as_bits(B_bits, K * N)
    c = _as_c(C, M, N, beta)
    D = np.empty((row_end - row_begin, N), dtype=np.float32)
    rc = _load().oracle_gemm_rows(_ptr(D), _ptr(A), _ptr(B), _ptr(c), M, N, K, row_begin, row_end,
                                  int(bool(transA)), int(bool(transB)), int(dtype),
                                  int(beta != 0.0))
    if rc != 0:
        raise RuntimeError(f"oracle_gemm_rows failed with code {rc}")
    return D


def _check_beta(beta):
    if beta not in (0.0, 1.0):
        raise ValueError(f"beta must be 0 or 1, got {beta}")


def tolerance(S) -> np.ndarray:
    """Elementwise bound 2^-10 * S + 1e-6 on |D - D_ref|."""
    return TOL_REL * np.asarray(S, dtype=np.float64) + TOL_ABS


def compare(D, D_ref, S, exact: bool = False):
    """Check D against the oracle.

    Returns (ok, report). With exact=True every element must equal D_ref by
    value (so -0 == +0); otherwise |D - D_ref| <= 2^-10 * S + 1e-6. A NaN or
    infinity in D always fails.
    """
    d = np.asarray(D, dtype=np.float32).astype(np.float64)
    r = np.asarray(D_ref, dtype=np.float32).astype(np.float64)
    if d.shape != r.shape:
        return False, f"shape {d.shape} != {r.shape}"
    finite = np.isfinite(d)
    err = np.abs(d - r)
    if exact:
        bad = ~(finite & (d == r))
    else:
        bad = ~(finite & (err <= tolerance(S)))
    n_bad = int(bad.sum())
    if n_bad == 0:
        worst = float(np.max(err / tolerance(S))) if d.size and not exact else 0.0
        return True, f"ok ({d.size} elements, worst err/bound {worst:.3g})"
    idx = np.unravel_index(int(np.argmax(bad)), d.shape)
    return False, (f"{n_bad}/{d.size} elements out of bound; first at {idx}: got {d[idx]!r}, "
                   f"oracle {r[idx]!r}, bound {tolerance(S)[idx] if not exact else 0.0!r}")
