"""Python binding of libtpgemm.so: the tile-primitive matrix multiply D = A.B + beta.C.

Argument marshalling only. Every step of the computation runs in the CUDA
kernels of ``libtpgemm.so``; this module turns torch tensors (or raw integer
device pointers) and streams into the C-ABI call declared in
``include/tpgemm.h``. The functions keep the C names; ``gemm`` is a
convenience wrapper that allocates D with torch when no output is given.

There is no fallback: if the library has not been built, every call raises.
Build it with ``tile_primitive_tensor_gb300.build.build()``.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libtpgemm.so")
HEADER_PATH = os.path.join(os.path.dirname(_HERE), "include", "tpgemm.h")

# tpgemm_dtype
TPGEMM_F16 = 0
TPGEMM_BF16 = 1
# tpgemm_status
TPGEMM_OK = 0
TPGEMM_ERR_SHAPE = 1
TPGEMM_ERR_DTYPE = 2
TPGEMM_ERR_BETA = 3
TPGEMM_ERR_NULL = 4
TPGEMM_ERR_ALIGN = 5
TPGEMM_ERR_ALIAS = 6
TPGEMM_ERR_ARCH = 7
TPGEMM_ERR_LAUNCH = 8
TPGEMM_ERR_TIMEOUT = 9
TPGEMM_ERR_PATH = 10
# tpgemm_path
TPGEMM_PATH_AUTO = 0
TPGEMM_PATH_TCGEN05 = 1
TPGEMM_PATH_MMA_SYNC = 2


class TpgemmError(RuntimeError):
    def __init__(self, status: int, detail: str):
        self.status = status
        self.detail = detail
        super().__init__(f"tpgemm status {status} ({tpgemm_status_string(status)}): {detail}")


_lib = None
_lock = threading.Lock()


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is not built; run tile_primitive_tensor_gb300.build.build() "
                "(nvcc for sm_103a). There is no CPU fallback.")
        lib = ctypes.CDLL(LIB_PATH)
        vp, i64, ci, cf = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
        gemm_args = [vp, vp, vp, vp, i64, i64, i64, ci, ci, ci, cf, vp]
        lib.tpgemm_gemm.argtypes = gemm_args
        lib.tpgemm_gemm.restype = ci
        lib.tpgemm_gemm_path.argtypes = gemm_args + [ci]
        lib.tpgemm_gemm_path.restype = ci
        lib.tpgemm_gemm_noalloc.argtypes = gemm_args
        lib.tpgemm_gemm_noalloc.restype = ci
        lib.tpgemm_gemm_host.argtypes = [vp, vp, vp, vp, i64, i64, i64, ci, ci, ci, cf, vp,
                                         ctypes.c_size_t, vp]
        lib.tpgemm_gemm_host.restype = ci
        lib.tpgemm_gemm_host_workspace_bytes.argtypes = [i64, i64, i64, ci, cf]
        lib.tpgemm_gemm_host_workspace_bytes.restype = ctypes.c_size_t
        lib.tpgemm_status_string.argtypes = [ci]
        lib.tpgemm_status_string.restype = ctypes.c_char_p
        lib.tpgemm_last_error_detail.argtypes = []
        lib.tpgemm_last_error_detail.restype = ctypes.c_char_p
        lib.tpgemm_last_device_error.argtypes = []
        lib.tpgemm_last_device_error.restype = ci
        lib.tpgemm_describe_plan.argtypes = [i64, i64, i64, ci, ci, ci, cf, ci, ctypes.c_char_p, ci]
        lib.tpgemm_describe_plan.restype = ci
        lib.tpgemm_version.argtypes = []
        lib.tpgemm_version.restype = ctypes.c_char_p
        _lib = lib
        return lib


def library():
    """The loaded ctypes handle of libtpgemm.so."""
    return _load()


def header_functions():
    """Names of the functions declared in include/tpgemm.h."""
    text = open(HEADER_PATH).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tpgemm_\w+)\s*\(", text)))


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return int(x.data_ptr())
    raise TypeError(f"expected a tensor or an integer device pointer, got {type(x)!r}")


def _stream(s) -> int | None:
    if s is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(s, int):
        return s
    if hasattr(s, "cuda_stream"):
        return int(s.cuda_stream)
    raise TypeError(f"expected a torch.cuda.Stream, an integer cudaStream_t or None, got {type(s)!r}")


def tpgemm_gemm(D, A, B, C, M, N, K, transA, transB, dtype, beta, stream=None) -> int:
    """Enqueue D = A.B + beta.C; returns the tpgemm_status code."""
    return int(_load().tpgemm_gemm(_ptr(D), _ptr(A), _ptr(B), _ptr(C), int(M), int(N), int(K),
                                   int(bool(transA)), int(bool(transB)), int(dtype), float(beta),
                                   _stream(stream)))


def tpgemm_gemm_path(D, A, B, C, M, N, K, transA, transB, dtype, beta, stream=None,
                     path=TPGEMM_PATH_AUTO) -> int:
    return int(_load().tpgemm_gemm_path(_ptr(D), _ptr(A), _ptr(B), _ptr(C), int(M), int(N),
                                        int(K), int(bool(transA)), int(bool(transB)), int(dtype),
                                        float(beta), _stream(stream), int(path)))


def tpgemm_gemm_noalloc(D, A, B, C, M, N, K, transA, transB, dtype, beta, stream=None) -> int:
    """tpgemm_gemm that allocates no device memory (static stream-K scratch)."""
    return int(_load().tpgemm_gemm_noalloc(_ptr(D), _ptr(A), _ptr(B), _ptr(C), int(M), int(N),
                                           int(K), int(bool(transA)), int(bool(transB)),
                                           int(dtype), float(beta), _stream(stream)))


def tpgemm_gemm_host_workspace_bytes(M, N, K, dtype, beta) -> int:
    return int(_load().tpgemm_gemm_host_workspace_bytes(int(M), int(N), int(K), int(dtype),
                                                        float(beta)))


def tpgemm_gemm_host(D_host, A_host, B_host, C_host, M, N, K, transA, transB, dtype, beta,
                     workspace, workspace_bytes, stream=None) -> int:
    """Enqueue D = A.B + beta.C on host buffers (copies pipelined with the multiply)."""
    return int(_load().tpgemm_gemm_host(_ptr(D_host), _ptr(A_host), _ptr(B_host), _ptr(C_host),
                                        int(M), int(N), int(K), int(bool(transA)),
                                        int(bool(transB)), int(dtype), float(beta),
                                        _ptr(workspace), int(workspace_bytes), _stream(stream)))


def tpgemm_status_string(status: int) -> str:
    return _load().tpgemm_status_string(int(status)).decode()


def tpgemm_last_error_detail() -> str:
    return _load().tpgemm_last_error_detail().decode()


def tpgemm_last_device_error() -> int:
    return int(_load().tpgemm_last_device_error())


def tpgemm_describe_plan(M, N, K, transA, transB, dtype, beta, path=TPGEMM_PATH_AUTO):
    buf = ctypes.create_string_buffer(512)
    st = int(_load().tpgemm_describe_plan(int(M), int(N), int(K), int(bool(transA)),
                                          int(bool(transB)), int(dtype), float(beta), int(path),
                                          buf, 512))
    return st, buf.value.decode()


def tpgemm_version() -> str:
    return _load().tpgemm_version().decode()


def check(status: int) -> None:
    if status != TPGEMM_OK:
        raise TpgemmError(status, tpgemm_last_error_detail())


def dtype_code(torch_dtype) -> int:
    import torch
    if torch_dtype == torch.float16:
        return TPGEMM_F16
    if torch_dtype == torch.bfloat16:
        return TPGEMM_BF16
    raise TypeError(f"A and B must be float16 or bfloat16, got {torch_dtype}")


def gemm(A, B, C=None, *, beta=None, transA=False, transB=False, out=None, stream=None,
         path=TPGEMM_PATH_AUTO):
    """D = A.B + beta.C on CUDA tensors; returns D (float32 [M, N]).

    A is [M, K] (or [K, M] with transA), B is [K, N] (or [N, K] with transB),
    C is float32 [M, N]. beta defaults to 1 when C is given, else 0. ``out``
    may be C itself for the in-place form D += A.B.
    """
    import torch
    if beta is None:
        beta = 0.0 if C is None else 1.0
    if A.dim() != 2 or B.dim() != 2:
        raise ValueError("A and B must be 2-D")
    M, K = (A.shape[1], A.shape[0]) if transA else (A.shape[0], A.shape[1])
    Kb, N = (B.shape[1], B.shape[0]) if transB else (B.shape[0], B.shape[1])
    if K != Kb:
        raise ValueError(f"inner dimensions differ: A gives K={K}, B gives K={Kb}")
    if A.dtype != B.dtype:
        raise TypeError("A and B must have the same dtype")
    for name, t in (("A", A), ("B", B), ("C", C), ("out", out)):
        if t is not None and not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous (dense row-major)")
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=A.device)
    check(tpgemm_gemm_path(out, A, B, C if beta else C, M, N, K, transA, transB,
                           dtype_code(A.dtype), beta, stream, path))
    return out
