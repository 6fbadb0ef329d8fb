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
# Debug build (device-side bounds checks; built on request by build(debug=True)).
LIB_PATH_DEBUG = os.path.join(_HERE, "_lib", "libtpgemm_debug.so")
HEADER_PATH = os.path.join(os.path.dirname(_HERE), "include", "tpgemm.h")

# tpgemm_dtype
TPGEMM_F16 = 0
TPGEMM_BF16 = 1
TPGEMM_E4M3 = 2
TPGEMM_E5M2 = 3
TPGEMM_E2M1 = 4  # fp4, packed two per byte (element 2i in the low nibble of byte i)
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
TPGEMM_ERR_BOUNDS = 11
# tpgemm_path
TPGEMM_PATH_AUTO = 0
TPGEMM_PATH_TCGEN05 = 1
TPGEMM_PATH_MMA_SYNC = 2
# tpgemm_cp_swizzle
TPGEMM_CP_SWIZZLE_NONE = 0
TPGEMM_CP_SWIZZLE_32B = 1
TPGEMM_CP_SWIZZLE_64B = 2
TPGEMM_CP_SWIZZLE_128B = 3
# tpgemm_cp_shape
TPGEMM_CP_AUTO = 0
TPGEMM_CP_128x256b = 1
TPGEMM_CP_4x256b = 2
TPGEMM_CP_128x128b = 3
TPGEMM_CP_64x128b_WARPX2_02_13 = 4
TPGEMM_CP_64x128b_WARPX2_01_23 = 5
TPGEMM_CP_32x128b_WARPX4 = 6
# tpgemm_tmem_shape
TPGEMM_TMEM_32x32b = 0
TPGEMM_TMEM_16x64b = 1
TPGEMM_TMEM_16x128b = 2
TPGEMM_TMEM_16x256b = 3
# tpgemm_cp_lanes
TPGEMM_CP_LANES_ROWS = 0
TPGEMM_CP_LANES_QUADRANTS = 1
TPGEMM_CP_LANES_PAIRS_02_13 = 2
TPGEMM_CP_LANES_PAIRS_01_23 = 3
TPGEMM_CP_LANES_ALL_QUADS = 4


class CpDesc(ctypes.Structure):
    """tpgemm_cp_desc: a shared-memory region and where its rows go in tensor memory."""
    _fields_ = [("rows", ctypes.c_int), ("row_bits", ctypes.c_int), ("swizzle", ctypes.c_int),
                ("lbo_bytes", ctypes.c_uint32), ("sbo_bytes", ctypes.c_uint32),
                ("smem_offset", ctypes.c_uint32), ("tmem_col", ctypes.c_int),
                ("lane_offset", ctypes.c_int), ("lanes", ctypes.c_int), ("shape", ctypes.c_int),
                ("cta_group", ctypes.c_int)]


class TpgemmError(RuntimeError):
    def __init__(self, status: int, detail: str):
        self.status = status
        self.detail = detail
        super().__init__(f"tpgemm status {status} ({tpgemm_status_string(status)}): {detail}")


_lib = None
_lock = threading.Lock()


def _open(path):
    """A ctypes handle of a libtpgemm build with every declared signature set."""
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is not built; run tile_primitive_tensor_gb300.build.build() "
            "(nvcc for sm_103a). There is no CPU fallback.")
    lib = ctypes.CDLL(path)
    vp, i64, ci, cf = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
    gemm_args = [vp, vp, vp, vp, i64, i64, i64, ci, ci, ci, cf, vp]
    lib.tpgemm_gemm.argtypes = gemm_args
    lib.tpgemm_gemm.restype = ci
    lib.tpgemm_gemm_path.argtypes = gemm_args + [ci]
    lib.tpgemm_gemm_path.restype = ci
    lib.tpgemm_gemm_noalloc.argtypes = gemm_args
    lib.tpgemm_gemm_noalloc.restype = ci
    lib.tpgemm_test_gemm_withhold_fill.argtypes = gemm_args
    lib.tpgemm_test_gemm_withhold_fill.restype = ci
    lib.tpgemm_reload_tuning.argtypes = []
    lib.tpgemm_reload_tuning.restype = None
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
    lib.tpgemm_last_plan.argtypes = [ctypes.c_char_p, ci]
    lib.tpgemm_last_plan.restype = ci
    u32 = ctypes.c_uint32
    lib.tpgemm_encode_smem_desc.argtypes = [u32, u32, u32, ci]
    lib.tpgemm_encode_smem_desc.restype = ctypes.c_uint64
    lib.tpgemm_encode_idesc.argtypes = [ci, ci, ci, ci, ci]
    lib.tpgemm_encode_idesc.restype = u32
    lib.tpgemm_encode_idesc_mx.argtypes = [ci, ci, ci, ci, ci]
    lib.tpgemm_encode_idesc_mx.restype = u32
    sz = ctypes.c_size_t
    lib.tpgemm_gemm_mx.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i64, ci, cf, vp, sz, vp]
    lib.tpgemm_gemm_mx.restype = ci
    lib.tpgemm_gemm_mx_workspace_bytes.argtypes = [i64, i64, i64]
    lib.tpgemm_gemm_mx_workspace_bytes.restype = sz
    lib.tpgemm_version.argtypes = []
    lib.tpgemm_version.restype = ctypes.c_char_p
    lib.tpgemm_cp_parse_shape.argtypes = [ctypes.c_char_p, ctypes.POINTER(ci)]
    lib.tpgemm_cp_parse_shape.restype = ci
    lib.tpgemm_cp_plan.argtypes = [ctypes.POINTER(CpDesc), ctypes.c_char_p, ci]
    lib.tpgemm_cp_plan.restype = ci
    lib.tpgemm_cp_roundtrip.argtypes = [vp, vp, ctypes.c_size_t, ctypes.POINTER(CpDesc),
                                        ctypes.c_uint32, ci, vp]
    lib.tpgemm_cp_roundtrip.restype = ci
    lib.tpgemm_cp_roundtrip_repeat.argtypes = [vp, vp, ctypes.c_size_t, ctypes.POINTER(CpDesc),
                                               ctypes.c_uint32, ci, ci, ci, ci, vp]
    lib.tpgemm_cp_roundtrip_repeat.restype = ci
    lib.tpgemm_tmem_ldst_roundtrip.argtypes = [vp, vp, vp, ci, ci, ci, ci, ctypes.c_uint32,
                                               vp]
    lib.tpgemm_tmem_ldst_roundtrip.restype = ci
    lib.tpgemm_vcopy_plan.argtypes = [ctypes.POINTER(VcopyDesc), ctypes.c_char_p, ci]
    lib.tpgemm_vcopy_plan.restype = ci
    lib.tpgemm_vcopy_roundtrip.argtypes = [vp, vp, ctypes.c_size_t, ctypes.POINTER(VcopyDesc),
                                           ci, i64, vp, vp]
    lib.tpgemm_vcopy_roundtrip.restype = ci
    return lib


_lib_debug = None


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _open(LIB_PATH)
        return _lib


def debug_library():
    """The ctypes handle of libtpgemm_debug.so (same C ABI, device-side bounds
    checks that report TPGEMM_ERR_BOUNDS); build it with build(debug=True)."""
    global _lib_debug
    with _lock:
        if _lib_debug is None:
            _lib_debug = _open(LIB_PATH_DEBUG)
        return _lib_debug


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


def tpgemm_gemm_mx(D, A, B, C, SFA, SFB, M, N, K, dtype, beta, workspace, workspace_bytes,
                   stream=None) -> int:
    """Enqueue the block-scaled fp8 multiply (A [M,K], B [N,K], E8M0 scales
    SFA [M, ceil(K/32)], SFB [N, ceil(K/32)]); returns the tpgemm_status code."""
    return int(_load().tpgemm_gemm_mx(_ptr(D), _ptr(A), _ptr(B), _ptr(C), _ptr(SFA), _ptr(SFB),
                                      int(M), int(N), int(K), int(dtype), float(beta),
                                      _ptr(workspace), int(workspace_bytes), _stream(stream)))


def tpgemm_gemm_mx_workspace_bytes(M, N, K) -> int:
    return int(_load().tpgemm_gemm_mx_workspace_bytes(int(M), int(N), int(K)))


def tpgemm_encode_idesc_mx(dtype, m, n, a_sf_id, b_sf_id) -> int:
    return int(_load().tpgemm_encode_idesc_mx(int(dtype), int(m), int(n), int(a_sf_id),
                                              int(b_sf_id)))


def tpgemm_test_gemm_withhold_fill(D, A, B, C, M, N, K, transA, transB, dtype, beta,
                                   stream=None) -> int:
    """Test aid: the tcgen05 GEMM with CTA 0's first stage fill withheld."""
    return int(_load().tpgemm_test_gemm_withhold_fill(
        _ptr(D), _ptr(A), _ptr(B), _ptr(C), int(M), int(N), int(K), int(bool(transA)),
        int(bool(transB)), int(dtype), float(beta), _stream(stream)))


def tpgemm_reload_tuning() -> None:
    """Re-read the TPGEMM_* planner overrides from the environment."""
    _load().tpgemm_reload_tuning()


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
    buf = ctypes.create_string_buffer(640)
    st = int(_load().tpgemm_describe_plan(int(M), int(N), int(K), int(bool(transA)),
                                          int(bool(transB)), int(dtype), float(beta), int(path),
                                          buf, 640))
    return st, buf.value.decode()


def tpgemm_encode_smem_desc(start_addr, lbo_bytes, sbo_bytes, swizzle) -> int:
    return int(_load().tpgemm_encode_smem_desc(int(start_addr), int(lbo_bytes), int(sbo_bytes),
                                               int(swizzle)))


def tpgemm_encode_idesc(dtype, a_mn_major, b_mn_major, m, n) -> int:
    return int(_load().tpgemm_encode_idesc(int(dtype), int(bool(a_mn_major)),
                                           int(bool(b_mn_major)), int(m), int(n)))


def tpgemm_last_plan():
    buf = ctypes.create_string_buffer(640)
    st = int(_load().tpgemm_last_plan(buf, 640))
    return st, buf.value.decode()


class VcopyDesc(ctypes.Structure):
    """tpgemm_vcopy_desc: a global region, its shared placement and the copying scope."""
    _fields_ = [("rows", ctypes.c_int), ("cols", ctypes.c_int), ("elem_bytes", ctypes.c_int),
                ("g_row_stride", ctypes.c_int64), ("g_offset", ctypes.c_int64),
                ("s_row_stride", ctypes.c_int), ("s_offset", ctypes.c_int),
                ("s_swizzle", ctypes.c_int), ("threads", ctypes.c_int)]


def vcopy_desc(rows, cols, elem_bytes, *, g_row_stride=None, g_offset=0, s_row_stride=None,
               s_offset=0, s_swizzle=0, threads=32) -> VcopyDesc:
    return VcopyDesc(int(rows), int(cols), int(elem_bytes),
                     int(cols if g_row_stride is None else g_row_stride), int(g_offset),
                     int(cols if s_row_stride is None else s_row_stride), int(s_offset),
                     int(s_swizzle), int(threads))


def tpgemm_vcopy_plan(desc: VcopyDesc):
    buf = ctypes.create_string_buffer(512)
    st = int(_load().tpgemm_vcopy_plan(ctypes.byref(desc), buf, 512))
    return st, buf.value.decode()


def tpgemm_vcopy_roundtrip(dst, src, buffer_bytes, desc: VcopyDesc, ctas=1, cta_stride=0,
                           smem_out=None, stream=None) -> int:
    return int(_load().tpgemm_vcopy_roundtrip(_ptr(dst), _ptr(src), int(buffer_bytes),
                                              ctypes.byref(desc), int(ctas), int(cta_stride),
                                              _ptr(smem_out), _stream(stream)))


def cp_desc(rows, row_bits, *, swizzle=TPGEMM_CP_SWIZZLE_NONE, lbo=0, sbo=0, smem_offset=0,
            tmem_col=0, lane_offset=0, lanes=TPGEMM_CP_LANES_ROWS, shape=TPGEMM_CP_AUTO,
            cta_group=1) -> CpDesc:
    return CpDesc(int(rows), int(row_bits), int(swizzle), int(lbo), int(sbo), int(smem_offset),
                  int(tmem_col), int(lane_offset), int(lanes), int(shape), int(cta_group))


def tpgemm_cp_parse_shape(name: str):
    """(status, tpgemm_cp_shape) for a form name such as "64x128b.warpx2::02_13"."""
    out = ctypes.c_int(0)
    st = int(_load().tpgemm_cp_parse_shape(name.encode(), ctypes.byref(out)))
    return st, out.value


def tpgemm_cp_plan(desc: CpDesc):
    """(status, text): the planned tcgen05.cp instructions, or the rejection reason."""
    buf = ctypes.create_string_buffer(16384)
    st = int(_load().tpgemm_cp_plan(ctypes.byref(desc), buf, 16384))
    return st, buf.value.decode()


def tpgemm_cp_roundtrip(tmem_out, smem_image, image_bytes, desc: CpDesc, fill_base, ncols,
                        stream=None) -> int:
    """Enqueue image -> shared memory -> tcgen05.cp -> tensor memory -> tmem_out."""
    return int(_load().tpgemm_cp_roundtrip(_ptr(tmem_out), _ptr(smem_image), int(image_bytes),
                                           ctypes.byref(desc), int(fill_base) & 0xFFFFFFFF,
                                           int(ncols), _stream(stream)))


def tpgemm_cp_roundtrip_repeat(tmem_out, smem_image, image_bytes, desc: CpDesc, fill_base, ncols,
                               repeat, ctas, issuers=1, stream=None) -> int:
    """The round trip on `ctas` CTAs, each issuing the planned copy `repeat` times from
    `issuers` threads."""
    return int(_load().tpgemm_cp_roundtrip_repeat(_ptr(tmem_out), _ptr(smem_image),
                                                  int(image_bytes), ctypes.byref(desc),
                                                  int(fill_base) & 0xFFFFFFFF, int(ncols),
                                                  int(repeat), int(ctas), int(issuers),
                                                  _stream(stream)))


def tpgemm_tmem_ldst_roundtrip(regs_out, tmem_out, regs_in, st_shape, ld_shape, cols, tmem_col,
                               fill_base, stream=None) -> int:
    """Registers -> tensor memory (st_shape) -> .32x32b read-back and ld_shape load."""
    return int(_load().tpgemm_tmem_ldst_roundtrip(_ptr(regs_out), _ptr(tmem_out), _ptr(regs_in),
                                                  int(st_shape), int(ld_shape), int(cols),
                                                  int(tmem_col), int(fill_base) & 0xFFFFFFFF,
                                                  _stream(stream)))


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
    if torch_dtype == torch.float8_e4m3fn:
        return TPGEMM_E4M3
    if torch_dtype == torch.float8_e5m2:
        return TPGEMM_E5M2
    raise TypeError(f"A and B must be float16, bfloat16, float8_e4m3fn or float8_e5m2, "
                    f"got {torch_dtype}")


def gemm_mx(A, B, SFA, SFB, C=None, *, beta=None, out=None, workspace=None, stream=None,
            dtype=None):
    """Block-scaled fp8 / fp4 D = (A.SA)(B.SB)^T + beta.C on CUDA tensors.

    A is fp8 [M, K], B fp8 [N, K] (same dtype), or both fp4 as uint8 [M, K/2]
    and [N, K/2] (two codes per byte) with dtype=TPGEMM_E2M1; SFA uint8
    [M, ceil(K/32)] and SFB uint8 [N, ceil(K/32)] E8M0 scales, C float32 [M, N].
    The scale-packing workspace is allocated here with torch unless given."""
    import torch
    if beta is None:
        beta = 0.0 if C is None else 1.0
    M, K = A.shape
    N = B.shape[0]
    if dtype == TPGEMM_E2M1:
        K *= 2
    code = dtype if dtype is not None else dtype_code(A.dtype)
    if B.shape[1] != A.shape[1] or A.dtype != B.dtype:
        raise ValueError("A must be [M, K] and B [N, K] of the same fp8 / fp4 dtype")
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=A.device)
    wsb = tpgemm_gemm_mx_workspace_bytes(M, N, K)
    if workspace is None:
        workspace = torch.empty(wsb, dtype=torch.uint8, device=A.device)
    check(tpgemm_gemm_mx(out, A, B, C, SFA, SFB, M, N, K, code, beta, workspace,
                         workspace.numel() * workspace.element_size(), stream))
    return out


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
