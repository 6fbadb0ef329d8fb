"""The C-ABI boundary without a GPU: the library loads, exports every function
that include/tpgemm.h declares, and rejects bad arguments on the host with a
readable reason before anything is enqueued.

The rejection cases mirror the acceptance table of the TVM TIRx synchronous
gemm page ("TVM TIRx 同步 GEMM 深度解析", section 二 What it accepts, and its
tests section: non-unit alpha, fractional beta, unsupported dtypes), restated
for a fixed library entry point: M % 16, N % 8, K % 8; A/B float16 or
bfloat16; beta in {0, 1}. Pointers here are fake addresses; the library never
dereferences them on the rejection paths.
"""
import ctypes
import os
import subprocess
import sys

import pytest

import tile_primitive_tensor_gb300 as tp
from tile_primitive_tensor_gb300 import build as tpbuild

BASE = 0x7F0000000000  # fake, 16-byte aligned device addresses
MB = 1 << 20


@pytest.fixture(scope="module")
def lib():
    tpbuild.build()
    return tp.library()


def call(M=64, N=64, K=64, D=BASE, A=BASE + 64 * MB, B=BASE + 128 * MB, C=BASE + 192 * MB,
         tA=0, tB=0, dtype=tp.TPGEMM_F16, beta=1.0, path=tp.TPGEMM_PATH_AUTO):
    st = tp.tpgemm_gemm_path(D, A, B, C, M, N, K, tA, tB, dtype, beta, 0, path)
    return st, tp.tpgemm_last_error_detail()


def test_exports_every_declared_function(lib):
    names = tp.header_functions()
    assert "tpgemm_gemm" in names and len(names) >= 7
    for n in names:
        assert hasattr(lib, n), f"{n} declared in tpgemm.h but not exported"
    out = subprocess.run(["nm", "-D", "--defined-only", tp.LIB_PATH], capture_output=True,
                         text=True).stdout
    for n in names:
        assert f" T {n}" in out


def test_status_strings(lib):
    for s in range(0, 12):
        assert tp.tpgemm_status_string(s) not in ("", "unknown status")
    assert tp.tpgemm_status_string(99) == "unknown status"
    assert tp.tpgemm_version().count(".") == 2


@pytest.mark.parametrize("M,N,K,frag", [
    (8, 64, 64, "M=8"), (64, 12, 64, "N=12"), (64, 64, 4, "K=4"), (0, 64, 64, "positive"),
    (64, -8, 64, "positive"), (64, 64, 0, "positive"), (24, 64, 64, "M=24"),
    (1 << 30, 64, 64, "2^30"),
    (1 << 19, 1 << 18, 64, "one GPU's memory"), (1 << 20, 64, 1 << 18, "one GPU's memory"),
    (64, 1 << 20, 1 << 18, "one GPU's memory"),
])
def test_rejects_shape(lib, M, N, K, frag):
    st, why = call(M=M, N=N, K=K)
    assert st == tp.TPGEMM_ERR_SHAPE
    assert frag in why


@pytest.mark.parametrize("dtype", [5, 6, -1, 7])
def test_rejects_dtype(lib, dtype):
    # f16 accumulators, tf32, int8 and mixed types have no enumerator: any
    # code other than F16 / BF16 / E4M3 / E5M2 / E2M1 is refused.
    st, why = call(dtype=dtype)
    assert st == tp.TPGEMM_ERR_DTYPE and "dtype" in why


@pytest.mark.parametrize("dtype", [tp.TPGEMM_E4M3, tp.TPGEMM_E5M2])
def test_fp8_rules(lib, dtype):
    # fp8: K a multiple of 16 (whole 16-byte rows), both operands K-contiguous
    # (A [M,K], B [N,K]), tcgen05 kernel only.
    st, why = call(K=72, dtype=dtype, tB=1)
    assert st == tp.TPGEMM_ERR_SHAPE and "multiple of 16" in why
    for tA, tB in ((0, 0), (1, 1), (1, 0)):
        st, text = tp.tpgemm_describe_plan(256, 256, 256, tA, tB, dtype, 0.0)
        assert st == tp.TPGEMM_ERR_PATH and "K-contiguous" in tp.tpgemm_last_error_detail()
    st, text = tp.tpgemm_describe_plan(256, 256, 256, 0, 1, dtype, 0.0)
    assert st == tp.TPGEMM_OK and "kind=f8f6f4" in text and "x128 " in text, text
    st, text = tp.tpgemm_describe_plan(16, 8, 32, 0, 1, dtype, 0.0)
    assert st == tp.TPGEMM_OK and text.startswith("path=tcgen05"), text
    st, _ = tp.tpgemm_describe_plan(256, 256, 256, 0, 1, dtype, 0.0, tp.TPGEMM_PATH_MMA_SYNC)
    assert st == tp.TPGEMM_ERR_PATH
    # operand bytes for aliasing and the host workspace are one per element
    n = tp.tpgemm_gemm_host_workspace_bytes(64, 64, 64, dtype, 0.0)
    assert n == 4096 + 4096 + 16384


@pytest.mark.parametrize("beta", [0.5, 2.0, -1.0, float("nan"), 1e-30])
def test_rejects_fractional_beta(lib, beta):
    st, why = call(beta=beta)
    assert st == tp.TPGEMM_ERR_BETA and "beta" in why


def test_rejects_null_and_misaligned(lib):
    assert call(D=None)[0] == tp.TPGEMM_ERR_NULL
    assert call(A=None)[0] == tp.TPGEMM_ERR_NULL
    assert call(B=None)[0] == tp.TPGEMM_ERR_NULL
    assert call(C=None, beta=1.0)[0] == tp.TPGEMM_ERR_NULL
    for kw in ({"D": BASE + 8}, {"A": BASE + 64 * MB + 2}, {"B": BASE + 128 * MB + 4},
               {"C": BASE + 192 * MB + 12}):
        st, why = call(**kw)
        assert st == tp.TPGEMM_ERR_ALIGN and "16-byte" in why


def test_rejects_aliasing(lib):
    # D = 64x64 f32 = 16 KB at BASE; A starting inside it
    st, why = call(A=BASE + 4096)
    assert st == tp.TPGEMM_ERR_ALIAS and "A" in why
    st, why = call(B=BASE + 16 * 1024 - 16)
    assert st == tp.TPGEMM_ERR_ALIAS and "B" in why
    st, why = call(C=BASE + 16)
    assert st == tp.TPGEMM_ERR_ALIAS and "C" in why
    # B just past the end of D is fine (the call then fails on the missing GPU only)
    st, _ = call(B=BASE + 16 * 1024)
    assert st not in (tp.TPGEMM_ERR_ALIAS,)


def test_c_ignored_when_beta_zero(lib):
    # With beta = 0, C may be NULL, misaligned or overlapping: it is never read.
    for C in (None, BASE + 3, BASE + 16):
        st, why = call(C=C, beta=0.0)
        assert st not in (tp.TPGEMM_ERR_NULL, tp.TPGEMM_ERR_ALIGN, tp.TPGEMM_ERR_ALIAS), why


def test_in_place_accepted(lib):
    # D == C is the in-place form; validation passes (then no GPU here, or a launch).
    st, why = call(C=BASE, beta=1.0)
    assert st not in (tp.TPGEMM_ERR_ALIAS, tp.TPGEMM_ERR_NULL, tp.TPGEMM_ERR_ALIGN), why


def test_plans_for_workloads(lib):
    import workloads as wl
    expect = {
        "atom_16x8x16_f16_int": "path=mma_sync",
        "gemm_256_bf16_transB_beta1": "path=mma_sync",
        "gemm_4096_f16": "path=tcgen05 orientation=swapped",  # B [K,N]: Q = A K-contiguous
        "gemm_8192_bf16_transB_beta1": "path=tcgen05 orientation=normal",
        "skinny_144x16392x4104_f16_beta1": "path=tcgen05 orientation=swapped",
    }
    for w in wl.WORKLOADS:
        st, text = tp.tpgemm_describe_plan(w.M, w.N, w.K, w.transA, w.transB, w.dtype, w.beta)
        assert st == tp.TPGEMM_OK, text
        assert text.startswith(expect[w.name]), (w.name, text)
    st, text = tp.tpgemm_describe_plan(256, 256, 256, 0, 1, tp.TPGEMM_BF16, 1.0,
                                       tp.TPGEMM_PATH_TCGEN05)
    assert st == tp.TPGEMM_OK and "tcgen05" in text
    st, text = tp.tpgemm_describe_plan(64, 64, 64, 0, 0, 0, 1.0, 7)
    assert st == tp.TPGEMM_ERR_PATH


def test_binding_fails_loudly_without_library(tmp_path):
    """A fresh interpreter whose package copy has no built library raises."""
    import shutil
    pkg = os.path.dirname(tp.__file__)
    dst = tmp_path / "tile_primitive_tensor_gb300"
    shutil.copytree(pkg, dst, ignore=shutil.ignore_patterns("_lib", "_build", "__pycache__"))
    code = ("import tile_primitive_tensor_gb300 as t\n"
            "try:\n    t.tpgemm_version()\nexcept RuntimeError as e:\n    print('RAISED', e)\n")
    r = subprocess.run([sys.executable, "-c", code], cwd=tmp_path, capture_output=True, text=True)
    assert "RAISED" in r.stdout and "not built" in r.stdout


def test_host_path_workspace_and_rejections(lib):
    # A (2MK) + B (2KN) + C (4MN, beta = 1) + D (4MN), each 256-byte aligned.
    n = tp.tpgemm_gemm_host_workspace_bytes(64, 64, 64, tp.TPGEMM_F16, 1.0)
    assert n == 8192 + 8192 + 16384 + 16384
    assert tp.tpgemm_gemm_host_workspace_bytes(64, 64, 64, tp.TPGEMM_F16, 0.0) == 8192 + 8192 + 16384
    assert tp.tpgemm_gemm_host_workspace_bytes(64, 12, 64, tp.TPGEMM_F16, 1.0) == 0
    assert tp.tpgemm_gemm_host_workspace_bytes(64, 64, 64, 5, 1.0) == 0
    H = 0x10000
    args = dict(M=64, N=64, K=64, transA=0, transB=0, dtype=tp.TPGEMM_F16, beta=1.0)

    def host(D=H, A=H, B=H, C=H, ws=BASE, wsb=n, **kw):
        a = {**args, **kw}
        return tp.tpgemm_gemm_host(D, A, B, C, a["M"], a["N"], a["K"], a["transA"], a["transB"],
                                   a["dtype"], a["beta"], ws, wsb, 0)
    assert host(M=8) == tp.TPGEMM_ERR_SHAPE
    assert host(beta=0.5) == tp.TPGEMM_ERR_BETA
    assert host(dtype=9) == tp.TPGEMM_ERR_DTYPE
    assert host(A=None) == tp.TPGEMM_ERR_NULL
    assert host(C=None) == tp.TPGEMM_ERR_NULL
    assert host(ws=None) == tp.TPGEMM_ERR_NULL
    assert host(ws=BASE + 64) == tp.TPGEMM_ERR_ALIGN
    assert host(wsb=n - 1) == tp.TPGEMM_ERR_NULL and "needed" in tp.tpgemm_last_error_detail()


def test_header_is_plain_c_and_links(lib, tmp_path):
    """include/tpgemm.h compiles as C99 and a C program links against libtpgemm.so,
    calling entry points that need no GPU (status strings, plans, a rejection)."""
    src = tmp_path / "use.c"
    src.write_text(r"""
#include <stdio.h>
#include <string.h>
#include "tpgemm.h"
int main(void) {
    char buf[512];
    tpgemm_cp_desc d;
    tpgemm_cp_shape sh;
    memset(&d, 0, sizeof d);
    if (tpgemm_describe_plan(8192, 8192, 8192, 0, 1, TPGEMM_BF16, 1.0f, TPGEMM_PATH_AUTO, buf,
                             (int)sizeof buf) != TPGEMM_OK) return 1;
    if (strncmp(buf, "path=tcgen05", 12) != 0) return 2;
    if (tpgemm_cp_parse_shape("64x128b", &sh) != TPGEMM_ERR_SHAPE) return 3;
    d.rows = 128; d.row_bits = 256; d.lbo_bytes = 2048; d.sbo_bytes = 128; d.cta_group = 1;
    if (tpgemm_cp_plan(&d, buf, (int)sizeof buf) != TPGEMM_OK) return 4;
    if (tpgemm_gemm(NULL, NULL, NULL, NULL, 16, 8, 16, 0, 0, TPGEMM_F16, 0.0f, NULL)
        != TPGEMM_ERR_NULL) return 5;
    printf("%s|%s\n", tpgemm_version(), tpgemm_status_string(TPGEMM_ERR_ALIAS));
    return 0;
}
""")
    inc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
    libdir = os.path.dirname(tp.LIB_PATH)
    exe = tmp_path / "use"
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", inc, str(src), "-L", libdir,
                        "-ltpgemm", f"-Wl,-rpath,{libdir}", "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, (r.returncode, r.stdout, r.stderr)
    assert r.stdout.strip() == f"{tp.tpgemm_version()}|{tp.tpgemm_status_string(6)}"


def test_last_plan_before_any_gemm_reports_none():
    # A fresh thread has enqueued nothing (the record is thread-local).
    import threading
    got = {}
    t = threading.Thread(target=lambda: got.update(r=tp.tpgemm_last_plan()))
    t.start()
    t.join()
    st, text = got["r"]
    assert st == tp.TPGEMM_ERR_NULL and text == ""


def test_describe_plan_names_its_scratch(lib, tune):
    # 8192^3: 1024 pair tiles on 76 pairs leave 36 for the last wave, each
    # split into two K halves (stream-K, its flags allocated per stream);
    # TPGEMM_TC_SK=0 splits them along N instead and needs no scratch.
    st, text = tp.tpgemm_describe_plan(8192, 8192, 8192, 0, 1, tp.TPGEMM_BF16, 1.0)
    assert st == tp.TPGEMM_OK and " stream_k=1 scratch=allocated " in text, text
    assert "units=988+36x1 " in text and "sk_clusters=72" in text, text
    tune.setenv("TPGEMM_TC_SK", "0")
    st, text = tp.tpgemm_describe_plan(8192, 8192, 8192, 0, 1, tp.TPGEMM_BF16, 1.0)
    assert st == tp.TPGEMM_OK and " stream_k=0 scratch=none " in text, text
    assert "units=988+36x2 " in text and "sk_clusters=0" in text, text
    # A short K loop keeps the tail split by default (256^3: 4 K blocks).
    tune.delenv("TPGEMM_TC_SK")
    st, text = tp.tpgemm_describe_plan(256, 256, 256, 0, 1, tp.TPGEMM_BF16, 1.0,
                                       tp.TPGEMM_PATH_TCGEN05)
    assert st == tp.TPGEMM_OK and " stream_k=0 " in text, text


# ------------------------------------------------ block-scaled fp8 (MX) boundary
def call_mx(M=256, N=256, K=256, D=BASE, A=BASE + 64 * MB, B=BASE + 128 * MB, C=BASE + 192 * MB,
            SFA=BASE + 256 * MB, SFB=BASE + 257 * MB, dtype=tp.TPGEMM_E4M3, beta=1.0,
            ws=BASE + 320 * MB, ws_bytes=None):
    if ws_bytes is None:
        ws_bytes = tp.tpgemm_gemm_mx_workspace_bytes(M, N, K)
    st = tp.tpgemm_gemm_mx(D, A, B, C, SFA, SFB, M, N, K, dtype, beta, ws, ws_bytes, 0)
    return st, tp.tpgemm_last_error_detail()


def test_mx_workspace_size(lib):
    # 512 bytes per 128-row chunk and 128-element K stage, each chunk stored 4
    # times for tiles of more than 128 rows; sized for the largest of the tile
    # heights a plan can use (multiples of 32 up to 192, or all rows when they
    # fit one tile), A's then B's from a 256-byte boundary. 256 x 256 x 256:
    # 160- or 192-row tiles, 2 tiles x 2 chunks x 4 copies x 2 stages each.
    # 144 x 16392 x 4112 (33 stages): A as one 144-row tile (8 chunk copies),
    # B in 103 tiles of 160 rows (824).
    assert tp.tpgemm_gemm_mx_workspace_bytes(256, 256, 256) == 2 * 16 * 2 * 512
    assert tp.tpgemm_gemm_mx_workspace_bytes(144, 16392, 4112) == (8 + 824) * 33 * 512
    assert tp.tpgemm_gemm_mx_workspace_bytes(0, 8, 16) == 0


@pytest.mark.parametrize("kw,status,frag", [
    ({"dtype": tp.TPGEMM_F16}, tp.TPGEMM_ERR_DTYPE, "E4M3"),
    ({"K": 264}, tp.TPGEMM_ERR_SHAPE, "multiple of 16"),
    ({"SFA": None}, tp.TPGEMM_ERR_NULL, "SFA is NULL"),
    ({"SFB": None}, tp.TPGEMM_ERR_NULL, "SFB is NULL"),
    ({"ws": None}, tp.TPGEMM_ERR_NULL, "workspace is NULL"),
    ({"ws_bytes": 32767}, tp.TPGEMM_ERR_NULL, "32768 needed"),
    ({"ws": BASE + 320 * MB + 16}, tp.TPGEMM_ERR_ALIGN, "256-byte aligned"),
    ({"ws": BASE}, tp.TPGEMM_ERR_ALIAS, "workspace overlaps"),
    ({"SFA": BASE + 16}, tp.TPGEMM_ERR_ALIAS, "scale matrix"),
])
def test_mx_rejections(lib, kw, status, frag):
    st, why = call_mx(**kw)
    assert st == status, why
    assert frag in why



def test_fp4_boundary_rules(lib):
    # fp4: K a multiple of 128 (unpacked by the TMA 128 elements at a time),
    # A and B 32-byte aligned, no host-buffer path.
    st, why = call(M=256, N=256, K=192, tA=0, tB=1, dtype=tp.TPGEMM_E2M1, beta=0.0)
    assert st == tp.TPGEMM_ERR_SHAPE and "multiple of 128" in why
    st, why = call(M=256, N=256, K=256, A=BASE + 64 * MB + 16, tA=0, tB=1, dtype=tp.TPGEMM_E2M1,
                   beta=0.0)
    assert st == tp.TPGEMM_ERR_ALIGN and "32-byte" in why
    st, why = call_mx(K=192, dtype=tp.TPGEMM_E2M1)
    assert st == tp.TPGEMM_ERR_SHAPE and "multiple of 128" in why
    assert tp.tpgemm_gemm_host_workspace_bytes(256, 256, 256, tp.TPGEMM_E2M1, 0.0) == 0



def test_debug_build_compiles_and_exports_the_same_abi():
    # The TPGEMM_DEBUG build (device-side bounds checks) is a second library
    # with the same C ABI; it builds here (nvcc cross-compiles) and loads
    # without a GPU.
    path = tpbuild.build(debug=True)
    assert path.endswith("libtpgemm_debug.so")
    dbg = tp.debug_library()
    assert dbg.tpgemm_version().decode().endswith("-debug")
    for n in tp.header_functions():
        assert hasattr(dbg, n), n
