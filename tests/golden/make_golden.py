"""Write the small golden fixtures in this folder.

Every stored expected value here comes from the CPU oracle (``oracle/``) on
the seeded inputs of ``workloads.py``; nothing is taken from the CUDA library.
Run from the repository root:  python tests/golden/make_golden.py
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import workloads as wl  # noqa: E402

CASES = [
    # (workload, header lines)
    (wl.WORKLOADS[0], [
        "Single mma atom D[16,8] = A[16,16] . B[16,8], fp16 integer inputs in [-2, 2], beta = 0.",
        "Shape and semantics: TVM TIRx synchronous gemm page (同步 GEMM 深度解析), section 三",
        "(one warp computes 16x16 . 16x8, exactly one m16n8k16 atom) and section 语义定义.",
    ]),
    (wl.WORKLOADS[1].with_shape(48, 40, 24, name="ragged_48x40x24_bf16_transB_beta1", seed=2001), [
        "Ragged bf16 case M=48 N=40 K=24 (K not a multiple of 16), B stored [N,K], beta = 1.",
        "Semantics: TVM TIRx synchronous gemm page, sections 语义定义, 二 (transpose flags set",
        "the logical orientation only; beta = 1 starts the accumulator from C).",
    ]),
]


def fmt_bits(a):
    return "\n".join(" ".join(f"{int(v):04x}" for v in row) for row in a)


def fmt_f32(a):
    return "\n".join(" ".join(f"{int(v):08x}" for v in row.view(np.uint32)) for row in a)


def write_case(w, header):
    A, B, C = wl.make_inputs(w)
    Ab, Bb = wl.bits(A), wl.bits(B)
    Cn = None if C is None else C.numpy()
    D, _ = oracle.gemm(Ab, Bb, Cn, w.M, w.N, w.K, w.transA, w.transB, w.dtype, w.beta)
    path = os.path.join(HERE, f"{w.name}.txt")
    with open(path, "w") as f:
        for h in header:
            f.write(f"# {h}\n")
        f.write("# Expected D written by tests/golden/make_golden.py from the CPU oracle.\n")
        f.write(f"# M={w.M} N={w.N} K={w.K} dtype={'f16' if w.dtype == 0 else 'bf16'} "
                f"beta={w.beta} transA={int(w.transA)} transB={int(w.transB)} seed={w.seed}\n")
        f.write(f"[A_bits {A.shape[0]}x{A.shape[1]}]\n{fmt_bits(Ab.reshape(A.shape))}\n")
        f.write(f"[B_bits {B.shape[0]}x{B.shape[1]}]\n{fmt_bits(Bb.reshape(B.shape))}\n")
        if Cn is not None:
            f.write(f"[C_f32bits {w.M}x{w.N}]\n{fmt_f32(Cn)}\n")
        f.write(f"[D_f32bits {w.M}x{w.N}]\n{fmt_f32(D)}\n")
    return path


def read_case(path):
    """Parse a fixture into a dict of header fields and numpy arrays."""
    out = {}
    key = None
    rows = []
    meta = {}
    for line in open(path):
        line = line.strip()
        if line.startswith("# M="):
            for tok in line[2:].split():
                k, v = tok.split("=")
                meta[k] = v
        if not line or line.startswith("#"):
            continue
        if line.startswith("["):
            if key:
                out[key] = rows
            key, rows = line[1:-1].split()[0], []
            continue
        rows.append([int(t, 16) for t in line.split()])
    if key:
        out[key] = rows
    arrs = {}
    for k, v in out.items():
        a = np.array(v, dtype=np.uint64)
        arrs[k] = a.astype(np.uint16) if k.endswith("_bits") else a.astype(np.uint32).view(np.float32)
    arrs["meta"] = meta
    return arrs


if __name__ == "__main__":
    oracle.build()
    for w, h in CASES:
        print(write_case(w, h))
