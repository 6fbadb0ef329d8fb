"""Seeded synthetic inputs for the tile-primitive matrix multiply D = A.B + beta.C.

This module only draws random operands. It holds none of the product's
arithmetic, so both the CPU oracle and the CUDA library can be fed from it
without sharing any code with each other.

Storage conventions (dense, row-major, no leading dimensions):
  A is [M, K], or [K, M] when transA is set (the logical A is its transpose);
  B is [K, N], or [N, K] when transB is set;
  C and D are [M, N] float32.
A and B are float16 or bfloat16 (the same dtype), or both fp8 e4m3 / e5m2.
Values are drawn in float32 and rounded to the dtype with round-to-nearest-even
(torch's cast), so both sides consume the very same bit patterns.

The five workloads are the shapes of the method's test matrix: a single
m16n8k16 atom, a 256^3 transposed-B case with beta = 1, a 4096^3 square case
(plus an integer-valued variant), an 8192^3 bf16 case, and a skinny ragged
144 x 16392 x 4104 case that exercises tail tiles and the memory-bound regime.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch

F16 = 0
BF16 = 1
E4M3 = 2
E5M2 = 3
E2M1 = 4  # fp4: stored packed, two codes per byte (element 2i in the low nibble of byte i)
_TORCH_DTYPE = {F16: torch.float16, BF16: torch.bfloat16, E4M3: torch.float8_e4m3fn,
                E5M2: torch.float8_e5m2}
_DTYPE_NAME = {F16: "f16", BF16: "bf16", E4M3: "e4m3", E5M2: "e5m2", E2M1: "e2m1"}


def elem_bytes(dtype: int) -> float:
    return {E4M3: 1, E5M2: 1, E2M1: 0.5}.get(dtype, 2)


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic problem: shape, dtype, value distributions and flags."""

    name: str
    M: int
    N: int
    K: int
    dtype: int            # F16, BF16, E4M3, E5M2 or E2M1
    a_dist: tuple         # ("int", lo, hi) | ("uniform", lo, hi) | ("normal", mean, std)
    b_dist: tuple
    c_dist: Optional[tuple]  # None when beta == 0
    beta: float
    transA: bool
    transB: bool
    seed: int

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    @property
    def algorithmic_bytes(self) -> int:
        """Each operand read once, D written once; C only when beta = 1."""
        e = elem_bytes(self.dtype)
        b = int(e * (self.M * self.K + self.K * self.N)) + 4 * self.M * self.N
        if self.beta != 0.0:
            b += 4 * self.M * self.N
        return b

    @property
    def integer_valued(self) -> bool:
        return self.a_dist[0] == "int" and self.b_dist[0] == "int" and (
            self.c_dist is None or self.c_dist[0] == "int")

    def describe(self) -> dict:
        return {
            "workload": self.name, "M": self.M, "N": self.N, "K": self.K,
            "dtype": _DTYPE_NAME[self.dtype], "beta": self.beta,
            "transA": self.transA, "transB": self.transB, "seed": self.seed,
        }

    def with_shape(self, M: int, N: int, K: int, name: Optional[str] = None,
                   seed: Optional[int] = None) -> "Workload":
        return dataclasses.replace(self, M=M, N=N, K=K, name=name or f"{self.name}@{M}x{N}x{K}",
                                   seed=self.seed if seed is None else seed)


WORKLOADS = [
    Workload("atom_16x8x16_f16_int", 16, 8, 16, F16, ("int", -2, 2), ("int", -2, 2), None,
             0.0, False, False, 1000),
    Workload("gemm_256_bf16_transB_beta1", 256, 256, 256, BF16, ("normal", 0.0, 1.0),
             ("normal", 0.0, 1.0), ("normal", 0.0, 1.0), 1.0, False, True, 1001),
    Workload("gemm_4096_f16", 4096, 4096, 4096, F16, ("uniform", -1.0, 1.0),
             ("uniform", -1.0, 1.0), None, 0.0, False, False, 1002),
    Workload("gemm_8192_bf16_transB_beta1", 8192, 8192, 8192, BF16, ("normal", 0.0, 0.02),
             ("normal", 0.0, 0.02), ("normal", 0.0, 1.0), 1.0, False, True, 1003),
    Workload("skinny_144x16392x4104_f16_beta1", 144, 16392, 4104, F16, ("normal", 0.0, 1.0),
             ("normal", 0.0, 0.02), ("normal", 0.0, 1.0), 1.0, False, False, 1004),
]
# Integer-valued variant of the 4096^3 case (values in [-3, 3]); every partial
# sum is exactly representable in float32, so results must match bit for bit.
WORKLOAD_4096_INT = Workload("gemm_4096_f16_int", 4096, 4096, 4096, F16, ("int", -3, 3),
                             ("int", -3, 3), None, 0.0, False, False, 1031)

# fp8 cases of the tcgen05 kind::f8f6f4 path: both operands K-contiguous (A
# [M,K], B [N,K]); an integer-valued variant is exact (|sum| <= 9 * 4096).
FP8_WORKLOADS = [
    Workload("gemm_8192_e4m3_transB_beta1", 8192, 8192, 8192, E4M3, ("normal", 0.0, 1.0),
             ("normal", 0.0, 1.0), ("normal", 0.0, 1.0), 1.0, False, True, 1040),
    Workload("gemm_4096_e5m2_transB", 4096, 4096, 4096, E5M2, ("uniform", -1.0, 1.0),
             ("uniform", -1.0, 1.0), None, 0.0, False, True, 1041),
    Workload("gemm_4096_e4m3_int_transB", 4096, 4096, 4096, E4M3, ("int", -3, 3),
             ("int", -3, 3), None, 0.0, False, True, 1042),
    Workload("skinny_144x16392x4112_e4m3_transB_beta1", 144, 16392, 4112, E4M3,
             ("normal", 0.0, 1.0), ("normal", 0.0, 1.0), ("normal", 0.0, 1.0), 1.0, False, True,
             1043),
]


# Block-scaled (MX) fp8 cases: the fp8 operands above plus E8M0 block scales,
# one per MX_BLOCK consecutive K elements of each row of A (SFA [M, KB]) and of
# each column of B (SFB [N, KB]), KB = ceil(K / MX_BLOCK), drawn uniformly from
# the integers sf_dist = (lo, hi) (127 is a scale of 1).
MX_BLOCK = 32


@dataclasses.dataclass(frozen=True)
class MxWorkload(Workload):
    sf_dist: tuple = (120, 134)

    @property
    def kb(self) -> int:
        return -(-self.K // MX_BLOCK)

    @property
    def algorithmic_bytes(self) -> int:
        """The fp8 operands, C and D as for Workload, plus one byte per scale."""
        return super().algorithmic_bytes + (self.M + self.N) * self.kb

    @property
    def integer_valued(self) -> bool:
        # integer operands (fp8) or any fp4 codes (multiples of 1/2 up to 6),
        # with scales within [126, 128] and K <= 4096, keep every partial sum a
        # multiple of 1/16 below 2^20: exact in float32
        lo, hi = self.sf_dist
        ops = self.dtype == E2M1 and self.K <= 4096 or super().integer_valued
        return ops and lo >= 126 and hi <= 128 and (self.c_dist is None or
                                                    self.c_dist[0] == "int")

    def describe(self) -> dict:
        return {**super().describe(), "block_scale": f"E8M0 per {MX_BLOCK} K",
                "scales": list(self.sf_dist)}


MX_WORKLOADS = [
    MxWorkload("mx_256_e4m3_transB_beta1", 256, 256, 256, E4M3, ("normal", 0.0, 1.0),
               ("normal", 0.0, 1.0), ("normal", 0.0, 1.0), 1.0, False, True, 1050),
    MxWorkload("mx_8192_e4m3_transB_beta1", 8192, 8192, 8192, E4M3, ("normal", 0.0, 1.0),
               ("normal", 0.0, 1.0), ("normal", 0.0, 1.0), 1.0, False, True, 1051),
    MxWorkload("mx_4096_e5m2_transB", 4096, 4096, 4096, E5M2, ("uniform", -1.0, 1.0),
               ("uniform", -1.0, 1.0), None, 0.0, False, True, 1052),
    MxWorkload("mx_4096_e4m3_int_transB", 4096, 4096, 4096, E4M3, ("int", -3, 3),
               ("int", -3, 3), None, 0.0, False, True, 1053, sf_dist=(126, 128)),
    MxWorkload("mx_skinny_144x16392x4112_e4m3_transB_beta1", 144, 16392, 4112, E4M3,
               ("normal", 0.0, 1.0), ("normal", 0.0, 1.0), ("normal", 0.0, 1.0), 1.0, False,
               True, 1054),
]

# Block-scaled fp4 (MXFP4): every E2M1 code equally likely. Values are
# multiples of 1/2 up to 6, so with scales in [1/2, 2] every partial sum below
# K = 4096 is a multiple of 1/16 under 2^20: exact in float32.
MX_WORKLOADS += [
    MxWorkload("mxfp4_8192_transB_beta1", 8192, 8192, 8192, E2M1, ("codes", 0, 15),
               ("codes", 0, 15), ("normal", 0.0, 1.0), 1.0, False, True, 1060),
    MxWorkload("mxfp4_4096_int_transB", 4096, 4096, 4096, E2M1, ("codes", 0, 15),
               ("codes", 0, 15), None, 0.0, False, True, 1061, sf_dist=(126, 128)),
]

BY_NAME = {w.name: w for w in WORKLOADS + [WORKLOAD_4096_INT] + FP8_WORKLOADS + MX_WORKLOADS}


def _draw(shape, dist, gen: torch.Generator) -> torch.Tensor:
    kind = dist[0]
    if kind == "int":
        lo, hi = dist[1], dist[2]
        return torch.randint(lo, hi + 1, shape, generator=gen, dtype=torch.int32).to(torch.float32)
    if kind == "uniform":
        lo, hi = dist[1], dist[2]
        return torch.rand(shape, generator=gen, dtype=torch.float32) * (hi - lo) + lo
    if kind == "normal":
        mean, std = dist[1], dist[2]
        return torch.randn(shape, generator=gen, dtype=torch.float32) * std + mean
    if kind == "codes":  # fp4: 4-bit codes drawn uniformly from [lo, hi]
        lo, hi = dist[1], dist[2]
        return torch.randint(lo, hi + 1, shape, generator=gen, dtype=torch.int32)
    raise ValueError(f"unknown distribution {dist!r}")


def pack_fp4(codes: torch.Tensor) -> torch.Tensor:
    """Two 4-bit codes per byte along the last dimension: element 2i in the low
    nibble of byte i, element 2i + 1 in the high nibble."""
    c = codes.to(torch.uint8) & 0xF
    return (c[..., 0::2] | (c[..., 1::2] << 4)).contiguous()


def unpack_fp4(packed: torch.Tensor) -> torch.Tensor:
    p = packed.to(torch.int32)
    out = torch.stack([p & 0xF, (p >> 4) & 0xF], dim=-1)
    return out.reshape(*packed.shape[:-1], packed.shape[-1] * 2)


def stored_shapes(w: Workload):
    a = (w.K, w.M) if w.transA else (w.M, w.K)
    b = (w.N, w.K) if w.transB else (w.K, w.N)
    return a, b, (w.M, w.N)


def make_inputs(w: Workload, c_fill: Optional[float] = None):
    """Return CPU tensors (A, B, C) for a workload.

    A and B are in the workload's dtype and stored orientation; C is
    float32 [M, N], or None when beta == 0 (unless c_fill is given, in which
    case C is a constant-filled tensor, e.g. NaN to prove C is not read).
    """
    gen = torch.Generator("cpu").manual_seed(w.seed)
    sa, sb, sc = stored_shapes(w)
    if w.dtype == E2M1:
        A = pack_fp4(_draw(sa, w.a_dist, gen))
        B = pack_fp4(_draw(sb, w.b_dist, gen))
    else:
        td = _TORCH_DTYPE[w.dtype]
        A = _draw(sa, w.a_dist, gen).to(td)
        B = _draw(sb, w.b_dist, gen).to(td)
    C = None
    if w.c_dist is not None:
        C = _draw(sc, w.c_dist, gen)
    if c_fill is not None:
        C = torch.full(sc, c_fill, dtype=torch.float32)
    return A, B, C


def make_scales(w: MxWorkload):
    """E8M0 block scales (SFA [M, KB], SFB [N, KB]) of an MX workload as uint8
    CPU tensors, from their own seeded stream (the operands stay those of
    make_inputs for the same seed)."""
    gen = torch.Generator("cpu").manual_seed(w.seed + 7919)
    lo, hi = w.sf_dist
    sfa = torch.randint(lo, hi + 1, (w.M, w.kb), generator=gen, dtype=torch.int32)
    sfb = torch.randint(lo, hi + 1, (w.N, w.kb), generator=gen, dtype=torch.int32)
    return sfa.to(torch.uint8), sfb.to(torch.uint8)


def bits(t: torch.Tensor):
    """The raw bit patterns of a float16/bfloat16 CPU tensor as numpy uint16; of an
    fp8 tensor, its byte patterns widened to uint16."""
    if t.dtype in (torch.float8_e4m3fn, torch.float8_e5m2):
        return t.contiguous().view(torch.uint8).numpy().astype("uint16")
    assert t.dtype in (torch.float16, torch.bfloat16)
    return t.contiguous().view(torch.int16).numpy().view("uint16")


def operand_bits(w: Workload, t: torch.Tensor):
    """The element codes of an operand of workload w as numpy uint16, one per
    element (fp4 unpacked from its two-per-byte storage)."""
    if w.dtype == E2M1:
        return unpack_fp4(t).numpy().astype("uint16")
    return bits(t)


def torch_dtype(dtype: int):
    return _TORCH_DTYPE[dtype]
