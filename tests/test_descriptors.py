"""The tcgen05 descriptor encoders, checked on the host against hand-computed
bit patterns (no GPU).

The encoders are the very functions the kernels use (``csrc/ptx.cuh``), called
through the library's host entry points. Each expected value below was
assembled by hand, field by field, from the PTX ISA's tables for tcgen05:

Shared-memory matrix descriptor (64 bits):
  bits  0-13  start address >> 4 (address bits 4-17)
  bits 16-29  leading-dimension byte offset >> 4
  bits 32-45  stride-dimension byte offset >> 4
  bits 46-48  fixed 0b001
  bits 49-51  base offset (0)
  bit  52     LBO mode (0: relative)
  bits 61-63  layout type: 0 none, 2 128-byte swizzle, 4 64-byte, 6 32-byte

Instruction descriptor of kind::f16 / kind::f8f6f4, dense (32 bits):
  bits  4-5   D format (1: f32)
  bits  7-9   A format (f16 0, bf16 1; e4m3 0, e5m2 1)
  bits 10-12  B format
  bit  15     A major-ness (0: K-major, 1: MN-major)
  bit  16     B major-ness
  bits 17-22  N >> 3
  bits 24-28  M >> 4
A field shifted by one position, or a wrong width, changes at least one of
these words.
"""
import re

import pytest

import tile_primitive_tensor_gb300 as tp
from tile_primitive_tensor_gb300 import build as tpbuild


@pytest.fixture(scope="module", autouse=True)
def lib():
    tpbuild.build()
    return tp.library()


SMEM_CASES = [
    # (start, lbo, sbo, swizzle, expected, how the fields add up)
    (0x400, 16, 1024, tp.TPGEMM_CP_SWIZZLE_128B, 0x4000404000010040,
     "K-major stage: start 0x40, LBO 1 << 16, SBO 0x40 << 32, 1 << 46, 2 << 61"),
    (0x21A30, 8192, 1024, tp.TPGEMM_CP_SWIZZLE_128B, 0x40004040020021A3,
     "MN-major atoms: start 0x21A3, LBO 0x200 << 16, SBO 0x40 << 32, 1 << 46, 2 << 61"),
    (0x0, 16, 512, tp.TPGEMM_CP_SWIZZLE_64B, 0x8000402000010000,
     "64-byte swizzle: LBO 1 << 16, SBO 0x20 << 32, 1 << 46, 4 << 61"),
    (0x3FFF0, 16, 256, tp.TPGEMM_CP_SWIZZLE_32B, 0xC000401000013FFF,
     "32-byte swizzle, largest start: 0x3FFF, LBO 1 << 16, SBO 0x10 << 32, 1 << 46, 6 << 61"),
    (0x1230, 128, 256, tp.TPGEMM_CP_SWIZZLE_NONE, 0x0000401000080123,
     "no swizzle: start 0x123, LBO 8 << 16, SBO 0x10 << 32, 1 << 46"),
    (0x40010, 16, 1024, tp.TPGEMM_CP_SWIZZLE_128B, 0x4000404000010001,
     "start beyond 256 KB keeps address bits 4-17 only: 0x4001 & 0x3FFF = 1"),
]


@pytest.mark.parametrize("start,lbo,sbo,swz,expected,how", SMEM_CASES,
                         ids=[c[-1].split(":")[0] for c in SMEM_CASES])
def test_shared_memory_descriptor(start, lbo, sbo, swz, expected, how):
    got = tp.tpgemm_encode_smem_desc(start, lbo, sbo, swz)
    assert got == expected, f"{how}: got {got:#018x}, want {expected:#018x}"


IDESC_CASES = [
    # (dtype, a_mn, b_mn, M, N, expected, how)
    (tp.TPGEMM_BF16, 0, 0, 128, 256, 0x08400490,
     "bf16 K/K 128x256: 1 << 4, 1 << 7, 1 << 10, 32 << 17, 8 << 24"),
    (tp.TPGEMM_F16, 1, 0, 256, 144, 0x10248010,
     "f16 A MN-major, 256x144: 1 << 4, 1 << 15, 18 << 17, 16 << 24"),
    (tp.TPGEMM_E5M2, 0, 0, 128, 64, 0x08100490,
     "e5m2 K/K 128x64: 1 << 4, 1 << 7, 1 << 10, 8 << 17, 8 << 24"),
    (tp.TPGEMM_F16, 1, 1, 128, 16, 0x08058010,
     "f16 MN/MN 128x16: 1 << 4, 1 << 15, 1 << 16, 2 << 17, 8 << 24"),
    (tp.TPGEMM_E4M3, 0, 0, 256, 256, 0x10400010,
     "e4m3 K/K 256x256: 1 << 4, 32 << 17, 16 << 24"),
    (tp.TPGEMM_E2M1, 0, 0, 128, 128, 0x08201690,
     "e2m1 K/K 128x128: 1 << 4, 5 << 7, 5 << 10, 16 << 17, 8 << 24"),
]


@pytest.mark.parametrize("dtype,a_mn,b_mn,m,n,expected,how", IDESC_CASES,
                         ids=[c[-1].split(":")[0] for c in IDESC_CASES])
def test_instruction_descriptor(dtype, a_mn, b_mn, m, n, expected, how):
    got = tp.tpgemm_encode_idesc(dtype, a_mn, b_mn, m, n)
    assert got == expected, f"{how}: got {got:#010x}, want {expected:#010x}"


def test_instruction_descriptor_rejects_unknown_dtype():
    assert tp.tpgemm_encode_idesc(7, 0, 0, 128, 128) == 0


def test_start_address_patch_equals_full_encode():
    # The kernels encode once with start 0 and OR in each stage's address.
    base = tp.tpgemm_encode_smem_desc(0, 16, 1024, tp.TPGEMM_CP_SWIZZLE_128B)
    assert base & 0x3FFF == 0
    for addr in (0x400, 0x8C20, 0x3FFF0):
        assert base | (addr >> 4) == tp.tpgemm_encode_smem_desc(addr, 16, 1024,
                                                                tp.TPGEMM_CP_SWIZZLE_128B)


@pytest.mark.parametrize("swz,lbo,sbo,expected", [
    # A swizzled source keeps LBO = 16 bytes (each instruction stays inside one
    # swizzle row); an unswizzled one carries the caller's LBO.
    (tp.TPGEMM_CP_SWIZZLE_128B, 2048, 1024, 0x4000404000010000),
    (tp.TPGEMM_CP_SWIZZLE_NONE, 2048, 128, 0x0000400800800000),
])
def test_tcgen05_cp_plan_descriptor(swz, lbo, sbo, expected):
    d = tp.cp_desc(128, 256, swizzle=swz, lbo=lbo, sbo=sbo, lanes=tp.TPGEMM_CP_LANES_ROWS,
                   shape=tp.TPGEMM_CP_128x256b)
    st, text = tp.tpgemm_cp_plan(d)
    assert st == tp.TPGEMM_OK, text
    got = int(re.search(r"desc=(0x[0-9a-f]+)", text).group(1), 16)
    assert got == expected, f"got {got:#018x}, want {expected:#018x}"


# Block-scaled kind::mxf8f6f4 instruction descriptor (32 bits), hand-assembled
# from the PTX ISA's table for the block-scaled kinds:
#   bits  4-5   B scale-factor ID     bits 17-22  N >> 3
#   bits  7-9   A format (e4m3 0,     bit  23     scale type (1: E8M0)
#               e5m2 1)               bits 24-28  M >> 4
#   bits 10-12  B format              bits 29-30  A scale-factor ID
#   bits 15/16  A/B major (0: K)      (no D-format field: always f32)
IDESC_MX_CASES = [
    (tp.TPGEMM_E4M3, 128, 128, 0, 0, 0x08A00000,
     "e4m3 128x128 ids 0/0: 16 << 17, 1 << 23, 8 << 24"),
    (tp.TPGEMM_E5M2, 128, 144, 3, 2, 0x68A404A0,
     "e5m2 128x144 ids 3/2: 2 << 4, 1 << 7, 1 << 10, 18 << 17, 1 << 23, 8 << 24, 3 << 29"),
    (tp.TPGEMM_E4M3, 128, 16, 1, 1, 0x28840010,
     "e4m3 128x16 ids 1/1: 1 << 4, 2 << 17, 1 << 23, 8 << 24, 1 << 29"),
    (tp.TPGEMM_E2M1, 256, 192, 0, 0, 0x10B01680,
     "e2m1 256x192 ids 0/0: 5 << 7, 5 << 10, 24 << 17, 1 << 23, 16 << 24"),
]


@pytest.mark.parametrize("dtype,m,n,a_id,b_id,expected,how", IDESC_MX_CASES,
                         ids=[c[-1].split(":")[0] for c in IDESC_MX_CASES])
def test_block_scaled_instruction_descriptor(dtype, m, n, a_id, b_id, expected, how):
    got = tp.tpgemm_encode_idesc_mx(dtype, m, n, a_id, b_id)
    assert got == expected, f"{how}: got {got:#010x}, want {expected:#010x}"


def test_block_scaled_descriptor_takes_fp8_only():
    assert tp.tpgemm_encode_idesc_mx(tp.TPGEMM_BF16, 128, 128, 0, 0) == 0
