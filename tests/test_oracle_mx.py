"""Pins for the block-scaled (MX) fp8 oracle (no GPU).

The synchronous gemm page ("TVM TIRx 同步 GEMM 深度解析", section 七) lists
block scaling (SFA, SFB) among the operand forms of gemm_async without
defining it; the oracle takes the OCP Microscaling reading: every `block` (32)
consecutive K elements of a row of A, or of a column of B, share one E8M0
scale 2^(e - 127), and each element's value is its fp8 value times its scale.

These tests tie ``oracle.gemm_mx`` to facts that do not come from it: all
scales 1 reproduce the plain fp8 oracle bit for bit (itself pinned in
test_oracle.py), per-row and per-column powers of two multiply the result
exactly, a hand-worked two-block sum, exact rational arithmetic with an
independent decoder (torch's fp8 conversion) on ragged tiny shapes,
transpose invariance, and NaN scales. The same pins run against planted
mistakes (wrong block size, transposed scale matrix, wrong bias, scales of B
ignored, the ragged last block unscaled, A's and B's scales exchanged), each
made by transforming the inputs of the real oracle, and each must fail one.
"""
from fractions import Fraction

import numpy as np
import pytest

E4M3, E5M2 = 2, 3
TORCH_FP8 = {E4M3: "float8_e4m3fn", E5M2: "float8_e5m2"}


# ------------------------------------------------------------------ helpers
def fp8_bits(x, dtype):
    """Round float32 values to fp8 (torch's RNE cast); 16-bit patterns."""
    import torch
    t = torch.as_tensor(np.asarray(x, dtype=np.float32)).to(getattr(torch, TORCH_FP8[dtype]))
    return t.view(torch.uint8).numpy().astype(np.uint16)


def fp8_values(bits, dtype):
    """Decode with torch (not the oracle's decoder)."""
    import torch
    b = torch.as_tensor(np.asarray(bits, dtype=np.uint8))
    return b.view(getattr(torch, TORCH_FP8[dtype])).to(torch.float64).numpy()


def f32_rne(fr: Fraction) -> np.float32:
    """Round a rational to the nearest float32, ties to even, without double rounding."""
    d = np.float32(float(fr))
    cands = [d, np.nextafter(d, np.float32(np.inf)), np.nextafter(d, np.float32(-np.inf))]
    best = min(cands, key=lambda c: (abs(Fraction(float(c)) - fr),
                                     int(np.asarray(c).view(np.uint32)) & 1))
    return np.float32(best)


def random_case(rng, M, N, K, dtype, block, lo=120, hi=134, tB=True):
    """Finite fp8 operands (A [M,K], B [N,K] or [K,N]) and E8M0 scales in [lo, hi]."""
    kb = -(-K // block)
    a = rng.standard_normal((M, K)) * 2
    b = rng.standard_normal((N, K)) * 2
    A = fp8_bits(a, dtype)
    Bnk = fp8_bits(b, dtype)
    B = Bnk if tB else np.ascontiguousarray(Bnk.T)
    SFA = rng.integers(lo, hi + 1, (M, kb)).astype(np.uint8)
    SFB = rng.integers(lo, hi + 1, (N, kb)).astype(np.uint8)
    return A, B, SFA, SFB


# ---------------------------------------------------------------------- pins
# Each pin takes (gemm_mx, o) and returns (ok, why); gemm_mx has the signature
# of oracle.gemm_mx and o is the oracle module (its plain fp8 gemm is pinned
# elsewhere).
def pin_unit_scales_equal_plain(gemm_mx, o):
    rng = np.random.default_rng(1)
    for dtype, (M, N, K), tB in ((E4M3, (16, 24, 96), True), (E5M2, (8, 40, 70), False)):
        A, B, _, _ = random_case(rng, M, N, K, dtype, 32, tB=tB)
        kb = -(-K // 32)
        one = np.full((M, kb), 127, np.uint8), np.full((N, kb), 127, np.uint8)
        C = rng.standard_normal((M, N)).astype(np.float32)
        D, S = gemm_mx(A, B, C, one[0], one[1], M, N, K, False, tB, dtype, 1.0)
        Dp, Sp = o.gemm(A, B, C, M, N, K, False, tB, dtype, 1.0)
        if not (np.array_equal(D.view(np.uint32), Dp.view(np.uint32)) and np.array_equal(S, Sp)):
            return False, "scales of 1 do not reproduce the plain fp8 product"
    return True, ""


def pin_row_col_powers_of_two(gemm_mx, o):
    # SFA[i, :] = 127 + e_i and SFB[j, :] = 127 + f_j scale D[i, j] by 2^(e_i + f_j),
    # exactly (beta = 0, no overflow or underflow at these sizes).
    rng = np.random.default_rng(2)
    M, N, K = 12, 20, 128
    A, B, _, _ = random_case(rng, M, N, K, E4M3, 32)
    e = rng.integers(-6, 7, M)
    f = rng.integers(-6, 7, N)
    SFA = np.repeat((127 + e)[:, None], 4, 1).astype(np.uint8)
    SFB = np.repeat((127 + f)[:, None], 4, 1).astype(np.uint8)
    D, _ = gemm_mx(A, B, None, SFA, SFB, M, N, K, False, True, E4M3, 0.0)
    Dp, _ = o.gemm(A, B, None, M, N, K, False, True, E4M3, 0.0)
    want = np.ldexp(Dp, e[:, None] + f[None, :]).astype(np.float32)
    return np.array_equal(D, want), "per-row / per-column powers of two are not exact"


def pin_two_blocks_hand_worked(gemm_mx, o):
    # K = 64, two blocks. A row: all 1.0. B column: 1.0 in block 0, 2.0 in
    # block 1. Scales: A block 0 x2 (128), block 1 x0.5 (126); B block 0 x1
    # (127), block 1 x4 (129). D = 32 (1 2 1 1) + 32 (1 0.5 2 4) = 64 + 128 = 192.
    A = fp8_bits(np.ones((1, 64)), E4M3)
    B = fp8_bits(np.concatenate([np.ones(32), 2 * np.ones(32)])[None, :], E4M3)  # [N=1, K]
    SFA = np.array([[128, 126]], np.uint8)
    SFB = np.array([[127, 129]], np.uint8)
    D, S = gemm_mx(A, B, None, SFA, SFB, 1, 1, 64, False, True, E4M3, 0.0)
    return D[0, 0] == 192.0 and S[0, 0] == 192.0, f"two-block sum {D[0, 0]}, want 192"


def pin_exact_rational(gemm_mx, o):
    # Tiny ragged shapes (K not a multiple of the block), both formats, both
    # orientations of B, beta 0 and 1, against exact fractions built from
    # torch's decoding and 2^(e - 127).
    rng = np.random.default_rng(3)
    for (M, N, K, block, dtype, tB, beta) in ((2, 3, 5, 2, E4M3, True, 0.0),
                                               (3, 2, 40, 32, E5M2, False, 1.0),
                                               (2, 2, 70, 32, E4M3, True, 1.0),
                                               (1, 4, 33, 32, E5M2, True, 0.0)):
        A, B, SFA, SFB = random_case(rng, M, N, K, dtype, block, tB=tB)
        C = rng.standard_normal((M, N)).astype(np.float32)
        D, _ = gemm_mx(A, B, C if beta else None, SFA, SFB, M, N, K, False, tB, dtype, beta,
                       block)
        a = fp8_values(A, dtype).reshape(M, K)
        b = fp8_values(B, dtype).reshape((N, K) if tB else (K, N))
        b = b if tB else b.T  # [N, K]
        for i in range(M):
            for j in range(N):
                s = Fraction(0)
                for k in range(K):
                    sa = Fraction(2) ** (int(SFA[i, k // block]) - 127)
                    sb = Fraction(2) ** (int(SFB[j, k // block]) - 127)
                    s += Fraction(a[i, k]) * sa * Fraction(b[j, k]) * sb
                if beta:
                    s += Fraction(float(C[i, j]))
                if D[i, j] != f32_rne(s):
                    return False, f"({i},{j}) of {M}x{N}x{K} block {block}: {D[i, j]} vs {float(s)}"
    return True, ""


def pin_transpose_invariance(gemm_mx, o):
    # The same logical A and B stored the other way give the same D, bit for
    # bit; the scale matrices do not depend on the storage.
    rng = np.random.default_rng(4)
    M, N, K = 8, 12, 96
    A, B, SFA, SFB = random_case(rng, M, N, K, E4M3, 32)
    D1, _ = gemm_mx(A, B, None, SFA, SFB, M, N, K, False, True, E4M3, 0.0)
    At = np.ascontiguousarray(A.reshape(M, K).T)
    Bt = np.ascontiguousarray(B.reshape(N, K).T)
    D2, _ = gemm_mx(At, Bt, None, SFA, SFB, M, N, K, True, False, E4M3, 0.0)
    return np.array_equal(D1.view(np.uint32), D2.view(np.uint32)), "transposed storage differs"


def pin_nan_scale(gemm_mx, o):
    # E8M0 255 is NaN: one such block scale of row i poisons row i only.
    rng = np.random.default_rng(5)
    M, N, K = 4, 6, 64
    A, B, SFA, SFB = random_case(rng, M, N, K, E4M3, 32)
    SFA = SFA.copy()
    SFA[2, 1] = 255
    D, _ = gemm_mx(A, B, None, SFA, SFB, M, N, K, False, True, E4M3, 0.0)
    rows = np.isnan(D).all(axis=1)
    return list(rows) == [False, False, True, False], "NaN scale does not poison exactly its row"


PINS = [pin_unit_scales_equal_plain, pin_row_col_powers_of_two, pin_two_blocks_hand_worked,
        pin_exact_rational, pin_transpose_invariance, pin_nan_scale]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_mx_oracle_pin(oracle_lib, pin):
    ok, why = pin(oracle_lib.gemm_mx, oracle_lib)
    assert ok, why


def test_e8m0_decode_exhaustive(oracle_lib):
    for e in range(255):
        assert oracle_lib.decode_e8m0(e) == 2.0 ** (e - 127)
    assert np.isnan(oracle_lib.decode_e8m0(255))


# ------------------------------------------- planted mistakes (input transforms)
def _mutant(transform):
    """A copy of the oracle whose scale handling is wrong in one way."""
    def make(o):
        def g(A, B, C, SFA, SFB, M, N, K, tA, tB, dtype, beta, block=32):
            SFA, SFB, block2 = transform(np.asarray(SFA, np.uint8), np.asarray(SFB, np.uint8),
                                         M, N, K, block)
            return o.gemm_mx(A, B, C, SFA, SFB, M, N, K, tA, tB, dtype, beta, block2)
        return g
    make.__name__ = transform.__name__
    return make


@_mutant
def block_size_16(SFA, SFB, M, N, K, block):
    # scale index k // 16 instead of k // 32 (clamped to the last scale)
    b2 = block // 2
    kb2 = -(-K // b2)
    idx = np.minimum(np.arange(kb2), SFA.shape[1] - 1)
    return SFA[:, idx], SFB[:, idx], b2


@_mutant
def scale_of_b_transposed(SFA, SFB, M, N, K, block):
    # SFB read as [KB][N] instead of [N][KB]
    kb = SFB.shape[1]
    return SFA, np.ascontiguousarray(SFB.reshape(kb, N).T), block


@_mutant
def bias_128(SFA, SFB, M, N, K, block):
    # 2^(e - 128): every scale halved
    return (np.maximum(SFA.astype(int) - 1, 0).astype(np.uint8),
            np.maximum(SFB.astype(int) - 1, 0).astype(np.uint8), block)


@_mutant
def scales_of_b_ignored(SFA, SFB, M, N, K, block):
    return SFA, np.full_like(SFB, 127), block


@_mutant
def last_block_unscaled(SFA, SFB, M, N, K, block):
    if K % block == 0:
        return SFA, SFB, block
    a, b = SFA.copy(), SFB.copy()
    a[:, -1] = 127
    b[:, -1] = 127
    return a, b, block


@_mutant
def scales_exchanged(SFA, SFB, M, N, K, block):
    # A's and B's scales swapped where the shapes allow it
    if M == N:
        return SFB, SFA, block
    return SFA, SFB, block


MUTANTS = [block_size_16, scale_of_b_transposed, bias_128, scales_of_b_ignored,
           last_block_unscaled, scales_exchanged]


@pytest.mark.parametrize("mutant", MUTANTS, ids=lambda m: m.__name__)
def test_planted_mx_mistake_is_caught(oracle_lib, mutant):
    g = mutant(oracle_lib)
    failures = []
    for pin in PINS:
        try:
            ok, _ = pin(g, oracle_lib)
        except Exception:  # a mutant that crashes a pin is caught too
            ok = False
        if not ok:
            failures.append(pin.__name__)
    assert failures, f"{mutant.__name__} passed every pin"


# ------------------------------------------------------------------- fp4 e2m1
E2M1 = 4
# The OCP Microscaling E2M1 table: codes 0..7 are +0, 0.5, 1, 1.5, 2, 3, 4, 6
# and codes 8..15 the same magnitudes negative.
E2M1_TABLE = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_decode_matches_the_ocp_table(oracle_lib):
    codes = np.arange(16, dtype=np.uint16)
    got = oracle_lib.decode(codes, E2M1)
    want = np.array(E2M1_TABLE + [-v for v in E2M1_TABLE])
    assert np.array_equal(got, want)
    assert np.signbit(got[8]) and not np.signbit(got[0])


def test_fp4_block_scaled_exact_rational(oracle_lib):
    # Random codes and scales on ragged tiny shapes against exact fractions
    # built from the table above.
    rng = np.random.default_rng(11)
    for (M, N, K, block, beta) in ((2, 3, 40, 32, 1.0), (3, 2, 70, 32, 0.0), (2, 2, 9, 4, 1.0)):
        a = rng.integers(0, 16, (M, K)).astype(np.uint16)
        b = rng.integers(0, 16, (N, K)).astype(np.uint16)  # stored [N, K]
        kb = -(-K // block)
        SFA = rng.integers(120, 135, (M, kb)).astype(np.uint8)
        SFB = rng.integers(120, 135, (N, kb)).astype(np.uint8)
        C = rng.standard_normal((M, N)).astype(np.float32)
        D, _ = oracle_lib.gemm_mx(a, b, C if beta else None, SFA, SFB, M, N, K, False, True,
                                  E2M1, beta, block)
        val = lambda c: (-1 if c >= 8 else 1) * Fraction(E2M1_TABLE[c & 7])  # noqa: E731
        for i in range(M):
            for j in range(N):
                s = Fraction(0)
                for k in range(K):
                    s += (val(int(a[i, k])) * Fraction(2) ** (int(SFA[i, k // block]) - 127) *
                          val(int(b[j, k])) * Fraction(2) ** (int(SFB[j, k // block]) - 127))
                if beta:
                    s += Fraction(float(C[i, j]))
                assert D[i, j] == f32_rne(s), (M, N, K, i, j)


def test_fp4_pack_and_unpack_are_inverse():
    import torch

    import workloads as wl
    codes = torch.randint(0, 16, (5, 12), generator=torch.Generator().manual_seed(3))
    packed = wl.pack_fp4(codes)
    assert packed.shape == (5, 6) and packed.dtype == torch.uint8
    assert int(packed[0, 0]) == int(codes[0, 0]) | (int(codes[0, 1]) << 4)
    assert torch.equal(wl.unpack_fp4(packed), codes)
