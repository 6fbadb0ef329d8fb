"""Pins for the CPU oracle (no GPU).

The oracle is the definition of D = A.B + beta.C evaluated in double and
rounded once to float32. These tests tie it to facts that do not come from
the oracle itself: exhaustive decoding against numpy's own float16 and the
bf16 = upper-half-of-binary32 definition, hand-derived closed forms for a
single 16x8x16 atom, identity and permutation matrices, the beta relation,
transpose invariance, brute-force enumeration against exact integer sums,
and exact rational arithmetic on random real inputs.

Every pin is a function of a ``gemm`` callable, so the same pins are also run
against deliberately broken copies of the oracle (a dropped term, a flipped
transpose, a wrong sign on C, float32 accumulation, truncating rounding, a
decoder that flushes subnormals) to show that each such mistake is caught.
The semantics come from the TVM TIRx synchronous gemm page ("TVM TIRx 同步
GEMM 深度解析"): section 语义定义 (D = alpha*A*B + beta*C), section 二
(alpha = 1, beta in {0, 1}, fp16/bf16 inputs, fp32 accumulator, transpose
flags as logical orientation) and section 四 step 3 (initialise from C or 0,
accumulate over K).
"""
import itertools
from fractions import Fraction

import numpy as np
import pytest

import workloads as wl

F16, BF16 = 0, 1
NP16 = {F16: np.float16}


# ---------------------------------------------------------------------------
# helpers that encode values as 16-bit patterns independently of the oracle
# ---------------------------------------------------------------------------
def f16_bits(x):
    return np.asarray(x, dtype=np.float16).view(np.uint16)


def bf16_bits(x):
    """Round float32 values to bf16 with round-to-nearest-even (via torch)."""
    import torch
    t = torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def enc(x, dtype):
    return f16_bits(x) if dtype == F16 else bf16_bits(x)


def ref_decode(bits, dtype):
    """Decode with numpy only (not the oracle's decoder)."""
    b = np.asarray(bits, dtype=np.uint16)
    if dtype == F16:
        return b.view(np.float16).astype(np.float64)
    with np.errstate(invalid="ignore"):
        return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f32_round_exact(fr: Fraction) -> np.float32:
    """Correct rounding of a rational that is exactly a double (asserted)."""
    d = float(fr)
    assert Fraction(d) == fr, "sum not exactly representable in double; pick smaller inputs"
    return np.float32(d)


# ---------------------------------------------------------------------------
# the pins: each takes gemm(A_bits, B_bits, C, M, N, K, tA, tB, dtype, beta)
# -> (D, S) and a decode(bits, dtype) callable, and returns (ok, why)
# ---------------------------------------------------------------------------
def pin_decode_f16(gemm, decode):
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = decode(bits, F16)
    want = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(want)
    ok = np.array_equal(np.isnan(got), nan) and np.array_equal(got[~nan], want[~nan]) and \
        np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))
    return ok, "fp16 decode differs from numpy.float16"


def pin_decode_bf16(gemm, decode):
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = decode(bits, BF16)
    with np.errstate(invalid="ignore"):
        want = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    nan = np.isnan(want)
    ok = np.array_equal(np.isnan(got), nan) and np.array_equal(got[~nan], want[~nan]) and \
        np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))
    return ok, "bf16 decode differs from (bits << 16) as binary32"


def pin_atom_ones_ramp(gemm, decode):
    # A = all ones (16x16), B[k][j] = j - 4  =>  D[i][j] = 16 (j - 4) exactly.
    for dtype in (F16, BF16):
        A = enc(np.ones((16, 16)), dtype)
        B = enc(np.tile(np.arange(8) - 4.0, (16, 1)), dtype)
        D, _ = gemm(A, B, None, 16, 8, 16, False, False, dtype, 0.0)
        want = np.tile(16.0 * (np.arange(8) - 4), (16, 1)).astype(np.float32)
        if not np.array_equal(D, want):
            return False, "ones x ramp atom"
    return True, ""


def atom_mod5_closed_form():
    """D[i][j] for A[i][k] = ((i+2k) mod 5) - 2, B[k][j] = ((3k+j) mod 5) - 2, K = 16.

    Derivation (by hand): both factors have period 5 in k. Over one period,
    with x = (i+2k) mod 5, k = 3(x-i) mod 5 and so (3k+j) mod 5 = (i+j-x) mod 5;
    summing (x-2)((c-x) mod 5 - 2) over x = 0..4 for c = (i+j) mod 5 gives
    P(c) = 0, 5, 5, 0, -10 for c = 0..4. K = 16 is three full periods (k = 0..14)
    plus k = 15, which repeats k = 0: D = 3 P(c) + ((i mod 5) - 2)((j mod 5) - 2).
    """
    P = [0, 5, 5, 0, -10]
    i = np.arange(16)[:, None]
    j = np.arange(8)[None, :]
    return (3 * np.take(P, (i + j) % 5) + ((i % 5) - 2) * ((j % 5) - 2)).astype(np.float32)


def pin_atom_mod5(gemm, decode):
    i = np.arange(16)[:, None]
    k = np.arange(16)[None, :]
    Aval = ((i + 2 * k) % 5) - 2
    kk = np.arange(16)[:, None]
    j = np.arange(8)[None, :]
    Bval = ((3 * kk + j) % 5) - 2
    want = atom_mod5_closed_form()
    # four entries summed by hand from the derivation above
    hand = {(0, 0): 4, (1, 0): 17, (0, 1): 17, (2, 2): -30, (3, 4): 17, (15, 7): 15, (4, 1): -2}
    for (r, c), v in hand.items():
        assert want[r, c] == v
    for dtype in (F16, BF16):
        D, _ = gemm(enc(Aval, dtype), enc(Bval, dtype), None, 16, 8, 16, False, False, dtype, 0.0)
        if not np.array_equal(D, want):
            return False, "mod-5 atom closed form"
    return True, ""


def pin_identity(gemm, decode):
    rng = np.random.default_rng(7)
    for dtype in (F16, BF16):
        n, N = 48, 40
        eye = enc(np.eye(n), dtype)
        B = enc(rng.standard_normal((n, N)).astype(np.float32), dtype)
        D, _ = gemm(eye, B, None, n, N, n, False, False, dtype, 0.0)
        if not np.array_equal(D, ref_decode(B, dtype).reshape(n, N).astype(np.float32)):
            return False, "I.B != B"
        M = 24
        A = enc(rng.standard_normal((M, n)).astype(np.float32), dtype)
        eyeN = enc(np.eye(n), dtype)
        D, _ = gemm(A, eyeN, None, M, n, n, False, False, dtype, 0.0)
        if not np.array_equal(D, ref_decode(A, dtype).reshape(M, n).astype(np.float32)):
            return False, "A.I != A"
    return True, ""


def pin_permutation(gemm, decode):
    rng = np.random.default_rng(11)
    n = 32
    for dtype in (F16, BF16):
        perm = rng.permutation(n)
        P = np.zeros((n, n))
        P[np.arange(n), perm] = 1.0
        B = enc(rng.standard_normal((n, n)).astype(np.float32), dtype)
        Bv = ref_decode(B, dtype).reshape(n, n)
        for tA in (False, True):
            Ast = enc(P.T if tA else P, dtype)
            D, _ = gemm(Ast, B, None, n, n, n, tA, False, dtype, 0.0)
            if not np.array_equal(D, Bv[perm].astype(np.float32)):
                return False, f"P.B rows not permuted (transA={tA})"
        # right-multiplication permutes columns: (B.P)[:, c] = B[:, j] where P[j, c] = 1
        D, _ = gemm(B, enc(P, dtype), None, n, n, n, False, False, dtype, 0.0)
        inv = np.argsort(perm)
        if not np.array_equal(D, Bv[:, inv].astype(np.float32)):
            return False, "B.P columns not permuted"
    return True, ""


def pin_beta(gemm, decode):
    rng = np.random.default_rng(3)
    M, N, K = 32, 24, 40
    for dtype in (F16, BF16):
        A = enc(rng.integers(-3, 4, (M, K)), dtype)
        B = enc(rng.integers(-3, 4, (K, N)), dtype)
        C = rng.integers(-50, 51, (M, N)).astype(np.float32)
        D0, _ = gemm(A, B, None, M, N, K, False, False, dtype, 0.0)
        D1, _ = gemm(A, B, C, M, N, K, False, False, dtype, 1.0)
        if not np.array_equal(D1 - C, D0):
            return False, "D(beta=1) - C != D(beta=0)"
        Cnan = np.full((M, N), np.nan, dtype=np.float32)
        Dn, _ = gemm(A, B, Cnan, M, N, K, False, False, dtype, 0.0)
        if np.isnan(Dn).any() or not np.array_equal(Dn, D0):
            return False, "beta = 0 read C"
        # in-place form of the page's demo (C position passed D itself)
        D2, _ = gemm(A, B, D0, M, N, K, False, False, dtype, 1.0)
        if not np.array_equal(D2, 2 * D0):
            return False, "D += A.B with C = D"
    return True, ""


def pin_transpose(gemm, decode):
    rng = np.random.default_rng(5)
    M, N, K = 24, 40, 56
    for dtype in (F16, BF16):
        a = rng.standard_normal((M, K)).astype(np.float32)
        b = rng.standard_normal((K, N)).astype(np.float32)
        A, At = enc(a, dtype), enc(a.T.copy(), dtype)
        B, Bt = enc(b, dtype), enc(b.T.copy(), dtype)
        C = rng.standard_normal((M, N)).astype(np.float32)
        D00, _ = gemm(A, B, C, M, N, K, False, False, dtype, 1.0)
        for tA, tB in itertools.product((False, True), repeat=2):
            D, _ = gemm(At if tA else A, Bt if tB else B, C, M, N, K, tA, tB, dtype, 1.0)
            if not np.array_equal(D.view(np.uint32), D00.view(np.uint32)):
                return False, f"transpose combo ({tA},{tB}) differs"
    return True, ""


def pin_bruteforce_ternary(gemm, decode):
    vals = (-1.0, 0.0, 1.0)
    for (M, N, K) in [(1, 1, 1), (1, 1, 2), (2, 1, 1), (1, 2, 2), (2, 2, 1), (2, 2, 2)]:
        for combo in itertools.product(vals, repeat=M * K + K * N):
            a = np.array(combo[:M * K]).reshape(M, K)
            b = np.array(combo[M * K:]).reshape(K, N)
            want = (a.astype(np.int64) @ b.astype(np.int64)).astype(np.float32)
            D, _ = gemm(f16_bits(a), f16_bits(b), None, M, N, K, False, False, F16, 0.0)
            if not np.array_equal(D, want):
                return False, f"ternary brute force {M}x{N}x{K} {combo}"
    return True, ""


def pin_exact_rational(gemm, decode):
    """Random real inputs: D must be the correctly rounded exact sum."""
    rng = np.random.default_rng(13)
    M, N, K = 8, 8, 24
    for dtype in (F16, BF16):
        A = enc(rng.standard_normal((M, K)).astype(np.float32), dtype)
        B = enc(rng.standard_normal((K, N)).astype(np.float32), dtype)
        C = rng.standard_normal((M, N)).astype(np.float32)
        a = ref_decode(A, dtype).reshape(M, K)
        b = ref_decode(B, dtype).reshape(K, N)
        for beta in (0.0, 1.0):
            D, S = gemm(A, B, C, M, N, K, False, False, dtype, beta)
            for i in range(M):
                for j in range(N):
                    s = sum(Fraction(a[i, k]) * Fraction(b[k, j]) for k in range(K))
                    sa = sum(abs(Fraction(a[i, k]) * Fraction(b[k, j])) for k in range(K))
                    if beta:
                        s += Fraction(float(C[i, j]))
                    if D[i, j] != f32_round_exact(s):
                        return False, f"not correctly rounded at ({i},{j}) beta={beta}"
                    if S[i, j] != float(sa):
                        return False, f"sum |ab| wrong at ({i},{j})"
    return True, ""


def pin_numpy_matmul(gemm, decode):
    """Moderate random case against numpy's float64 matmul of independently decoded inputs."""
    rng = np.random.default_rng(17)
    M, N, K = 64, 48, 96
    for dtype in (F16, BF16):
        A = enc(rng.standard_normal((K, M)).astype(np.float32), dtype)   # stored [K, M]
        B = enc(rng.standard_normal((N, K)).astype(np.float32), dtype)   # stored [N, K]
        C = rng.standard_normal((M, N)).astype(np.float32)
        a = ref_decode(A, dtype).reshape(K, M).T
        b = ref_decode(B, dtype).reshape(N, K).T
        D, S = gemm(A, B, C, M, N, K, True, True, dtype, 1.0)
        want = a @ b + C.astype(np.float64)
        # both are within a few double ulps of the exact sum; after rounding to
        # float32 they agree to one float32 ulp at most (ties aside)
        ulp = np.spacing(np.abs(want).astype(np.float32)).astype(np.float64)
        if not np.all(np.abs(D.astype(np.float64) - want) <= ulp):
            return False, "differs from numpy float64 matmul by more than 1 ulp"
        wantS = np.abs(a) @ np.abs(b)
        if not np.allclose(S, wantS, rtol=1e-12, atol=0):
            return False, "S differs from |A|.|B|"
    return True, ""


PINS = [pin_decode_f16, pin_decode_bf16, pin_atom_ones_ramp, pin_atom_mod5, pin_identity,
        pin_permutation, pin_beta, pin_transpose, pin_bruteforce_ternary, pin_exact_rational,
        pin_numpy_matmul]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_oracle_pin(oracle_lib, pin):
    ok, why = pin(oracle_lib.gemm, oracle_lib.decode)
    assert ok, why


# ---------------------------------------------------------------------------
# planted mistakes: every broken copy of the oracle must fail at least one pin
# ---------------------------------------------------------------------------
def _mutant_dropped_term(o):
    def g(A, B, C, M, N, K, tA, tB, dtype, beta):
        A2 = np.array(A, dtype=np.uint16).reshape((K, M) if tA else (M, K)).copy()
        if tA:
            A2[K - 1, :] = 0
        else:
            A2[:, K - 1] = 0
        return o.gemm(A2.ravel(), B, C, M, N, K, tA, tB, dtype, beta)
    return g, o.decode


def _mutant_transposed_b(o):
    def g(A, B, C, M, N, K, tA, tB, dtype, beta):
        if K == N:
            return o.gemm(A, B, C, M, N, K, tA, not tB, dtype, beta)
        return o.gemm(A, B, C, M, N, K, tA, tB, dtype, beta)
    return g, o.decode


def _mutant_transposed_a(o):
    def g(A, B, C, M, N, K, tA, tB, dtype, beta):
        if K == M:
            return o.gemm(A, B, C, M, N, K, not tA, tB, dtype, beta)
        return o.gemm(A, B, C, M, N, K, tA, tB, dtype, beta)
    return g, o.decode


def _mutant_minus_c(o):
    def g(A, B, C, M, N, K, tA, tB, dtype, beta):
        if C is not None and beta:
            C = -np.asarray(C, dtype=np.float32)
        return o.gemm(A, B, C, M, N, K, tA, tB, dtype, beta)
    return g, o.decode


def _mutant_always_adds_c(o):
    def g(A, B, C, M, N, K, tA, tB, dtype, beta):
        return o.gemm(A, B, C, M, N, K, tA, tB, dtype, 1.0 if C is not None else beta)
    return g, o.decode


def _numpy_variant(o, accum, final_round):
    """A restatement with a planted arithmetic mistake (float32 sums or truncation)."""
    def g(A, B, C, M, N, K, tA, tB, dtype, beta):
        a = o.decode(np.asarray(A, dtype=np.uint16), dtype).reshape((K, M) if tA else (M, K))
        b = o.decode(np.asarray(B, dtype=np.uint16), dtype).reshape((N, K) if tB else (K, N))
        a = a.T if tA else a
        b = b.T if tB else b
        D = np.empty((M, N), np.float32)
        S = np.abs(a) @ np.abs(b)
        for i in range(M):
            for j in range(N):
                s = accum(0.0)
                for k in range(K):
                    s = accum(s + accum(a[i, k] * b[k, j]))
                if beta:
                    s = accum(s + accum(C[i, j]))
                D[i, j] = final_round(float(s))
        return D, S
    return g, o.decode


def _trunc_to_f32(x: float) -> np.float32:
    f = np.float32(x)
    if abs(float(f)) > abs(x):
        f = np.nextafter(f, np.float32(0))
    return f


def _mutant_fp32_accum(o):
    return _numpy_variant(o, np.float32, np.float32)


def _mutant_truncating_round(o):
    return _numpy_variant(o, float, _trunc_to_f32)


def _mutant_flush_subnormals(o):
    def dec(bits, dtype):
        v = o.decode(bits, dtype)
        tiny = 2.0 ** -14 if dtype == F16 else 2.0 ** -126
        v = np.where(np.abs(v) < tiny, 0.0, v)
        return v
    return o.gemm, dec


MUTANTS = [_mutant_dropped_term, _mutant_transposed_b, _mutant_transposed_a, _mutant_minus_c,
           _mutant_always_adds_c, _mutant_fp32_accum, _mutant_truncating_round,
           _mutant_flush_subnormals]

# The brute-force and exact-rational pins loop in Python; the slow numpy
# mutants run them on their own small shapes only, which is enough to fail.
_SLOW_OK = {pin_bruteforce_ternary}


@pytest.mark.parametrize("mutant", MUTANTS, ids=lambda m: m.__name__)
def test_planted_mistake_is_caught(oracle_lib, mutant):
    gemm, decode = mutant(oracle_lib)
    failures = []
    for pin in PINS:
        if mutant in (_mutant_fp32_accum, _mutant_truncating_round) and pin in _SLOW_OK:
            continue
        try:
            ok, why = pin(gemm, decode)
        except Exception as e:  # a mutant that crashes a pin is caught too
            ok, why = False, repr(e)
        if not ok:
            failures.append(pin.__name__)
    assert failures, f"{mutant.__name__} passed every pin"


# ---------------------------------------------------------------------------
# the checker and the alternate entry points
# ---------------------------------------------------------------------------
def test_checker_rejects_and_accepts(oracle_lib):
    o = oracle_lib
    rng = np.random.default_rng(19)
    M, N, K = 16, 16, 32
    A = f16_bits(rng.standard_normal((M, K)))
    B = f16_bits(rng.standard_normal((K, N)))
    D, S = o.gemm(A, B, None, M, N, K, False, False, F16, 0.0)
    ok, _ = o.compare(D, D, S)
    assert ok
    bad = D.copy()
    bad[3, 5] = np.float32(D[3, 5] + 4 * o.tolerance(S)[3, 5])
    assert not o.compare(bad, D, S)[0]
    nan = D.copy()
    nan[0, 0] = np.nan
    assert not o.compare(nan, D, S)[0]
    assert not o.compare(nan, D, S, exact=True)[0]
    z = np.zeros((2, 2), np.float32)
    nz = -z
    assert o.compare(nz, z, np.zeros((2, 2)), exact=True)[0]
    off = D.copy()
    off[1, 1] = np.nextafter(off[1, 1], np.float32(np.inf))
    assert not o.compare(off, D, S, exact=True)[0]


def test_entries_and_rows_match_full(oracle_lib):
    o = oracle_lib
    w = wl.BY_NAME["gemm_256_bf16_transB_beta1"].with_shape(96, 72, 104)
    A, B, C = wl.make_inputs(w)
    Ab, Bb, Cn = wl.bits(A), wl.bits(B), C.numpy()
    D, S = o.gemm(Ab, Bb, Cn, w.M, w.N, w.K, w.transA, w.transB, w.dtype, w.beta)
    rng = np.random.default_rng(0)
    r = rng.integers(0, w.M, 200)
    c = rng.integers(0, w.N, 200)
    De, Se = o.gemm_entries(r, c, Ab, Bb, Cn, w.M, w.N, w.K, w.transA, w.transB, w.dtype, w.beta)
    assert np.array_equal(De.view(np.uint32), D[r, c].view(np.uint32))
    assert np.array_equal(Se, S[r, c])
    Dr = o.gemm_rows(10, 30, Ab, Bb, Cn, w.M, w.N, w.K, w.transA, w.transB, w.dtype, w.beta)
    assert np.array_equal(Dr.view(np.uint32), D[10:30].view(np.uint32))


def test_integer_workload_bounds():
    """Integer workloads stay exactly representable in float32 at every partial sum."""
    for w in (wl.WORKLOADS[0], wl.WORKLOAD_4096_INT):
        amax = max(abs(w.a_dist[1]), abs(w.a_dist[2]))
        bmax = max(abs(w.b_dist[1]), abs(w.b_dist[2]))
        assert amax * bmax * w.K < 2 ** 24


def test_workload_inputs_are_seeded():
    w = wl.WORKLOADS[1]
    A1, B1, C1 = wl.make_inputs(w)
    A2, B2, C2 = wl.make_inputs(w)
    assert np.array_equal(wl.bits(A1), wl.bits(A2)) and np.array_equal(C1.numpy(), C2.numpy())
    assert tuple(A1.shape) == (256, 256) and tuple(B1.shape) == (256, 256)
    w5 = wl.WORKLOADS[4]
    sa, sb, sc = wl.stored_shapes(w5)
    assert sa == (144, 4104) and sb == (4104, 16392) and sc == (144, 16392)


def test_golden_fixtures_reproduced(oracle_lib):
    """The stored fixtures (written by tests/golden/make_golden.py) still match the oracle."""
    import os
    import sys
    here = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
    sys.path.insert(0, here)
    import make_golden
    for w, _ in make_golden.CASES:
        g = make_golden.read_case(os.path.join(here, f"{w.name}.txt"))
        A, B, C = wl.make_inputs(w)
        assert np.array_equal(g["A_bits"].ravel(), wl.bits(A).ravel())
        assert np.array_equal(g["B_bits"].ravel(), wl.bits(B).ravel())
        D, _ = oracle_lib.gemm(g["A_bits"].ravel(), g["B_bits"].ravel(),
                               None if C is None else g["C_f32bits"], w.M, w.N, w.K, w.transA,
                               w.transB, w.dtype, w.beta)
        assert np.array_equal(D.view(np.uint32), g["D_f32bits"].view(np.uint32))


# ---------------------------------------------------------------------------
# fp8 (the tcgen05 kind::f8f6f4 path): decoders and exactness
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("code,name", [(2, "float8_e4m3fn"), (3, "float8_e5m2")])
def test_fp8_decode_exhaustive_against_torch(oracle_lib, code, name):
    # All 256 byte patterns against torch's own fp8 -> float64 conversion.
    import torch
    td = getattr(torch, name)
    pats = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = pats.view(td).to(torch.float64).numpy()
    got = oracle_lib.decode(pats.numpy().astype(np.uint16), code)
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], got[ok])


def test_fp8_gemm_matches_exact_integer_sums(oracle_lib):
    # Small integers are exact in both fp8 formats; D must be the exact sum.
    import torch
    rng = np.random.default_rng(5)
    M, N, K = 16, 24, 48
    a = rng.integers(-3, 4, (M, K))
    b = rng.integers(-3, 4, (N, K))  # stored [N, K]: transB
    for code, td in ((2, torch.float8_e4m3fn), (3, torch.float8_e5m2)):
        A = torch.tensor(a, dtype=torch.float32).to(td)
        B = torch.tensor(b, dtype=torch.float32).to(td)
        D, S = oracle_lib.gemm(wl.bits(A), wl.bits(B), None, M, N, K, False, True, code, 0.0)
        assert np.array_equal(D, (a @ b.T).astype(np.float32))
        assert np.array_equal(S, (np.abs(a) @ np.abs(b).T).astype(np.float64))
