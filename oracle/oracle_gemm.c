/*
 * CPU oracle for the tile-primitive matrix multiply  D = alpha*A*B + beta*C.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the plain, slow, obviously correct
 * definition that the CUDA library is checked against. Only the test suite,
 * the smoke check and the benchmark's CPU-baseline leg load it; the library
 * never does, and it shares no code, header or constant with the library.
 *
 * What it computes (the TVM TIRx "gemm" tile primitive, as described on the
 * page "TVM TIRx 同步 GEMM 深度解析：warp 级 mma.sync 的寄存器碎片排布与完整
 * 下放链路", sections 语义定义 and 二 What it accepts):
 *   - D = alpha*A*B + beta*C with alpha fixed at 1 and beta in {0, 1};
 *   - A and B are both float16 or both bfloat16, C and D are float32; the
 *     same with both fp8 e4m3 or both fp8 e5m2 (the fp8 gemm_async the pages
 *     mention beside the f16 one), patterns passed widened to 16 bits;
 *   - transpose_A / transpose_B only set the logical orientation: the operands
 *     are normalised to A[M,K], B[K,N], C and D [M,N] (section 维度一致性);
 *   - the accumulator is initialised from C when beta = 1 and from zero when
 *     beta = 0, then accumulated over K (section 四 step 3).
 *
 * Precision: every 16-bit (or 8-bit) input is decoded exactly to double, each
 * product is exact in double (at most 22 significant bits), the sum runs over k in
 * increasing order in double, C is added when beta = 1, and the result is
 * rounded once to float32 (round to nearest even, the C cast). The oracle
 * accepts any positive shape; the divisibility rules belong to the library.
 *
 * Storage: dense row-major. A is [M,K], or [K,M] when transA. B is [K,N], or
 * [N,K] when transB. C and D are [M,N].
 *
 * Alongside D it can return S[i,j] = sum_k |a(i,k) * b(k,j)| in double, the
 * scale of the elementwise acceptance bound |D - D_ref| <= 2^-10 * S + 1e-6.
 *
 * fp4 e2m1 (dtype 4) follows the same rules as fp8: patterns widened to 16
 * bits, one element per entry (the callers unpack the two 4-bit codes of each
 * stored byte).
 *
 * Block-scaled fp8 (oracle_gemm_mx): the same page lists block scaling (SFA,
 * SFB) among the operand forms of gemm_async (section 七) without defining
 * it. The reading taken is the OCP Microscaling (MX) one: every run of
 * `block` consecutive K elements of a row of A (of a column of B) shares one
 * scale, an 8-bit power of two (E8M0: 2^(e - 127), e = 255 is NaN), and the
 * element's value is its fp8 value times that scale:
 *   D[i,j] = sum_k (a(i,k) * sa(i, k / block)) * (b(k,j) * sb(j, k / block))
 *            (+ C[i,j] when beta = 1),
 * with SFA stored [M][KB] and SFB stored [N][KB], KB = ceil(K / block),
 * whatever the orientation of A and B. Every scaled element and every product
 * is exact in double; the sum runs in increasing k and is rounded once.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_F16 0
#define ORACLE_BF16 1
#define ORACLE_E4M3 2
#define ORACLE_E5M2 3
#define ORACLE_E2M1 4

/* IEEE-754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
 * Exponent field 0 encodes zero and subnormals (fraction * 2^-24); 31 encodes
 * infinity (fraction 0) or NaN. */
double oracle_decode_f16(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)m, -24);
    } else if (e == 31) {
        v = (m == 0) ? INFINITY : NAN;
    } else {
        v = ldexp((double)(1024 + m), e - 25);
    }
    return sign ? -v : v;
}

/* bfloat16: the upper half of an IEEE-754 binary32. 1 sign bit, 8 exponent
 * bits (bias 127), 7 fraction bits. Exponent 0 encodes zero and subnormals
 * (fraction * 2^-133); 255 encodes infinity or NaN. */
double oracle_decode_bf16(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 7) & 0xff;
    int m = h & 0x7f;
    double v;
    if (e == 0) {
        v = ldexp((double)m, -133);
    } else if (e == 255) {
        v = (m == 0) ? INFINITY : NAN;
    } else {
        v = ldexp((double)(128 + m), e - 134);
    }
    return sign ? -v : v;
}

/* fp8 e4m3 (the "fn" variant): 1 sign bit, 4 exponent bits (bias 7), 3
 * fraction bits, in the low byte. Exponent 0 encodes zero and subnormals
 * (fraction * 2^-9); the all-ones pattern S.1111.111 is NaN and there is no
 * infinity, so exponent 15 with fraction 0..6 is an ordinary number. */
double oracle_decode_e4m3(uint16_t h) {
    int sign = (h >> 7) & 1;
    int e = (h >> 3) & 0xf;
    int m = h & 0x7;
    double v;
    if (e == 0) {
        v = ldexp((double)m, -9);
    } else if (e == 15 && m == 7) {
        v = NAN;
    } else {
        v = ldexp((double)(8 + m), e - 10);
    }
    return sign ? -v : v;
}

/* fp8 e5m2: 1 sign bit, 5 exponent bits (bias 15), 2 fraction bits, in the
 * low byte. Exponent 0 encodes zero and subnormals (fraction * 2^-16); 31
 * encodes infinity (fraction 0) or NaN. */
double oracle_decode_e5m2(uint16_t h) {
    int sign = (h >> 7) & 1;
    int e = (h >> 2) & 0x1f;
    int m = h & 0x3;
    double v;
    if (e == 0) {
        v = ldexp((double)m, -16);
    } else if (e == 31) {
        v = (m == 0) ? INFINITY : NAN;
    } else {
        v = ldexp((double)(4 + m), e - 17);
    }
    return sign ? -v : v;
}

/* fp4 e2m1 (OCP Microscaling): 1 sign bit, 2 exponent bits (bias 1), 1
 * fraction bit, in the low 4 bits. Exponent 0 encodes zero and the subnormal
 * 0.5; there is no infinity and no NaN: the magnitudes are 0, 0.5, 1, 1.5, 2,
 * 3, 4 and 6. */
double oracle_decode_e2m1(uint16_t h) {
    int sign = (h >> 3) & 1;
    int e = (h >> 1) & 0x3;
    int m = h & 0x1;
    double v = (e == 0) ? ldexp((double)m, -1) : ldexp((double)(2 + m), e - 2);
    return sign ? -v : v;
}

static double decode(uint16_t h, int dtype) {
    switch (dtype) {
        case ORACLE_E2M1: return oracle_decode_e2m1(h);
        case ORACLE_BF16: return oracle_decode_bf16(h);
        case ORACLE_E4M3: return oracle_decode_e4m3(h);
        case ORACLE_E5M2: return oracle_decode_e5m2(h);
        default: return oracle_decode_f16(h);
    }
}

void oracle_decode(const uint16_t* src, double* dst, int64_t n, int dtype) {
    for (int64_t i = 0; i < n; ++i) dst[i] = decode(src[i], dtype);
}

/* Logical element a(i,k) of the M x K matrix A, whatever its storage. */
static uint16_t a_bits(const uint16_t* A, int64_t i, int64_t k, int64_t M, int64_t K, int transA) {
    return transA ? A[k * M + i] : A[i * K + k];
}

/* Logical element b(k,j) of the K x N matrix B, whatever its storage. */
static uint16_t b_bits(const uint16_t* B, int64_t k, int64_t j, int64_t N, int64_t K, int transB) {
    return transB ? B[j * K + k] : B[k * N + j];
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Full D. Returns 0 on success, -1 if the decode buffers cannot be allocated,
 * -2 on a bad argument. sumabs may be NULL. C is read only when beta != 0. */
int oracle_gemm(float* D, double* sumabs, const uint16_t* A, const uint16_t* B, const float* C,
                int64_t M, int64_t N, int64_t K, int transA, int transB, int dtype, int beta) {
    if (M <= 0 || N <= 0 || K <= 0 || !D || !A || !B || (beta && !C)) return -2;
    if (dtype < ORACLE_F16 || dtype > ORACLE_E2M1) return -2;
    /* Decode once into the normalised orientation: a[i*K+k] = a(i,k) and
     * bt[j*K+k] = b(k,j), so the sum over k walks both rows contiguously. */
    double* a = (double*)malloc(sizeof(double) * (size_t)(M * K));
    double* bt = (double*)malloc(sizeof(double) * (size_t)(N * K));
    if (!a || !bt) {
        free(a);
        free(bt);
        return -1;
    }
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < M; ++i)
        for (int64_t k = 0; k < K; ++k) a[i * K + k] = decode(a_bits(A, i, k, M, K, transA), dtype);
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < N; ++j)
        for (int64_t k = 0; k < K; ++k) bt[j * K + k] = decode(b_bits(B, k, j, N, K, transB), dtype);

#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < M; ++i) {
        const double* ai = a + i * K;
        for (int64_t j = 0; j < N; ++j) {
            const double* bj = bt + j * K;
            double s = 0.0, sa = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double p = ai[k] * bj[k];
                s += p;
                sa += fabs(p);
            }
            if (beta) s += (double)C[i * N + j];
            D[i * N + j] = (float)s;
            if (sumabs) sumabs[i * N + j] = sa;
        }
    }
    free(a);
    free(bt);
    return 0;
}

/* Selected entries only: D_out[t] = D[rows[t], cols[t]] (and its sum of
 * |products|), computed one by one straight from the 16-bit storage. This is
 * how outputs of problems too large for the full triple loop are checked. */
int oracle_gemm_entries(float* D_out, double* sumabs_out, const int64_t* rows, const int64_t* cols,
                        int64_t count, const uint16_t* A, const uint16_t* B, const float* C,
                        int64_t M, int64_t N, int64_t K, int transA, int transB, int dtype,
                        int beta) {
    if (M <= 0 || N <= 0 || K <= 0 || !D_out || !A || !B || (beta && !C) || count < 0) return -2;
    if (dtype < ORACLE_F16 || dtype > ORACLE_E2M1) return -2;
    for (int64_t t = 0; t < count; ++t)
        if (rows[t] < 0 || rows[t] >= M || cols[t] < 0 || cols[t] >= N) return -2;
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t t = 0; t < count; ++t) {
        int64_t i = rows[t], j = cols[t];
        double s = 0.0, sa = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double p = decode(a_bits(A, i, k, M, K, transA), dtype) *
                       decode(b_bits(B, k, j, N, K, transB), dtype);
            s += p;
            sa += fabs(p);
        }
        if (beta) s += (double)C[i * N + j];
        D_out[t] = (float)s;
        if (sumabs_out) sumabs_out[t] = sa;
    }
    return 0;
}

/* Rows [row_begin, row_end) of D only, written to D_rows[(i-row_begin)*N + j].
 * Same arithmetic as oracle_gemm; used to time the oracle on a bounded sample
 * of a large problem. */
int oracle_gemm_rows(float* D_rows, const uint16_t* A, const uint16_t* B, const float* C,
                     int64_t M, int64_t N, int64_t K, int64_t row_begin, int64_t row_end,
                     int transA, int transB, int dtype, int beta) {
    if (M <= 0 || N <= 0 || K <= 0 || !D_rows || !A || !B || (beta && !C)) return -2;
    if (row_begin < 0 || row_end > M || row_begin >= row_end) return -2;
    if (dtype < ORACLE_F16 || dtype > ORACLE_E2M1) return -2;
    int64_t R = row_end - row_begin;
    double* a = (double*)malloc(sizeof(double) * (size_t)(R * K));
    double* bt = (double*)malloc(sizeof(double) * (size_t)(N * K));
    if (!a || !bt) {
        free(a);
        free(bt);
        return -1;
    }
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < R; ++r)
        for (int64_t k = 0; k < K; ++k)
            a[r * K + k] = decode(a_bits(A, row_begin + r, k, M, K, transA), dtype);
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < N; ++j)
        for (int64_t k = 0; k < K; ++k) bt[j * K + k] = decode(b_bits(B, k, j, N, K, transB), dtype);
#pragma omp parallel for schedule(static) collapse(2)
    for (int64_t r = 0; r < R; ++r) {
        for (int64_t j = 0; j < N; ++j) {
            const double* ai = a + r * K;
            const double* bj = bt + j * K;
            double s = 0.0;
            for (int64_t k = 0; k < K; ++k) s += ai[k] * bj[k];
            if (beta) s += (double)C[(row_begin + r) * N + j];
            D_rows[r * N + j] = (float)s;
        }
    }
    free(a);
    free(bt);
    return 0;
}

/* E8M0 scale: an unsigned 8-bit biased exponent, 2^(e - 127); e = 255 is NaN. */
double oracle_decode_e8m0(uint8_t e) {
    return e == 255 ? NAN : ldexp(1.0, (int)e - 127);
}

/* Block-scaled D (see the header comment): A and B fp8 (dtype E4M3 or E5M2,
 * patterns widened to 16 bits as for oracle_gemm), SFA [M][KB] and SFB [N][KB]
 * E8M0 bytes. Returns 0 on success, -1 if the decode buffers cannot be
 * allocated, -2 on a bad argument. sumabs may be NULL. */
int oracle_gemm_mx(float* D, double* sumabs, const uint16_t* A, const uint16_t* B,
                   const float* C, const uint8_t* SFA, const uint8_t* SFB, int64_t M, int64_t N,
                   int64_t K, int transA, int transB, int dtype, int beta, int64_t block) {
    if (M <= 0 || N <= 0 || K <= 0 || block <= 0 || !D || !A || !B || !SFA || !SFB ||
        (beta && !C))
        return -2;
    if (dtype != ORACLE_E4M3 && dtype != ORACLE_E5M2 && dtype != ORACLE_E2M1) return -2;
    const int64_t KB = (K + block - 1) / block;
    double* a = (double*)malloc(sizeof(double) * (size_t)(M * K));
    double* bt = (double*)malloc(sizeof(double) * (size_t)(N * K));
    if (!a || !bt) {
        free(a);
        free(bt);
        return -1;
    }
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < M; ++i)
        for (int64_t k = 0; k < K; ++k)
            a[i * K + k] = decode(a_bits(A, i, k, M, K, transA), dtype) *
                           oracle_decode_e8m0(SFA[i * KB + k / block]);
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < N; ++j)
        for (int64_t k = 0; k < K; ++k)
            bt[j * K + k] = decode(b_bits(B, k, j, N, K, transB), dtype) *
                            oracle_decode_e8m0(SFB[j * KB + k / block]);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < M; ++i) {
        const double* ai = a + i * K;
        for (int64_t j = 0; j < N; ++j) {
            const double* bj = bt + j * K;
            double s = 0.0, sa = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double p = ai[k] * bj[k];
                s += p;
                sa += fabs(p);
            }
            if (beta) s += (double)C[i * N + j];
            D[i * N + j] = (float)s;
            if (sumabs) sumabs[i * N + j] = sa;
        }
    }
    free(a);
    free(bt);
    return 0;
}
