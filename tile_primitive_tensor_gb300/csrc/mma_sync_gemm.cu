// Warp-level mma.sync GEMM:  D = A.B + beta.C, f16/bf16 in, f32 accumulate and out.
//
// The lowering of the TVM TIRx synchronous gemm page ("TVM TIRx 同步 GEMM 深度
// 解析"), restated as a CUDA kernel for small problems and ragged shapes:
//   - section 二 / 四.1: the m16n8k16 instruction tiles the body; when the last
//     K step is 8 wide (K % 16 == 8) that step uses m16n8k8, the second entry
//     of the page's instruction table (k_pack = 2: two 16-bit elements per b32);
//   - section 三 / 四.2: fragment geometry. Lane l holds accumulator (rM, rN)
//     at row l/4 + 8 rM, column 2 (l%4) + rN (slot 2 rM + rN); A slot
//     4 kHi + 2 rM + kp at A[l/4 + 8 rM][2 (l%4) + kp + 8 kHi]; B slot
//     2 kHi + kp at B[2 (l%4) + kp + 8 kHi][l/4]. ldmatrix (.trans for
//     MN-contiguous operands) produces exactly these slots from shared memory;
//   - section 四.3: the accumulator starts from C when beta = 1 and from zero
//     when beta = 0, then accumulates in place over K with d = a.b + d.
// A CTA of 4 warps owns a 64 x 64 output tile (2 x 2 warps of 32 x 32), stages
// 64 x 32 slices of A and B into padded shared memory with 16-byte cp.async
// (double-buffered, zero-filled past the edges) and needs no spin-waits.
#include "ptx.cuh"
#include "tpgemm_internal.h"

namespace tpg {
namespace {

constexpr int kTM = kMmaTileM;  // 64
constexpr int kTN = kMmaTileN;  // 64
constexpr int kTK = 32;
constexpr int kPad = 8;         // 16-byte row padding: conflict-free ldmatrix rows

// Shared tile geometry for one operand: K-contiguous rows [64][32 + 8] or
// MN-contiguous rows [32][64 + 8] (16-bit elements).
template <bool MN>
struct Tile {
    static constexpr int rows = MN ? kTK : kTM;
    static constexpr int ld = (MN ? kTM : kTK) + kPad;
    static constexpr int elems = rows * ld;
};

// Stage one 64(mn) x 32(k) slice of an operand stored K-contiguous ([rows][K])
// or MN-contiguous ([K][rows]) into shared memory, 16 bytes per cp.async,
// zero-filling chunks beyond `rows_total` or K. 256 chunks over 128 threads.
template <bool MN>
__device__ __forceinline__ void stage_operand(uint16_t* sm, const uint16_t* g, int mn0, int k0,
                                              int rows_total, int K, int tid) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int q = tid + i * 128;
        int r, c;          // shared row, element column
        long long goff;
        bool valid;
        if (!MN) {         // [mn][k]: 64 rows x 4 chunks
            r = q >> 2;
            c = (q & 3) * 8;
            valid = (mn0 + r < rows_total) && (k0 + c < K);
            goff = (long long)(mn0 + r) * K + (k0 + c);
        } else {           // [k][mn]: 32 rows x 8 chunks
            r = q >> 3;
            c = (q & 7) * 8;
            valid = (k0 + r < K) && (mn0 + c < rows_total);
            goff = (long long)(k0 + r) * rows_total + (mn0 + c);
        }
        const uint32_t sa = smem_u32(sm + r * Tile<MN>::ld + c);
        cp_async_16(sa, valid ? static_cast<const void*>(g + goff) : static_cast<const void*>(g),
                    valid ? 16u : 0u);
    }
}

template <bool A_MN, bool B_MN, bool BF16>
__global__ void __launch_bounds__(128) mma_sync_gemm_kernel(float* __restrict__ D,
                                                            const uint16_t* __restrict__ A,
                                                            const uint16_t* __restrict__ B,
                                                            const float* C, int M, int N, int K,
                                                            int beta) {
    __shared__ __align__(128) uint16_t sA[2][Tile<A_MN>::elems];
    __shared__ __align__(128) uint16_t sB[2][Tile<B_MN>::elems];

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int wm = warp >> 1;    // warp row (0..1): 32 rows each
    const int wn = warp & 1;     // warp column (0..1): 32 columns each
    const int m0 = blockIdx.y * kTM;
    const int n0 = blockIdx.x * kTN;
    const int g = lane >> 2;     // fragment row group
    const int t4 = lane & 3;     // fragment column pair

    // Accumulators: [m16 tile][n8 tile][slot 2 rM + rN], initialised per beta.
    float acc[2][4][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
            const int row = m0 + wm * 32 + mt * 16 + g;
            const int col = n0 + wn * 32 + nt * 8 + 2 * t4;
#pragma unroll
            for (int rM = 0; rM < 2; ++rM) {
                float2 c = make_float2(0.f, 0.f);
                if (beta && row + 8 * rM < M && col < N)
                    c = *reinterpret_cast<const float2*>(C + (size_t)(row + 8 * rM) * N + col);
                acc[mt][nt][2 * rM] = c.x;
                acc[mt][nt][2 * rM + 1] = c.y;
            }
        }

    const int kTiles = (K + kTK - 1) / kTK;
    stage_operand<A_MN>(sA[0], A, m0, 0, M, K, tid);
    stage_operand<B_MN>(sB[0], B, n0, 0, N, K, tid);
    cp_async_commit();

    for (int kt = 0; kt < kTiles; ++kt) {
        const int cur = kt & 1;
        if (kt + 1 < kTiles) {
            stage_operand<A_MN>(sA[cur ^ 1], A, m0, (kt + 1) * kTK, M, K, tid);
            stage_operand<B_MN>(sB[cur ^ 1], B, n0, (kt + 1) * kTK, N, K, tid);
        }
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();

        const uint16_t* a_s = sA[cur];
        const uint16_t* b_s = sB[cur];
        const int k_base = kt * kTK;
#pragma unroll
        for (int ks = 0; ks < kTK; ks += 16) {
            const int k_left = K - (k_base + ks);
            if (k_left <= 0) break;
            const int q = lane >> 3;   // which 8x8 matrix this lane addresses
            const int r8 = lane & 7;   // row of that matrix
            uint32_t af[2][4];
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
                const int mb = wm * 32 + mt * 16;
                int sr, sc;
                if (!A_MN) {           // rows m, matrices (m0-7,k0-7)(m8-15,k0-7)(m0-7,k8-15)(m8-15,k8-15)
                    sr = mb + r8 + 8 * (q & 1);
                    sc = ks + 8 * (q >> 1);
                } else {               // rows k, transposed on load
                    sr = ks + r8 + 8 * (q >> 1);
                    sc = mb + 8 * (q & 1);
                }
                ldmatrix_x4<A_MN>(af[mt], smem_u32(a_s + sr * Tile<A_MN>::ld + sc));
            }
            uint32_t bf[2][4];         // [n16 pair]: b0,b1 of n8 tile 2p and b0,b1 of tile 2p+1
#pragma unroll
            for (int np = 0; np < 2; ++np) {
                const int nb = wn * 32 + np * 16;
                int sr, sc;
                if (!B_MN) {           // rows n: (n0-7,k0-7)(n0-7,k8-15)(n8-15,k0-7)(n8-15,k8-15)
                    sr = nb + r8 + 8 * (q >> 1);
                    sc = ks + 8 * (q & 1);
                } else {               // rows k, transposed on load
                    sr = ks + r8 + 8 * (q & 1);
                    sc = nb + 8 * (q >> 1);
                }
                ldmatrix_x4<B_MN>(bf[np], smem_u32(b_s + sr * Tile<B_MN>::ld + sc));
            }
            if (k_left >= 16) {
#pragma unroll
                for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                    for (int nt = 0; nt < 4; ++nt)
                        mma_m16n8k16<BF16>(acc[mt][nt], af[mt], bf[nt >> 1][2 * (nt & 1)],
                                           bf[nt >> 1][2 * (nt & 1) + 1]);
            } else {  // the 8-wide K tail: m16n8k8 on the low halves
#pragma unroll
                for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                    for (int nt = 0; nt < 4; ++nt)
                        mma_m16n8k8<BF16>(acc[mt][nt], af[mt][0], af[mt][1],
                                          bf[nt >> 1][2 * (nt & 1)]);
            }
        }
        __syncthreads();
    }

#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
            const int row = m0 + wm * 32 + mt * 16 + g;
            const int col = n0 + wn * 32 + nt * 8 + 2 * t4;
#pragma unroll
            for (int rM = 0; rM < 2; ++rM)
                if (row + 8 * rM < M && col < N)
                    *reinterpret_cast<float2*>(D + (size_t)(row + 8 * rM) * N + col) =
                        make_float2(acc[mt][nt][2 * rM], acc[mt][nt][2 * rM + 1]);
        }
}

template <bool A_MN, bool B_MN>
cudaError_t launch_typed(const MmaSyncArgs& a, cudaStream_t stream) {
    dim3 grid((a.N + kTN - 1) / kTN, (a.M + kTM - 1) / kTM);
    const auto* A = static_cast<const uint16_t*>(a.A);
    const auto* B = static_cast<const uint16_t*>(a.B);
    if (a.bf16)
        mma_sync_gemm_kernel<A_MN, B_MN, true>
            <<<grid, 128, 0, stream>>>(a.D, A, B, a.C, a.M, a.N, a.K, a.beta ? 1 : 0);
    else
        mma_sync_gemm_kernel<A_MN, B_MN, false>
            <<<grid, 128, 0, stream>>>(a.D, A, B, a.C, a.M, a.N, a.K, a.beta ? 1 : 0);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_mma_sync(const MmaSyncArgs& a, cudaStream_t stream) {
    // A stored [K, M] (transA) is MN-contiguous; B stored [K, N] (!transB) is.
    const bool a_mn = a.transA;
    const bool b_mn = !a.transB;
    if (!a_mn && !b_mn) return launch_typed<false, false>(a, stream);
    if (!a_mn && b_mn) return launch_typed<false, true>(a, stream);
    if (a_mn && !b_mn) return launch_typed<true, false>(a, stream);
    return launch_typed<true, true>(a, stream);
}

}  // namespace tpg
