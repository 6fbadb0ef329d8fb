// Scale packing for the block-scaled (MX) fp8 GEMM.
//
// The caller's scales are E8M0 bytes, one per 32 consecutive K elements of
// each row: sf[row][kb], kb = ceil(K / 32). The tcgen05 kernel consumes them
// one 128-element K stage at a time, per 128-row tile, through a
// tcgen05.cp.32x128b.warpx4 copy: that copy reads 32 rows of 16 bytes and
// writes row r to lane r of every lane quadrant, 16 bytes across four 32-bit
// columns. The block-scaled MMA reads the scale of operand row m from lane m,
// column m / 32 of its scale slot, and the byte named by the instruction's
// scale-factor ID. So the 16 bytes of copy row r must be the words of tile
// rows r, 32 + r, 64 + r, 96 + r, and byte b of each word the scale of K
// block 4 s + b of stage s.
//
// This pre-pass writes exactly that, per tile of tile_rows rows (128 for the
// kernel's P operand, the tile width for Q) split into 128-row chunks:
// out[((tile * ksteps + s) * chunks + j) * 128 + 4 r + c] = the four scales of
// row tile_rows tile + 128 j + 32 c + r for blocks 4 s .. 4 s + 3
// (little-endian, byte b = block 4 s + b). Rows past the tile or the matrix
// and blocks past K read as 127 (a scale of 1; the operands there are
// zero-filled by the TMA anyway). A stage's chunks of one tile are adjacent,
// so one TMA box loads them all.
#include <cstdint>

#include "tpgemm_internal.h"

namespace tpg {

namespace {

__global__ void __launch_bounds__(256)
    mx_pack_scales_kernel(const uint8_t* __restrict__ sf, int64_t rows, int kb, int ksteps,
                          int tile_rows, int chunks, int64_t words, uint32_t* __restrict__ out) {
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    for (int64_t w = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; w < words; w += stride) {
        const int idx = int(w & 127);
        int64_t rest = w >> 7;  // ((tile * ksteps + step) * chunks + j)
        const int j = int(rest % chunks);
        rest /= chunks;
        const int step = int(rest % ksteps);
        const int64_t tile = rest / ksteps;
        const int in_tile = 128 * j + 32 * (idx & 3) + (idx >> 2);
        const int64_t row = tile * tile_rows + in_tile;
        const bool live = in_tile < tile_rows && row < rows;
        uint32_t v = 0;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const int blk = 4 * step + b;
            const uint32_t e = (live && blk < kb) ? uint32_t(sf[row * kb + blk]) : 127u;
            v |= e << (8 * b);
        }
        out[w] = v;
    }
}

}  // namespace

size_t mx_packed_bytes(int64_t rows, int64_t K, int tile_rows) {
    const int64_t tiles = (rows + tile_rows - 1) / tile_rows;
    const int64_t chunks = (tile_rows + 127) / 128;
    const int64_t ksteps = (K + 127) / 128;
    return size_t(tiles) * size_t(chunks) * size_t(ksteps) * 512;
}

// Tile heights are 128, at most 192 when an operand has more rows than one
// tile, or all of the operand's rows (at most 192) when it fits one tile:
// at most 2 ceil(rows / 128) + 2 chunks per K stage.
size_t mx_packed_bytes_bound(int64_t rows, int64_t K) {
    const int64_t ksteps = (K + 127) / 128;
    return size_t(2 * ((rows + 127) / 128) + 2) * size_t(ksteps) * 512;
}

cudaError_t launch_mx_pack_scales(const uint8_t* sf, int64_t rows, int64_t K, int tile_rows,
                                  uint32_t* out, cudaStream_t stream) {
    if (tile_rows < 16 || tile_rows > 256) return cudaErrorInvalidValue;
    const int kb = int((K + kMxBlock - 1) / kMxBlock);
    const int ksteps = int((K + 127) / 128);
    const int chunks = (tile_rows + 127) / 128;
    const int64_t words = int64_t(mx_packed_bytes(rows, K, tile_rows) / 4);
    const int64_t want = (words + 255) / 256;
    const int blocks = int(want < 4096 ? want : 4096);
    mx_pack_scales_kernel<<<blocks, 256, 0, stream>>>(sf, rows, kb, ksteps, tile_rows, chunks,
                                                      words, out);
    return cudaGetLastError();
}

}  // namespace tpg
