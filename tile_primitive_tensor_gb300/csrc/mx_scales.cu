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
// out[(((tile * ksteps + s) * chunks + j) * reps + i) * 128 + 4 r + c] = the
// four scales of row tile_rows tile + 128 j + 32 c + r for blocks 4 s .. 4 s +
// 3 (little-endian, byte b = block 4 s + b), for every replica i < reps. A
// tile of more than 128 rows has reps = 4: its stage's 4 KB are then the
// 128-row, 32-byte-wide source of one tcgen05.cp.128x256b (row 32 i + r of
// chunk j's image is 16-byte unit j of source row 32 i + r), which puts the
// same words in every lane quadrant as a warpx4 copy of each chunk. Rows
// past the tile or the matrix and blocks past K read as 127 (a scale of 1;
// the operands there are zero-filled by the TMA anyway). A stage's chunks of
// one tile are adjacent, so one TMA box loads them all.
//
// One launch packs both operands. A block takes one 128-row chunk of one
// tile and kPackSteps consecutive K stages: it reads the chunk's rows along
// their scale bytes (two 16-byte loads per thread when the rows are 16-byte
// aligned, else consecutive threads on consecutive bytes of a row, so the
// reads coalesce), transposes them in shared memory, and writes each
// stage's 128 words as one contiguous run.
#include <algorithm>
#include <cstdint>

#include "tpgemm_internal.h"

namespace tpg {

namespace {

constexpr int kPackSteps = 16;  // K stages per block: 64 scale bytes of each row
static_assert(kPackSteps == 16, "a block's 256 threads read 128 rows x 2 x 32 bytes");

struct PackJob {
    const uint8_t* sf;
    uint32_t* out;
    int64_t rows;
    int kb, ksteps, tile_rows, chunks, reps, groups;
    int vec;         // rows start 16-byte aligned: vector loads
    int64_t blocks;  // tiles * chunks * groups
};

__device__ __forceinline__ void pack_block(const PackJob& jb, int64_t b, uint32_t (*w)[kPackSteps + 1]) {
    const int g = int(b % jb.groups);
    const int64_t tj = b / jb.groups;  // tile * chunks + j
    const int j = int(tj % jb.chunks);
    const int64_t tile = tj / jb.chunks;
    const int s0 = g * kPackSteps;
    const int nsteps = min(kPackSteps, jb.ksteps - s0);
    if (jb.vec && 4 * s0 + 4 * kPackSteps <= jb.kb) {
        // 16-byte aligned rows, the block's 64 bytes of each inside it: thread
        // t reads 32 bytes (stages s0 + 8 h .. + 7) of chunk row r = t / 2,
        // h = t % 2, with two vector loads in flight at once.
        const int r = int(threadIdx.x) >> 1;
        const int h = int(threadIdx.x) & 1;
        const int in_tile = 128 * j + r;
        const int64_t row = tile * jb.tile_rows + in_tile;
        uint32_t v[8];
        if (in_tile < jb.tile_rows && row < jb.rows) {
            const uint4* src =
                reinterpret_cast<const uint4*>(jb.sf + row * jb.kb + 4 * s0 + 32 * h);
            const uint4 x = src[0], y = src[1];
            v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
            v[4] = y.x; v[5] = y.y; v[6] = y.z; v[7] = y.w;
        } else {
#pragma unroll
            for (int q = 0; q < 8; ++q) v[q] = 0x7f7f7f7fu;
        }
        // w[4 r' + c][s] holds chunk row 32 c + r', stage s0 + s: the output
        // order, so the write-out below reads consecutive rows of w.
        const int idx = 4 * (r & 31) + (r >> 5);
#pragma unroll
        for (int q = 0; q < 8; ++q) w[idx][8 * h + q] = v[q];
    } else {
        // Any alignment: consecutive threads read consecutive bytes of a row
        // (a warp covers 32 bytes of one row), all 32 loads issued before
        // any store.
        constexpr int kRowBytes = 4 * kPackSteps;
        uint8_t v[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) {
            const int e = int(threadIdx.x) + 256 * k;
            const int in_tile = 128 * j + e / kRowBytes;
            const int64_t row = tile * jb.tile_rows + in_tile;
            const int blk = 4 * s0 + e % kRowBytes;
            v[k] = (in_tile < jb.tile_rows && row < jb.rows && blk < jb.kb)
                       ? jb.sf[row * jb.kb + blk]
                       : uint8_t(127);
        }
        uint8_t* wb = reinterpret_cast<uint8_t*>(w);
#pragma unroll
        for (int k = 0; k < 32; ++k) {
            const int e = int(threadIdx.x) + 256 * k;
            const int r = e / kRowBytes;
            const int byte = e % kRowBytes;
            const int idx = 4 * (r & 31) + (r >> 5);
            wb[(idx * (kPackSteps + 1) + (byte >> 2)) * 4 + (byte & 3)] = v[k];
        }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < nsteps * 128; e += blockDim.x) {
        const int st = e >> 7;
        const int i = e & 127;
        const uint32_t x = w[i][st];
        uint32_t* o = jb.out + (((tile * jb.ksteps + s0 + st) * jb.chunks + j) * jb.reps) * 128 + i;
        for (int k = 0; k < jb.reps; ++k) o[k * 128] = x;
    }
}

__global__ void __launch_bounds__(256) mx_pack_scales_kernel(PackJob a, PackJob b) {
    __shared__ uint32_t w[128][kPackSteps + 1];
    const int64_t blk = blockIdx.x;
    if (blk < a.blocks)
        pack_block(a, blk, w);
    else
        pack_block(b, blk - a.blocks, w);
}

bool make_job(const uint8_t* sf, int64_t rows, int64_t K, int tile_rows, uint32_t* out,
              PackJob& jb) {
    if (tile_rows < 16 || tile_rows > 256) return false;
    jb.sf = sf;
    jb.out = out;
    jb.rows = rows;
    jb.kb = int((K + kMxBlock - 1) / kMxBlock);
    jb.ksteps = int((K + 127) / 128);
    jb.tile_rows = tile_rows;
    jb.chunks = (tile_rows + 127) / 128;
    jb.reps = mx_reps(tile_rows);
    jb.vec = (reinterpret_cast<uintptr_t>(sf) % 16 == 0 && jb.kb % 16 == 0) ? 1 : 0;
    jb.groups = (jb.ksteps + kPackSteps - 1) / kPackSteps;
    const int64_t tiles = (rows + tile_rows - 1) / tile_rows;
    jb.blocks = tiles * jb.chunks * jb.groups;
    return true;
}

}  // namespace

size_t mx_packed_bytes(int64_t rows, int64_t K, int tile_rows) {
    const int64_t tiles = (rows + tile_rows - 1) / tile_rows;
    const int64_t chunks = (tile_rows + 127) / 128;
    const int64_t ksteps = (K + 127) / 128;
    return size_t(tiles) * size_t(chunks) * size_t(mx_reps(tile_rows)) * size_t(ksteps) * 512;
}

// Tile heights a plan uses: 128 (P), a multiple of 32 up to 192 (Q over
// several tiles), or all rows rounded up to 16 when they fit one Q tile.
size_t mx_packed_bytes_bound(int64_t rows, int64_t K) {
    size_t b = 0;
    for (int t = 32; t <= 192; t += 32) b = std::max(b, mx_packed_bytes(rows, K, t));
    if (rows <= 192) b = std::max(b, mx_packed_bytes(rows, K, int((rows + 15) / 16 * 16)));
    return b;
}

cudaError_t launch_mx_pack_scales(const uint8_t* sfa, int64_t rows_a, int tile_rows_a,
                                  uint32_t* out_a, const uint8_t* sfb, int64_t rows_b,
                                  int tile_rows_b, uint32_t* out_b, int64_t K,
                                  cudaStream_t stream) {
    PackJob a, b;
    if (!make_job(sfa, rows_a, K, tile_rows_a, out_a, a) ||
        !make_job(sfb, rows_b, K, tile_rows_b, out_b, b))
        return cudaErrorInvalidValue;
    const int64_t blocks = a.blocks + b.blocks;
    if (blocks < 1 || blocks > 0x7fffffff) return cudaErrorInvalidValue;
    mx_pack_scales_kernel<<<unsigned(blocks), 256, 0, stream>>>(a, b);
    return cudaGetLastError();
}

}  // namespace tpg
