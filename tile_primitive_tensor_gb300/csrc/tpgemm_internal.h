// Host-side interfaces between the C-ABI entry points (tpgemm_api.cu) and the
// two kernel translation units. Not part of the public ABI.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace tpg {

constexpr int kStatusTimeout = 9;  // matches TPGEMM_ERR_TIMEOUT
constexpr int kStatusBounds = 11;  // matches TPGEMM_ERR_BOUNDS (debug builds only)

// The calling thread's reason for its last non-OK status, as returned by
// tpgemm_last_error_detail (empty after a success).
void set_error_detail(const char* text);

// Bound of every wait inside a kernel: TPGEMM_WAIT_TIMEOUT_MS (default 2 s),
// from the planner-override snapshot (tpgemm_reload_tuning).
uint64_t wait_timeout_ns();

// Device status words of the GEMM kernel and of the tensor-memory copy kernel
// (0, or kStatusTimeout after an expired bounded wait, or in a debug build
// kStatusBounds after a failed bounds check, with the check's site);
// reading clears them.
cudaError_t tc_read_and_clear_device_status(int* status, int* bounds_site);
cudaError_t cp_read_and_clear_device_status(int* status);

// ---- warp-level mma.sync kernel (small problems) ----
struct MmaSyncArgs {
    float* D;
    const void* A;
    const void* B;
    const float* C;
    int M, N, K;
    bool transA, transB, bf16, beta;
};
constexpr int kMmaTileM = 64;
constexpr int kMmaTileN = 64;
cudaError_t launch_mma_sync(const MmaSyncArgs& a, cudaStream_t stream);

// ---- tcgen05 kernel ----
// The kernel computes a product X = P . Q^T over K with P rows mapped to the
// 128 tensor-memory lanes of a tile and Q rows to its accumulator columns.
// Normal orientation: P = A (rows m), Q = B^T (rows n), X = D.
// Swapped orientation (small M): P = B^T (rows n), Q = A (rows m), X = D^T,
// which the epilogue writes back transposed so that D stays [M, N].
struct TcParams {
    int Mp, Nq, K;          // rows of P, rows of Q, reduction length
    int tiles_p, tiles_q;   // tile counts along P (bp rows) and Q (bn rows)
    // P rows of one CTA's tile: 128 (every tensor-memory lane), or 64..112 in
    // steps of 16 for single-wave plans whose tiles share the one Q tile, so
    // that more SMs stream P. Lanes bp..127 then hold unused results; the lane
    // quadrant holding row bp - 16 (when bp % 32 == 16) stores through the
    // half-width C / D maps.
    int bp;
    uint32_t p_tx;          // bytes the P boxes deliver per stage (bp rows of row_tx bytes)
    uint32_t row_tx;        // bytes a K-contiguous box row counts on its mbarrier: 128
                            // (one swizzle row), 64 for fp4 (the packed bytes read; the
                            // TMA writes them as 128 bytes of shared memory)
    int num_tiles;
    int k_blocks;           // ceil(K / 64)
    int bn;                 // accumulator columns per tile = UMMA N (16..256, %16)
    int stages;             // depth of the TMA ring
    int p_mn, q_mn;         // operand stored MN-contiguous (1) or K-contiguous (0)
    int beta;               // 0 or 1
    int group;              // tiles along P per raster group (L2 reuse)
    int snake;              // 1: odd raster groups sweep Q backwards
    uint32_t idesc;         // tcgen05 instruction descriptor
    uint32_t p_bytes;       // shared bytes of one P stage tile
    uint32_t q_bytes;       // shared bytes of one Q stage tile
    uint32_t tx_bytes;      // bytes the TMA delivers per stage
    uint64_t timeout_ns;    // bound on every mbarrier wait
    int swap;               // orientation, for the epilogue's D coordinates
    int epi_bufs;           // 32 x 32 f32 staging tiles per lane quadrant (2..8), split
                            // between the quadrant's active epilogue warps
    int bk;                 // K elements per stage (128 bytes of a row): 64, or 128 for fp8
    int fp8;                // operands are e4m3 / e5m2: kind::f8f6f4 MMAs
    int epi_groups;         // active epilogue warpgroups (1 or 2); warp 2 + 4 g + i
                            // reads lane quadrant (i + 2) % 4, chunks c % groups == g
    int epi_help;           // one-group plans: 1 = warps 6..9 join the epilogue of the CTA's
                            // last segment (after any fills they issue), taking its odd
                            // chunks and staging them through the then idle TMA ring
    int k_rotate;           // 0, or tiles per group sharing a rotated first K block
    int k_reverse;          // 1: a cluster's second, fourth, ... whole unit (the odd waves of
                            // the persistent grid) walks its K blocks backwards, so it starts
                            // on the slices the previous wave read last
    int dep_early;          // 1: only threads touching global memory wait for the previous
                            // grid, each just before its first access; 0: all wait after set-up
    int producers;          // TMA-issuing threads (1..4, at most the ring depth): warp 0,
                            // then warps 6, 7, 8; fill g is issued by producer g % producers
    int mc;                 // CTAs per cluster: 2 for a CTA pair, else 1
    int tiles_ps;           // groups of mc consecutive P tiles: ceil(tiles_p / mc)
    int num_super;          // tiles_ps * tiles_q: work items of one cluster
    int pair;               // 1: CTA-pair MMA (cta_group::2, M = 256 per pair, mc = 2);
                            // each CTA loads its 128 P rows and half of the Q tile
    int tmem_cols;          // tensor-memory columns allocated (two accumulators)
    // Work units: the first full_units work items are whole tiles; the rest
    // (the last, partial wave of the persistent grid) are each split along Q
    // into tail_split narrower units so that wave finishes sooner.
    int full_units;
    int tail_split;         // 1, 2 or 4
    int num_units;          // full_units + (num_super - full_units) * tail_split
    uint32_t idesc_tail;    // instruction descriptor of a tail unit (N = bn / tail_split)
    int q_box_rows;         // rows of one K-contiguous Q TMA box of a whole tile
    int test_stall;         // tpgemm_test_gemm_withhold_fill only: CTA 0 never fills its
                            // first stage, so the bounded waits expire and the kernel
                            // reports a timeout
    // Stream-K: work items [full_units, num_super) are not given whole to one
    // cluster; each is split into two K halves (their K blocks, sk_total of
    // them, divided evenly among the first sk_ncl = 2 x leftover clusters).
    // The first half's cluster zeroes the tile's D region at kernel start and
    // publishes per-warp epoch flags; both halves then add their accumulators
    // (the first with beta.C) into D with TMA reductions, after the flag. Two
    // f32 addends onto zero give the same bits in either order.
    int sk;                 // 0 / 1
    int sk_total;
    int sk_ncl;             // clusters sharing the stream-K K blocks (<= the grid's)
    uint32_t* sk_flags;     // [gridDim.x][kTcEpiWarps] epoch flags, one per epilogue warp
    uint32_t sk_epoch;      // value of a flag once its zeros are written in this launch
    // Block-scaled fp8 (kind::mxf8f6f4, one E8M0 scale per 32 K). The scales
    // are packed by mx_pack_scales per (tile, 128-element K stage, 128-row
    // chunk of the tile) into 512 bytes: word 4 r + c holds the 4 scales of row
    // 32 c + r of the chunk for the stage's 4 K blocks (byte b for block b).
    // That is the source layout a tcgen05.cp.32x128b.warpx4 copy spreads so
    // that row m's word sits in tensor-memory column m / 32 of lane m (every
    // lane quadrant gets the 32 rows' 16 bytes). P tiles are bp <= 128 rows
    // (one chunk, rows past bp padded), Q tiles bn rows (sf_q_chunks chunks). A tile of more than 128
    // rows stores each chunk 4 times (mx_reps): rows 32 q + r of that 128-row
    // image are the chunk's row r, so one tcgen05.cp.128x256b writes both
    // chunks to every lane quadrant (each copy holds the tensor pipe about as
    // long as the MMAs of a 64-wide stage, whatever its size, so two copies per
    // stage cost less than three). Each stage's chunks are TMA-loaded (mapSP,
    // mapSQ) beside its operand tiles; the MMA thread copies them into the
    // stage's scale slot in tensor memory (4 columns for P, then 4 per Q chunk)
    // and issues the four K = 32 MMAs with scale-factor IDs 0..3. In a CTA pair
    // each CTA holds its own P chunk and all Q chunks.
    // Slot i lies in accumulator half i / sf_spr, at column sf_col0 + (i %
    // sf_spr) sf_cols past that half's start (past its tile's columns).
    int debug_plant;        // debug builds only: 1 offsets the epilogue's first
                            // tensor-memory load past the allocation, which the bounds
                            // check must catch (and skip)
    int mx;                 // 0 / 1
    int l2_p, l2_q;         // L2 policies of the P and Q loads: 0 normal, 1 evict_first,
                            // 2 evict_last (ptx.cuh l2_policy)
    int l2_cd;              // L2 policy of the C loads and D stores (read / written once)
    int sf_q_chunks;        // 128-row chunks of a Q tile's scales (1 or 2)
    int sf_q_rows;          // 512-byte rows of a Q stage's packed scales (chunks x reps)
    uint32_t sf_bytes;      // shared bytes of a stage's scale area (0 without MX)
    int sf_col0;            // first scale column in each accumulator half
    int sf_cols;            // tensor-memory columns of one stage's slot
    int sf_spr;             // scale slots per accumulator half
};

struct TcMaps {
    CUtensorMap P, Q, C, D;
    CUtensorMap Ph;         // MN-contiguous P: box of P rows 64 .. bp - 1 of a tile
    CUtensorMap Ch, Dh;     // C / D with a half-quadrant box (16 tensor-memory lanes)
    CUtensorMap Qt;         // Q with the (narrower) box of a tail unit
    CUtensorMap SP, SQ;     // packed scales of P / Q (block-scaled plans): 128 words x
                            // one chunk per row; boxes of 1 / sf_q_rows rows
};



constexpr int kTcMaxEpiBufs = 8;
size_t tc_smem_bytes(int stages, uint32_t stage_bytes, int epi_bufs);
// Producer warp, MMA warp, then kTcEpiWarps epilogue warps: up to two per
// tensor-memory lane quadrant (TcParams::epi_groups), splitting the
// accumulator's 32-column chunks between them.
constexpr int kTcEpiWarps = 8;
constexpr int kTcThreads = 32 * (2 + kTcEpiWarps);
constexpr int kTcMaxSmem = 232448;  // 227 KB opt-in per block on sm_100-class parts
cudaError_t launch_tc(const TcMaps& maps, const TcParams& p, int grid, cudaStream_t stream);
// Whether the TMA ring holds the chunks of a last-segment helper warp (half of
// a tile's 32-column chunks per lane quadrant, one 4 KB staging tile each).
bool tc_epi_help_fits(const TcParams& p);

// Clusters of p.mc CTAs of this kernel that fit the device at once (the
// persistent grid is this many clusters at most).
cudaError_t tc_max_active_clusters(const TcParams& p, int* clusters);

// Static stream-K flags (no allocation): one epoch flag per epilogue warp of
// up to kTcMaxFlagSlots CTAs, and its device address on the current device
// (taken on first use there).
constexpr int kTcMaxFlagSlots = 256;  // CTAs a stream-K flag area (allocated or static) covers
constexpr size_t kStaticScratchBytes = size_t(kTcMaxFlagSlots) * kTcEpiWarps * sizeof(uint32_t);
constexpr int kMaxStaticScratchDevices = 64;
cudaError_t tc_static_scratch(void** ptr);

// ---- block-scaled fp8: scale packing pre-pass (mx_scales.cu) ----
// sf [rows][kb] E8M0 bytes -> out [ceil(rows / tile_rows)][ksteps][chunks][reps][128]
// words (chunks = ceil(tile_rows / 128), reps = mx_reps(tile_rows)) in the
// layout TcParams describes; rows or blocks past the ends read as 127 (scale 1).
constexpr int kMxBlock = 32;                 // K elements per scale
__host__ __device__ constexpr int mx_reps(int tile_rows) { return tile_rows > 128 ? 4 : 1; }
size_t mx_packed_bytes(int64_t rows, int64_t K, int tile_rows);
// An upper bound of mx_packed_bytes over every tile height a plan can use.
size_t mx_packed_bytes_bound(int64_t rows, int64_t K);
// Packs both operands' scales in one launch (A's rows_a rows in tiles of
// tile_rows_a, B's likewise).
cudaError_t launch_mx_pack_scales(const uint8_t* sfa, int64_t rows_a, int tile_rows_a,
                                  uint32_t* out_a, const uint8_t* sfb, int64_t rows_b,
                                  int tile_rows_b, uint32_t* out_b, int64_t K,
                                  cudaStream_t stream);


}  // namespace tpg
