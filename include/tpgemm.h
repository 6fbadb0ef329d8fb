/*
 * tpgemm — the tile-primitive matrix multiply  D = A·B + beta·C  on one GB300
 * (sm_103a), as a C-ABI shared library (libtpgemm.so).
 *
 * The operation is the TVM TIRx "gemm" tile primitive as described on the page
 * "TVM TIRx 同步 GEMM 深度解析：warp 级 mma.sync 的寄存器碎片排布与完整下放链路":
 *   - section 语义定义: D = alpha·A·B + beta·C;
 *   - section 二 (What it accepts): A and B are both float16 or both bfloat16,
 *     C and D are float32, alpha = 1.0, beta ∈ {0.0, 1.0} (0 → D = A·B,
 *     1 → D = A·B + C), M % 16 = 0, N % 8 = 0, K % 8 = 0;
 *   - section 二 维度一致性: transpose_A / transpose_B only describe the logical
 *     orientation; operands are normalised to A[M,K], B[K,N], C and D [M,N];
 *   - section 三: the C position may be D itself (in-place accumulation).
 * The library computes it with hand-written sm_103a kernels: TMA loads into
 * 128-byte-swizzled shared memory, an mbarrier ring, single-thread-issued
 * tcgen05.mma accumulating in tensor memory, and a warpgroup tcgen05.ld
 * epilogue; small problems run a warp-level mma.sync.m16n8k16 kernel.
 *
 * Storage: dense row-major, no leading-dimension arguments.
 *   A: [M,K] elements, or [K,M] when transA != 0 (the logical A is its transpose).
 *   B: [K,N] elements, or [N,K] when transB != 0.
 *   C: [M,N] float32 (read only when beta == 1; may be NULL when beta == 0).
 *   D: [M,N] float32 (written).
 * For tpgemm_gemm all four are device pointers owned by the caller (for
 * tpgemm_gemm_host they are host pointers). The library keeps no pointer to
 * them after a call is enqueued. No call allocates device memory for itself,
 * with one exception: a plan whose last wave is split by K across clusters
 * (stream-K, on by default where it applies; environment TPGEMM_TC_SK=0
 * turns it off) needs an 8 KB array of flags, taken once per (device, stream)
 * with cudaMalloc on the first such call and kept until exit;
 * tpgemm_gemm_noalloc uses a static array instead. Calls in place (D == C)
 * and calls on a stream being captured into a CUDA graph never use that mode
 * (a graph replay would reuse the captured flag epoch): they split the last
 * wave along N, which needs nothing.
 *
 * Errors: every function returns a status. Argument errors are detected on the
 * host before anything is enqueued, and a readable reason is available from
 * tpgemm_last_error_detail() on the calling thread.
 */
#ifndef TPGEMM_H
#define TPGEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element type of A and B (both the same). The fp8 and fp4 types run on the
 * tcgen05 kernel only (tcgen05.mma kind::f8f6f4, the fp8 / fp4 gemm_async the
 * pages mention beside the f16 one) with A stored [M,K] (transA = 0) and B
 * stored [N,K] (transB = 1), both K-contiguous, and K % 16 == 0 (fp4: K % 128
 * == 0); other orientations return TPGEMM_ERR_PATH. tpgemm_gemm applies no
 * per-block scale: D = A.B + beta.C exactly as for f16, with the narrow values
 * as they are (tpgemm_gemm_mx is the block-scaled form). */
typedef enum {
    TPGEMM_F16 = 0,  /* IEEE binary16 */
    TPGEMM_BF16 = 1, /* bfloat16 */
    TPGEMM_E4M3 = 2, /* fp8 e4m3 (1 sign, 4 exponent bits, bias 7, 3 mantissa bits; no inf) */
    TPGEMM_E5M2 = 3, /* fp8 e5m2 (1 sign, 5 exponent bits, bias 15, 2 mantissa bits) */
    TPGEMM_E2M1 = 4  /* fp4 e2m1 (1 sign, 2 exponent bits, bias 1, 1 mantissa bit; no inf or
                        NaN), stored packed: element 2i in the low 4 bits of byte i and 2i + 1
                        in the high 4 bits along K; A and B 32-byte aligned, K % 128 == 0 */
} tpgemm_dtype;

typedef enum {
    TPGEMM_OK = 0,
    TPGEMM_ERR_SHAPE = 1,   /* M, N, K not positive, or M%16, N%8, K%8 != 0 (K%16 for fp8) */
    TPGEMM_ERR_DTYPE = 2,   /* dtype not one of tpgemm_dtype */
    TPGEMM_ERR_BETA = 3,    /* beta not exactly 0.0f or 1.0f */
    TPGEMM_ERR_NULL = 4,    /* D, A or B NULL, or C NULL with beta == 1 */
    TPGEMM_ERR_ALIGN = 5,   /* a pointer not 16-byte aligned */
    TPGEMM_ERR_ALIAS = 6,   /* D overlaps A or B, or overlaps C without being equal to it */
    TPGEMM_ERR_ARCH = 7,    /* current device is not compute capability 10.3 (sm_103) */
    TPGEMM_ERR_LAUNCH = 8,  /* a CUDA call failed while enqueueing (detail has the CUDA error) */
    TPGEMM_ERR_TIMEOUT = 9, /* a kernel's bounded wait expired (see tpgemm_last_device_error) */
    TPGEMM_ERR_PATH = 10,   /* the forced kernel path cannot run this problem */
    TPGEMM_ERR_BOUNDS = 11  /* (debug builds, libtpgemm_debug.so) a device-side bounds check
                               failed; the access was skipped (see tpgemm_last_device_error) */
} tpgemm_status;

/* Kernel path selection, for tests and measurement. AUTO is the default plan. */
typedef enum {
    TPGEMM_PATH_AUTO = 0,
    TPGEMM_PATH_TCGEN05 = 1, /* TMA + tcgen05.mma + tensor-memory epilogue */
    TPGEMM_PATH_MMA_SYNC = 2 /* warp-level mma.sync.m16n8k16 (k8 for a K%16 == 8 tail) */
} tpgemm_path;

/*
 * D = A·B + beta·C  (alpha = 1).
 *
 * D, A, B, C: device pointers, 16-byte aligned, layouts as above. D == C is
 *   allowed (in-place D += A·B when beta == 1); any other overlap of D with A,
 *   B or C is rejected with TPGEMM_ERR_ALIAS.
 * M, N, K: logical sizes, positive, M % 16 == 0, N % 8 == 0, K % 8 == 0, each
 *   below 2^30, with M·N <= 2^36 and M·K, K·N <= 2^37 elements (no operand larger
 *   than one GPU holds); otherwise TPGEMM_ERR_SHAPE.
 * transA, transB: 0 or non-zero; select the stored orientation of A and B.
 * dtype: one of tpgemm_dtype (the fp8 ones with the orientation and K rules above).
 * beta: exactly 0.0f or 1.0f.
 * stream: a cudaStream_t (0 for the legacy default stream) on the current
 *   device; the call is asynchronous and returns once the work is enqueued.
 *
 * Returns TPGEMM_OK, or an error status with nothing enqueued (argument
 * errors), or TPGEMM_ERR_LAUNCH if CUDA refused the launch.
 */
tpgemm_status tpgemm_gemm(float* D, const void* A, const void* B, const float* C, int64_t M,
                          int64_t N, int64_t K, int transA, int transB, tpgemm_dtype dtype,
                          float beta, void* stream);

/* As tpgemm_gemm, with an explicit kernel path (TPGEMM_ERR_PATH if the forced
 * path cannot run the problem). Used by the tests to cover both kernels. */
tpgemm_status tpgemm_gemm_path(float* D, const void* A, const void* B, const float* C, int64_t M,
                               int64_t N, int64_t K, int transA, int transB, tpgemm_dtype dtype,
                               float beta, void* stream, tpgemm_path path);

/*
 * tpgemm_gemm without any device-memory allocation. (The pages have no
 * counterpart; this is a library convenience.)
 *
 * For callers that cannot or must not allocate device memory at the time of
 * the call: code running under a fixed, pre-reserved device-memory budget
 * (a long-running service that reserves everything at start-up), code inside
 * another allocator's out-of-memory or reclaim path, or a process whose device
 * memory is all held by another framework's pool. Such callers cannot use the
 * stream-K flags that the library would otherwise cudaMalloc per stream.
 *
 * Same arguments, layouts and results as tpgemm_gemm (within the same
 * tolerance; the K-summation order differs). The tcgen05 kernel runs in its
 * stream-K mode whenever the plan has a partial last wave that fits it (each
 * leftover tile split into two K halves on two clusters, twice the leftover
 * tiles at most the grid's clusters) and the call is neither in place (D ==
 * C) nor on a capturing stream (those take the split along N), with its flags
 * in one file-scope static
 * device array of TPGEMM_NOALLOC_SCRATCH_BYTES bytes that every GPU loading
 * the library holds until exit; otherwise it runs the plan that needs none
 * (the last wave split along N). tpgemm_last_plan() tells which plan ran
 * ("stream_k=1 scratch=static" for the static array). It calls no cudaMalloc,
 * cudaFree or other allocating routine.
 *
 * The first call on a device takes the array's device address
 * (cudaGetSymbolAddress) and zeroes it, synchronising the device;
 * make that first call before any stream capture. All calls on a device
 * share the array and it keeps the last call's contents: calls that overlap
 * on the GPU (e.g. on two streams at once) race, so serialise them.
 *
 * Returns as tpgemm_gemm.
 */
#define TPGEMM_NOALLOC_SCRATCH_BYTES 8192u
tpgemm_status tpgemm_gemm_noalloc(float* D, const void* A, const void* B, const float* C,
                                  int64_t M, int64_t N, int64_t K, int transA, int transB,
                                  tpgemm_dtype dtype, float beta, void* stream);

/*
 * Planner overrides (not on the pages; for measurement and tests). The
 * environment variables TPGEMM_TC_* (tile width, P rows, ring depth, staging
 * tiles, epilogue groups and last-segment helper warps, producers, raster
 * group, K rotation and direction, CTA pair, orientation, tail split,
 * stream-K, cluster cap, L2 priorities), TPGEMM_HOST_BLOCKS and
 * TPGEMM_HOST_EDGE (row blocks of tpgemm_gemm_host) and TPGEMM_WAIT_TIMEOUT_MS
 * (the bound of every in-kernel wait, default 2000 ms)
 * are read once per process, at the first call that plans a GEMM. This call
 * reads them again; calls already running keep the values they started with.
 */
void tpgemm_reload_tuning(void);

/*
 * Test aid for failure detection (not on the pages): tpgemm_gemm on the
 * tcgen05 path, except that CTA 0 never issues the TMA fill of its first ring
 * stage. The kernel's bounded waits then expire (TPGEMM_WAIT_TIMEOUT_MS), it
 * records TPGEMM_ERR_TIMEOUT for tpgemm_last_device_error(), drains its own
 * copies and MMAs, frees tensor memory and returns; D is left undefined. The
 * context stays usable. No GPU fault or hang is involved.
 */
tpgemm_status tpgemm_test_gemm_withhold_fill(float* D, const void* A, const void* B,
                                             const float* C, int64_t M, int64_t N, int64_t K,
                                             int transA, int transB, tpgemm_dtype dtype,
                                             float beta, void* stream);

/*
 * Block-scaled fp8 multiply (MX):
 *   D[i,j] = sum_k (A[i,k] * 2^(SFA[i, k/32] - 127)) * (B[k,j] * 2^(SFB[j, k/32] - 127))
 *            + beta * C[i,j].
 * The sync-gemm page ("TVM TIRx 同步 GEMM 深度解析", section 七) lists block
 * scaling (SFA, SFB) among gemm_async's operand forms without defining it;
 * this is the OCP Microscaling reading: every 32 consecutive K elements of a
 * row of A (of a column of B) share one E8M0 scale, 2^(e - 127), e = 255 NaN.
 * Runs on the tcgen05 kernel as tcgen05.mma kind::mxf8f6f4.block_scale with
 * the scales copied into tensor memory by tcgen05.cp.
 *
 * A: [M,K] fp8 (dtype TPGEMM_E4M3 or TPGEMM_E5M2), K-contiguous. B: [N,K] fp8
 *   of the same dtype (stored as for tpgemm_gemm with transB = 1).
 * SFA: [M][ceil(K/32)] E8M0 bytes, row-major. SFB: [N][ceil(K/32)] E8M0 bytes.
 * C, D, M, N, K, beta, stream: as tpgemm_gemm (K % 16 == 0 as for fp8).
 * workspace: caller-owned device memory of at least
 *   tpgemm_gemm_mx_workspace_bytes(M, N, K) bytes, 256-byte aligned, that the
 *   call packs the scales into (the library allocates nothing); it must not
 *   overlap any operand and must stay untouched until the GEMM has run.
 * Returns as tpgemm_gemm, plus TPGEMM_ERR_NULL for a NULL scale matrix or a
 * missing / short workspace and TPGEMM_ERR_ALIAS for overlaps with it.
 */
tpgemm_status tpgemm_gemm_mx(float* D, const void* A, const void* B, const float* C,
                             const uint8_t* SFA, const uint8_t* SFB, int64_t M, int64_t N,
                             int64_t K, tpgemm_dtype dtype, float beta, void* workspace,
                             size_t workspace_bytes, void* stream);

/* Bytes of workspace tpgemm_gemm_mx needs: the packed scales of A and of B,
 * 512 bytes per (128 rows, 128 K) of an operand tile, four times over for
 * tiles of more than 128 rows, sized for the largest tiling a plan can choose
 * (about 0.8 MB per 1024 rows per 1024 K of the larger operand). 0 for
 * non-positive or oversized shapes. */
size_t tpgemm_gemm_mx_workspace_bytes(int64_t M, int64_t N, int64_t K);

/* Host copy of the block-scaled instruction descriptor encoder (test aid, as
 * tpgemm_encode_idesc): kind::mxf8f6f4 with E8M0 scales, A and B of `dtype`
 * (TPGEMM_E4M3 / _E5M2), both K-major, UMMA shape m x n, and the scale-factor
 * IDs of A and B (0..3). Returns 0 for another dtype. */
uint32_t tpgemm_encode_idesc_mx(tpgemm_dtype dtype, int m, int n, int a_sf_id, int b_sf_id);

/* Bytes of device workspace tpgemm_gemm_host needs for this problem: room for
 * A, B, D and (beta == 1) C, each 256-byte aligned. Returns 0 for a shape,
 * dtype or beta that tpgemm_gemm would reject. */
size_t tpgemm_gemm_host_workspace_bytes(int64_t M, int64_t N, int64_t K, tpgemm_dtype dtype,
                                        float beta);

/*
 * D = A·B + beta·C with A, B, C and D in HOST memory (layouts as for
 * tpgemm_gemm). Page-locked host memory lets the copies run asynchronously and
 * overlap; pageable memory works but serialises them.
 *
 * The call enqueues, ordered after the work already on `stream`: the copy of B
 * to the device, then for each row block of M (about 12 for large M, the first
 * and last of them shorter) the copy-in of its A rows (and C
 * rows), the multiply of that block by the tcgen05 / mma.sync kernels, and the
 * copy-out of its D rows. Copies run on two library-owned helper streams so
 * that block i+1's copy-in and block i-1's copy-out overlap block i's multiply;
 * `stream` is ordered after the last copy-out, so synchronising `stream` (or
 * an event recorded on it afterwards) makes D_host valid. The host buffers
 * must stay valid and unmodified until then.
 *
 * workspace: device memory owned by the caller, at least
 * tpgemm_gemm_host_workspace_bytes(M, N, K, dtype, beta) bytes, 256-byte
 * aligned; its contents on entry do not matter. The library allocates nothing.
 *
 * Returns TPGEMM_OK once everything is enqueued; argument errors
 * (TPGEMM_ERR_SHAPE / _DTYPE / _BETA / _NULL / _ALIGN) before anything is
 * enqueued; TPGEMM_ERR_LAUNCH if CUDA refused a copy or a launch.
 */
tpgemm_status tpgemm_gemm_host(float* D_host, const void* A_host, const void* B_host,
                               const float* C_host, int64_t M, int64_t N, int64_t K, int transA,
                               int transB, tpgemm_dtype dtype, float beta, void* workspace,
                               size_t workspace_bytes, void* stream);

/*
 * ------------------------------------------------------------------------
 * Shared memory -> tensor memory copy (tcgen05.cp), as a standalone primitive.
 *
 * The operation is the smem-tmem variant of copy_async described on the page
 * "TVM Blackwell tcgen05.cp 全解析": a matrix of `rows` rows x `row_bits` bits
 * in shared memory, named by a 64-bit shared-memory matrix descriptor, is
 * copied into tensor memory by single-thread tcgen05.cp instructions of one of
 * six shape / multicast forms (section 形状选择), with the row -> lane and
 * replica pattern of each form given in section 形状 → 行/复制模式映射表:
 *
 *   form                     rows  bits/row  row r goes to lane(s)
 *   128x256b                  128    256      r
 *   4x256b                      4    256      32 r            (rows 0..3)
 *   128x128b                  128    128      r
 *   64x128b.warpx2::02_13      64    128      r, r + 64
 *   64x128b.warpx2::01_23      64    128      (r % 32) + 64 (r / 32), + 32
 *   32x128b.warpx4             32    128      r, r + 32, r + 64, r + 96
 *
 * Bits [32 c, 32 c + 32) of a row go to tensor-memory column tmem_col + c.
 * Wider regions are copied by several instructions along the row (one per
 * 256 or 128 bits), and a 4x256b region of 4 j rows by j lane-tiled
 * instructions: row 4 i + q goes to lane 32 q + i (the first j lanes of each
 * warp's quadrant). The plan issues each instruction with the descriptor
 * encoded once and only its 14-bit start address patched (section 调度算法四步,
 * steps 3 and 4), and the caller-side completion is a tcgen05.commit to an
 * mbarrier (section 演示程序).
 *
 * Shared-memory layout of the source (the K-major canonical layout of the
 * matrix descriptor; byte offsets from a 1024-byte aligned buffer):
 *   SWIZZLE_NONE: 16-byte unit u of row r at
 *       smem_offset + (r / 8) sbo + (r % 8) 16 + u lbo
 *   SWIZZLE_32B / _64B / _128B (S = 32, 64, 128 bytes per swizzle row, U =
 *   S / 16 units each): unit u of row r at swz(smem_offset + (u / U) lbo +
 *   (r / 8) sbo + (r % 8) S + 16 (u % U)), where swz XORs address bits
 *   [4, 4 + log2 U) with bits [7, 7 + log2 U); a row wider than one swizzle row
 *   continues in the next swizzle atom, lbo bytes on.
 * The planner rejects strides under which two units would share bytes.
 */
typedef enum {
    TPGEMM_CP_SWIZZLE_NONE = 0,
    TPGEMM_CP_SWIZZLE_32B = 1,
    TPGEMM_CP_SWIZZLE_64B = 2,
    TPGEMM_CP_SWIZZLE_128B = 3
} tpgemm_cp_swizzle;

/*
 * The tcgen05 descriptor encoders the kernels use, callable on the host (not on
 * the pages: test aids). They let each field position be checked against the
 * PTX ISA's descriptor tables without a GPU. Pure functions; no CUDA calls.
 *
 * tpgemm_encode_smem_desc: the 64-bit shared-memory matrix descriptor with
 *   start address start_addr (bytes; its bits 4-17 are kept), leading- and
 *   stride-dimension byte offsets lbo_bytes / sbo_bytes (multiples of 16, below
 *   2^18), relative LBO mode, base offset 0 and the layout type of `swizzle`.
 * tpgemm_encode_idesc: the 32-bit instruction descriptor of a dense
 *   tcgen05.mma with an f32 accumulator: kind::f16 for TPGEMM_F16 / _BF16,
 *   kind::f8f6f4 for TPGEMM_E4M3 / _E5M2, A and B of `dtype`, each K-major (0)
 *   or MN-major (1), UMMA shape m x n. Returns 0 for an unknown dtype.
 */
uint64_t tpgemm_encode_smem_desc(uint32_t start_addr, uint32_t lbo_bytes, uint32_t sbo_bytes,
                                 tpgemm_cp_swizzle swizzle);
uint32_t tpgemm_encode_idesc(tpgemm_dtype dtype, int a_mn_major, int b_mn_major, int m, int n);

/* tcgen05.cp shape with its multicast qualifier. AUTO: the widest form whose
 * pattern matches the destination lanes (the page's candidate order
 * 128x256b, 4x256b, 128x128b, 64x128b.02_13, 64x128b.01_23, 32x128b.warpx4). */
typedef enum {
    TPGEMM_CP_AUTO = 0,
    TPGEMM_CP_128x256b = 1,
    TPGEMM_CP_4x256b = 2,
    TPGEMM_CP_128x128b = 3,
    TPGEMM_CP_64x128b_WARPX2_02_13 = 4,
    TPGEMM_CP_64x128b_WARPX2_01_23 = 5,
    TPGEMM_CP_32x128b_WARPX4 = 6
} tpgemm_cp_shape;

/* Where the region's rows go in tensor memory (lane_offset added to each). */
typedef enum {
    TPGEMM_CP_LANES_ROWS = 0,         /* row r -> lane r                        */
    TPGEMM_CP_LANES_QUADRANTS = 1,    /* row 4 i + q -> lane 32 q + i           */
    TPGEMM_CP_LANES_PAIRS_02_13 = 2,  /* row r -> lanes r, r + 64 (r < 64)      */
    TPGEMM_CP_LANES_PAIRS_01_23 = 3,  /* row r -> lanes (r%32) + 64 (r/32) + {0, 32} */
    TPGEMM_CP_LANES_ALL_QUADS = 4     /* row r -> lanes r + {0, 32, 64, 96}      */
} tpgemm_cp_lanes;

typedef struct {
    int rows;                  /* rows of the region                               */
    int row_bits;              /* bits per row: a positive multiple of 128         */
    tpgemm_cp_swizzle swizzle; /* source layout                                    */
    uint32_t lbo_bytes;        /* distance between a row's units (unswizzled) or
                                  between swizzle atoms along the row (swizzled)  */
    uint32_t sbo_bytes;        /* distance between 8-row groups (multiple of 16)   */
    uint32_t smem_offset;      /* region start in the staging buffer               */
    int tmem_col;              /* first tensor-memory column (multiple of 4)       */
    int lane_offset;           /* added to every destination lane                  */
    tpgemm_cp_lanes lanes;     /* destination row -> lane pattern                  */
    tpgemm_cp_shape shape;     /* instruction form, or AUTO                        */
    int cta_group;             /* 1, or 2 (the even CTA of a pair issues; each CTA
                                  copies its own shared memory to its own tensor
                                  memory)                                         */
} tpgemm_cp_desc;

/* Parse a form name ("128x256b", "4x256b", "128x128b", "64x128b.warpx2::02_13",
 * "64x128b.warpx2::01_23", "32x128b.warpx4"; the multicast part may also be
 * given alone after a '.'). TPGEMM_ERR_SHAPE with a readable reason for an
 * unknown shape, a 64x128b without its multicast, or an illegal combination
 * (e.g. "128x256b.warpx4"). */
tpgemm_status tpgemm_cp_parse_shape(const char* name, tpgemm_cp_shape* out);

/* The plan for a copy, as text into buf: the chosen form, the number of
 * instructions, the descriptor fields (LBO, SBO, swizzle mode) and, per
 * instruction, its shared-memory start offset and tensor-memory lane / column.
 * Returns TPGEMM_OK, or TPGEMM_ERR_SHAPE with the reason in
 * tpgemm_last_error_detail() (and in buf): form / lane-pattern mismatch,
 * region larger than the 128 lanes, column offset not 128-bit aligned, SBO not
 * a multiple of 16 bytes, a row wider than the swizzle row, a region that
 * does not tile into the form's rows and bits. */
tpgemm_status tpgemm_cp_plan(const tpgemm_cp_desc* d, char* buf, int buflen);

/*
 * Round trip through tensor memory, for tests and measurement: one CTA (two
 * for cta_group 2) copies `image_bytes` bytes from `smem_image` (device memory)
 * into a 1024-byte aligned shared-memory buffer, fills tensor-memory columns
 * [0, ncols) of all 128 lanes with fill(lane, col) = fill_base + lane * 65536
 * + col (tcgen05.st), issues the planned tcgen05.cp instructions, commits them
 * to an mbarrier and waits, then reads the same columns back (tcgen05.ld
 * 32x32b) into tmem_out[lane * ncols + col] (device memory, uint32). For
 * cta_group 2, smem_image holds the two CTAs' images back to back and
 * tmem_out the two CTAs' results. ncols: 32..512, a multiple of 32, covering
 * the copied columns; image_bytes: a multiple of 16, at most 196608.
 * Asynchronous on `stream`; argument errors as tpgemm_cp_plan, plus
 * TPGEMM_ERR_NULL / _ALIGN for the pointers.
 */
tpgemm_status tpgemm_cp_roundtrip(uint32_t* tmem_out, const void* smem_image, size_t image_bytes,
                                  const tpgemm_cp_desc* d, uint32_t fill_base, int ncols,
                                  void* stream);

/* tpgemm_cp_roundtrip on `ctas` CTAs at once (a multiple of cta_group), each
 * issuing the planned instruction list `repeat` times (1..2^20) before its
 * commit, for measuring the copy's throughput. Every CTA (every pair for
 * cta_group 2) reads the same image(s); CTA k writes rows [128 k, 128 k + 128)
 * of tmem_out, which must hold ctas * 128 * ncols words. With repeat > 1 the
 * later copies rewrite the same cells, so the result is that of one copy.
 * issuers (1..8): threads that share the list, lane 0 of warps 0..issuers-1,
 * each taking every issuers-th instruction and committing its own to the
 * mbarrier (1 is the single-thread protocol of the page; a tcgen05.cp holds
 * its issuing thread for about 90 ns, so more issuers copy proportionally
 * faster). */
tpgemm_status tpgemm_cp_roundtrip_repeat(uint32_t* tmem_out, const void* smem_image,
                                         size_t image_bytes, const tpgemm_cp_desc* d,
                                         uint32_t fill_base, int ncols, int repeat, int ctas,
                                         int issuers, void* stream);

/*
 * ------------------------------------------------------------------------
 * Tensor memory <-> registers (tcgen05.st / tcgen05.ld), the tmem<->local copy
 * of the page "TVM TIRx copy_async -> tcgen05_ldst": one warpgroup moves a
 * 128-lane x `cols`-column tile between tensor memory and its registers, `cols`
 * registers per thread. Shapes (register of thread t of a warp, in the warp's
 * 32 lanes; two issues of 16 lanes each, lanes +0 and +16, for the .16x*b
 * shapes, registers [0, cols/2) then [cols/2, cols)):
 *   .32x32b   thread t -> lane t, register j -> column j
 *   .16x64b   16 lanes x 2 columns per repeat
 *   .16x128b  16 lanes x 4 columns per repeat
 *   .16x256b  16 lanes x 8 columns per repeat; within one repeat, register s of
 *             thread t at lane t/4 + 8 (s/2), column 2 (t%4) + s%2 (the m16n8
 *             accumulator fragment of the mma.sync gemm page, section 三 D_FRAG)
 */
typedef enum {
    TPGEMM_TMEM_32x32b = 0,
    TPGEMM_TMEM_16x64b = 1,
    TPGEMM_TMEM_16x128b = 2,
    TPGEMM_TMEM_16x256b = 3
} tpgemm_tmem_shape;

/* Round trip, for tests: fill tensor-memory columns [0, 32) of all 128 lanes
 * with fill_base + 65536 lane + col, store regs_in ([128 threads][cols] uint32,
 * device) with st_shape at column tmem_col, read the 32 columns back with
 * .32x32b into tmem_out ([128][32]), then load with ld_shape into regs_out
 * ([128][cols]). cols: 2, 4, 8 or 16 (at least 2 / 4 / 8 for .16x64b / 128b /
 * 256b); tmem_col: a multiple of 8 with tmem_col + cols <= 32. */
tpgemm_status tpgemm_tmem_ldst_roundtrip(uint32_t* regs_out, uint32_t* tmem_out,
                                        const uint32_t* regs_in, tpgemm_tmem_shape st_shape,
                                        tpgemm_tmem_shape ld_shape, int cols, int tmem_col,
                                        uint32_t fill_base, void* stream);

/*
 * ------------------------------------------------------------------------
 * Vectorised global <-> shared copy, the gmem_smem path of the vec_auto copy
 * on the page "TVM TIRx CUDA 向量化内存拷贝实战 (gmem_smem)". A region of rows x
 * cols elements moves between a global buffer (row stride g_row_stride,
 * starting g_offset elements in) and a shared buffer (row stride
 * s_row_stride, starting s_offset elements in), by `threads` threads:
 *   - partition [outer, threads, vec]: the region's elements in row order,
 *     thread tid of round f copying the vec elements from (f threads + tid) vec;
 *   - vec: the widest of 16, 8, 4, 2, 1 bytes (whole elements) that divides the
 *     contiguous tail (a row, or the whole region when both sides are dense
 *     along rows), the elements per thread, both row strides and both offsets;
 *   - a swizzled shared buffer keeps each vector inside one 16-byte chunk and
 *     XORs byte offset bits [4, 4 + log2(S / 16)) with bits [7, ...), S = 32,
 *     64 or 128, offsets counted from the start of the shared buffer.
 * The gate: threads is 1, 32, 128 or a CTA of 64..1024 (whole warps), and the
 * element count is a multiple of threads (otherwise TPGEMM_ERR_SHAPE).
 */
typedef struct {
    int rows, cols;               /* region, elements                     */
    int elem_bytes;               /* 1, 2, 4 or 8                          */
    int64_t g_row_stride;         /* global row stride, elements (>= cols) */
    int64_t g_offset;             /* region start in the global buffer     */
    int s_row_stride;             /* shared row stride, elements (>= cols) */
    int s_offset;                 /* region start in the shared buffer     */
    tpgemm_cp_swizzle s_swizzle;  /* shared layout                          */
    int threads;                  /* the copying scope                     */
} tpgemm_vcopy_desc;

/* The plan as text ("vec_bytes=16 vec=4 outer=8 threads=32 ..."), or the
 * rejection reason (also in tpgemm_last_error_detail()). */
tpgemm_status tpgemm_vcopy_plan(const tpgemm_vcopy_desc* d, char* buf, int buflen);

/* Round trip global -> shared -> global on `ctas` CTAs of d->threads threads:
 * CTA k copies the region starting cta_stride * k elements into src (device,
 * buffer_bytes) through its shared buffer into the same place of dst (device,
 * buffer_bytes); nothing else of dst is written. smem_out (device, may be
 * NULL): each CTA's shared buffer after the first copy, zero outside the
 * region, at smem_out + k * (shared bytes of the plan). */
tpgemm_status tpgemm_vcopy_roundtrip(void* dst, const void* src, size_t buffer_bytes,
                                     const tpgemm_vcopy_desc* d, int ctas, int64_t cta_stride,
                                     void* smem_out, void* stream);

/* Static English name of a status. Never NULL. */
const char* tpgemm_status_string(tpgemm_status s);

/* Readable reason for the last non-OK status returned on this thread
 * (e.g. "N=12 is not a multiple of 8"). Thread-local; valid until the next
 * call on the same thread. Empty string if the last call succeeded. */
const char* tpgemm_last_error_detail(void);

/* Device-side status of the kernels launched so far on the current device:
 * TPGEMM_ERR_TIMEOUT if any bounded wait inside a kernel expired, in a debug
 * build (TPGEMM_DEBUG, libtpgemm_debug.so) TPGEMM_ERR_BOUNDS if a device-side
 * bounds check on a computed tensor-memory column, TMA coordinate or stream-K
 * flag index failed (the detail names the site; the access was skipped, the
 * result is undefined), else TPGEMM_OK. Synchronises the device first.
 * Reading it resets it to OK. */
tpgemm_status tpgemm_last_device_error(void);

/* The plan tpgemm_gemm would use for this problem, written as text into buf
 * (at most buflen bytes including the terminator): kernel path, tile shape,
 * operand roles, grid. Returns the status the call itself would return for
 * the arguments' shape, dtype and beta (pointers are not examined). */
tpgemm_status tpgemm_describe_plan(int64_t M, int64_t N, int64_t K, int transA, int transB,
                                   tpgemm_dtype dtype, float beta, tpgemm_path path, char* buf,
                                   int buflen);

/* The plan of the last GEMM this thread enqueued (tpgemm_gemm, tpgemm_gemm_path,
 * tpgemm_gemm_noalloc, or a block of tpgemm_gemm_host), as text in the format of
 * tpgemm_describe_plan, with the grid actually launched and where its stream-K
 * scratch lived ("scratch=none", "allocated" or "static"). Thread-local.
 * Returns TPGEMM_ERR_NULL (and an empty string) if this thread has enqueued
 * none. (Not on the pages: an introspection aid.) */
tpgemm_status tpgemm_last_plan(char* buf, int buflen);

/* Library version as "major.minor.patch". */
const char* tpgemm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TPGEMM_H */
