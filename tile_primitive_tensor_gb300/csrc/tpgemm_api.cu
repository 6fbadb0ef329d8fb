// C-ABI entry points of libtpgemm.so: argument validation, kernel planning,
// TMA tensor-map encoding and launch on the caller's stream.
//
// The acceptance rules are those of the TVM TIRx synchronous gemm page
// ("TVM TIRx 同步 GEMM 深度解析", section 二 What it accepts and its
// source-level conditions): M % 16 = 0, N % 8 = 0, K % 8 = 0; A and B both
// float16 or both bfloat16; C and D float32; alpha = 1; beta in {0, 1};
// transpose flags only select the stored orientation. As on that page, every
// rejection carries a readable reason (there via DispatchFail / RuntimeError,
// here via tpgemm_last_error_detail).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <string>

#include "ptx.cuh"
#include "tpgemm.h"
#include "tpgemm_internal.h"

namespace {

thread_local std::string g_detail;

tpgemm_status fail(tpgemm_status s, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_detail = buf;
    return s;
}

// ------------------------------------------------------------ device cache
struct DeviceInfo {
    bool valid = false;
    int major = 0, minor = 0, sms = 0;
};
constexpr int kMaxDevices = 64;
DeviceInfo g_devices[kMaxDevices];
std::mutex g_mutex;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

tpgemm_status device_info(DeviceInfo* out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return fail(TPGEMM_ERR_ARCH, "no CUDA device available: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return fail(TPGEMM_ERR_ARCH, "device index %d unsupported", dev);
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceInfo& d = g_devices[dev];
    if (!d.valid) {
        if (cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return fail(TPGEMM_ERR_ARCH, "cannot query device %d", dev);
        d.valid = true;
    }
    *out = d;
    return TPGEMM_OK;
}

tpgemm_status get_encoder(PFN_cuTensorMapEncodeTiled_v12000* fn) {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_encode) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                                         cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !p)
            return fail(TPGEMM_ERR_LAUNCH, "cuTensorMapEncodeTiled not available from the driver");
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    *fn = g_encode;
    return TPGEMM_OK;
}

// ---------------------------------------------------------- tuning overrides
// Planner overrides read from the environment, used to sweep plans on real
// problems and by the tests to cover every plan the heuristics can choose.
// They are read once per process (on first use) into an immutable snapshot;
// tpgemm_reload_tuning() takes a new one. -1 (or 0 for orient) = not set.
struct Tuning {
    int bn = -1, bp = -1, dep_early = -1, epi_bufs = -1, epi_groups = -1, group = -1;
    int krotate = -1, max_clusters = -1, pair = -1, producers = -1, sk = -1, stages = -1;
    int tail = -1, host_blocks = -1, l2_p = -1, l2_q = -1, l2_cd = -1, snake = -1, krev = -1;
    int epi_help = -1, host_edge = -1;
    int debug_plant = -1;  // debug builds only
    int orient = 0;  // 1 "swap", 2 "normal"
    long long wait_ms = -1;
};

Tuning read_tuning() {
    Tuning t;
    auto geti = [](const char* name, int* out) {
        if (const char* f = getenv(name)) *out = atoi(f);
    };
    geti("TPGEMM_TC_BN", &t.bn);
    geti("TPGEMM_TC_BP", &t.bp);
    geti("TPGEMM_TC_DEP_EARLY", &t.dep_early);
    geti("TPGEMM_TC_EPI_BUFS", &t.epi_bufs);
    geti("TPGEMM_TC_EPI_GROUPS", &t.epi_groups);
    geti("TPGEMM_TC_EPI_HELP", &t.epi_help);
    geti("TPGEMM_TC_GROUP", &t.group);
    geti("TPGEMM_TC_KROTATE", &t.krotate);
    geti("TPGEMM_TC_KREV", &t.krev);
    geti("TPGEMM_TC_MAX_CLUSTERS", &t.max_clusters);
    geti("TPGEMM_TC_PAIR", &t.pair);
    geti("TPGEMM_TC_PRODUCERS", &t.producers);
    geti("TPGEMM_TC_SK", &t.sk);
    geti("TPGEMM_TC_STAGES", &t.stages);
    geti("TPGEMM_TC_TAIL", &t.tail);
    geti("TPGEMM_HOST_BLOCKS", &t.host_blocks);
    geti("TPGEMM_HOST_EDGE", &t.host_edge);
    geti("TPGEMM_TC_L2_P", &t.l2_p);
    geti("TPGEMM_TC_L2_Q", &t.l2_q);
    geti("TPGEMM_TC_L2_CD", &t.l2_cd);
    geti("TPGEMM_TC_SNAKE", &t.snake);
    if (const char* f = getenv("TPGEMM_TC_ORIENT")) {
        if (!strcmp(f, "swap")) t.orient = 1;
        if (!strcmp(f, "normal")) t.orient = 2;
    }
    if (const char* f = getenv("TPGEMM_WAIT_TIMEOUT_MS")) t.wait_ms = atoll(f);
#ifdef TPGEMM_DEBUG
    geti("TPGEMM_DEBUG_PLANT", &t.debug_plant);
#endif
    return t;
}

std::atomic<const Tuning*> g_tuning{nullptr};
std::mutex g_tuning_mutex;

// Snapshots are never freed (a reload is rare), so a reference stays valid
// for the rest of the call that took it.
const Tuning& tuning() {
    const Tuning* t = g_tuning.load(std::memory_order_acquire);
    if (t) return *t;
    std::lock_guard<std::mutex> lock(g_tuning_mutex);
    t = g_tuning.load(std::memory_order_acquire);
    if (!t) {
        t = new Tuning(read_tuning());
        g_tuning.store(t, std::memory_order_release);
    }
    return *t;
}

// ------------------------------------------------------------- validation
bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

// The narrow types run as tcgen05.mma kind::f8f6f4 (or its block-scaled form).
bool is_f8f6f4(tpgemm_dtype d) {
    return d == TPGEMM_E4M3 || d == TPGEMM_E5M2 || d == TPGEMM_E2M1;
}

// Bits of one element of A and B (fp4 is stored two per byte).
int elem_bits(tpgemm_dtype d) { return d == TPGEMM_E2M1 ? 4 : (is_f8f6f4(d) ? 8 : 16); }

size_t operand_bytes(tpgemm_dtype d, int64_t elems) {
    return size_t(elems) * size_t(elem_bits(d)) / 8;
}

// The format code the instruction descriptor carries for A and B: kind::f16
// f16 = 0 / bf16 = 1; kind::f8f6f4 e4m3 = 0 / e5m2 = 1 / e2m1 = 5.
uint32_t format_code(tpgemm_dtype d) {
    return d == TPGEMM_E2M1 ? 5u : ((d == TPGEMM_BF16 || d == TPGEMM_E5M2) ? 1u : 0u);
}

tpgemm_status check_shape(int64_t M, int64_t N, int64_t K, tpgemm_dtype dtype, float beta) {
    if (M <= 0 || N <= 0 || K <= 0)
        return fail(TPGEMM_ERR_SHAPE, "M=%lld N=%lld K=%lld must all be positive", (long long)M,
                    (long long)N, (long long)K);
    if (M % 16) return fail(TPGEMM_ERR_SHAPE, "M=%lld is not a multiple of 16", (long long)M);
    if (N % 8) return fail(TPGEMM_ERR_SHAPE, "N=%lld is not a multiple of 8", (long long)N);
    if (K % 8) return fail(TPGEMM_ERR_SHAPE, "K=%lld is not a multiple of 8", (long long)K);
    // Coordinates and tile counts are 32-bit inside the kernels.
    const int64_t lim = int64_t(1) << 30;
    if (M >= lim || N >= lim || K >= lim)
        return fail(TPGEMM_ERR_SHAPE, "M, N, K must each be below 2^30");
    // No operand larger than one GPU can hold (this also keeps tile counts,
    // whose product is at most M N / 2^11, within 32 bits).
    if (M * N > (int64_t(1) << 36) || M * K > (int64_t(1) << 37) || K * N > (int64_t(1) << 37))
        return fail(TPGEMM_ERR_SHAPE,
                    "M=%lld N=%lld K=%lld: an operand exceeds one GPU's memory (at most 2^36 "
                    "elements of C / D and 2^37 of A or B)",
                    (long long)M, (long long)N, (long long)K);
    if (dtype != TPGEMM_F16 && dtype != TPGEMM_BF16 && !is_f8f6f4(dtype))
        return fail(TPGEMM_ERR_DTYPE,
                    "dtype %d is not TPGEMM_F16 (0), TPGEMM_BF16 (1), TPGEMM_E4M3 (2), "
                    "TPGEMM_E5M2 (3) or TPGEMM_E2M1 (4)",
                    int(dtype));
    if (dtype == TPGEMM_E2M1 && K % 128)
        return fail(TPGEMM_ERR_SHAPE,
                    "K=%lld is not a multiple of 128 (fp4 rows are loaded and unpacked 128 "
                    "elements at a time)",
                    (long long)K);
    if (is_f8f6f4(dtype) && K % 16)
        return fail(TPGEMM_ERR_SHAPE,
                    "K=%lld is not a multiple of 16 (fp8 rows must be whole 16-byte units)",
                    (long long)K);
    if (!(beta == 0.0f || beta == 1.0f))
        return fail(TPGEMM_ERR_BETA, "beta=%g; only 0 and 1 are supported", double(beta));
    return TPGEMM_OK;
}

tpgemm_status check_pointers(float* D, const void* A, const void* B, const float* C, int64_t M,
                             int64_t N, int64_t K, float beta, tpgemm_dtype dtype) {
    if (!D) return fail(TPGEMM_ERR_NULL, "D is NULL");
    if (!A) return fail(TPGEMM_ERR_NULL, "A is NULL");
    if (!B) return fail(TPGEMM_ERR_NULL, "B is NULL");
    if (beta == 1.0f && !C) return fail(TPGEMM_ERR_NULL, "C is NULL with beta = 1");
    auto misaligned = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; };
    if (misaligned(D)) return fail(TPGEMM_ERR_ALIGN, "D=%p is not 16-byte aligned", (void*)D);
    if (misaligned(A)) return fail(TPGEMM_ERR_ALIGN, "A=%p is not 16-byte aligned", A);
    if (misaligned(B)) return fail(TPGEMM_ERR_ALIGN, "B=%p is not 16-byte aligned", B);
    // The TMA unpacks fp4 from 32-byte aligned rows.
    auto misaligned32 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 31u) != 0; };
    if (dtype == TPGEMM_E2M1 && misaligned32(A))
        return fail(TPGEMM_ERR_ALIGN, "A=%p is not 32-byte aligned (fp4)", A);
    if (dtype == TPGEMM_E2M1 && misaligned32(B))
        return fail(TPGEMM_ERR_ALIGN, "B=%p is not 32-byte aligned (fp4)", B);
    if (beta == 1.0f && misaligned(C))
        return fail(TPGEMM_ERR_ALIGN, "C=%p is not 16-byte aligned", (const void*)C);
    const size_t dn = size_t(M) * size_t(N) * 4;
    if (overlaps(D, dn, A, operand_bytes(dtype, M * K)))
        return fail(TPGEMM_ERR_ALIAS, "D overlaps A");
    if (overlaps(D, dn, B, operand_bytes(dtype, K * N)))
        return fail(TPGEMM_ERR_ALIAS, "D overlaps B");
    if (beta == 1.0f && static_cast<const void*>(C) != static_cast<const void*>(D) &&
        overlaps(D, dn, C, dn))
        return fail(TPGEMM_ERR_ALIAS, "D overlaps C without being equal to it");
    return TPGEMM_OK;
}

// ----------------------------------------------------------------- planning
enum class Kernel { MmaSync, Tc };

struct Plan {
    Kernel kernel = Kernel::Tc;
    tpg::TcParams tc{};
    int grid = 0;      // persistent grid (CTAs)
    int max_grid = 0;  // CTAs of every cluster the device holds at once
    int sms = 0;
    bool swap = false;
};

// Bound on every mbarrier wait inside the tcgen05 kernel: 2 s, or
// TPGEMM_WAIT_TIMEOUT_MS (read at every call, so a test can shorten it).
using tpg::wait_timeout_ns;

// Shared bytes of one stage tile of an operand with `rows` rows along MN and
// 64 K elements: K-contiguous tiles are rows x 128 bytes; MN-contiguous tiles
// are whole 64-row atoms of 64 K rows x 128 bytes.
uint32_t stage_tile_bytes(int rows, bool mn) {
    return mn ? uint32_t((rows + 63) / 64) * 8192u : uint32_t(rows) * 128u;
}

// Accumulator width (UMMA N) for the normal orientation. With the CTA-pair
// MMA, the widest tile (256, or N rounded up to 32 when narrower) measured
// best at 4096^3 and 8192^3. A single CTA takes the multiple of 32 in
// [128, 256] that minimises (persistent waves) x (tile width + a fixed
// per-tile cost), i.e. the least wave-quantisation loss; ties go to the
// wider tile (fewer re-reads of A).
int pick_bn(int64_t M, int64_t N, int sms, bool pair) {
    // TPGEMM_TC_BN (a multiple of 32 in [32, 256]) forces the width; the
    // tests use it to cover every width the heuristic can choose.
    {
        const int v = tuning().bn;
        if (v >= 32 && v <= 256 && v % 32 == 0) return v;
    }
    if (N <= 64) return int(((N + 15) / 16) * 16);
    if (N <= 128) return 128;
    if (pair) return N >= 256 ? 256 : int(((N + 31) / 32) * 32);
    int best = 256;
    int64_t best_cost = -1;
    for (int bn = 256; bn >= 128; bn -= 32) {
        const int64_t tiles = ((M + 127) / 128) * ((N + bn - 1) / bn);
        const int64_t waves = (tiles + sms - 1) / sms;
        const int64_t cost = waves * (bn + 32);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = bn;
        }
    }
    return best;
}

tpgemm_status plan_tc(int64_t M, int64_t N, int64_t K, bool transA, bool transB,
                      tpgemm_dtype dtype, float beta, int sms, Plan* out, bool mx = false) {
    const bool fp8 = is_f8f6f4(dtype);
    tpg::TcParams p{};
    // Small M: swap operands so N runs along the 128 tensor-memory lanes and
    // all of M fits one accumulator (UMMA N = M <= 256, a multiple of 16).
    // Small M: all of M fits one accumulator (swap_small). Otherwise the
    // orientation is chosen so that the MMA's B operand (Q) is K-contiguous
    // when one orientation allows it: with A stored [M,K] and B stored [K,N]
    // the swapped orientation makes Q = A. Measured on GB300: an MN-contiguous
    // B operand costs 7-11 %, an MN-contiguous A operand about 2 % (8192^3
    // with B [K,N]: 726 -> 674 us). TPGEMM_TC_ORIENT=swap|normal overrides.
    // Block-scaled plans (mx) keep the first half of tensor memory past the
    // tile's columns for the scale slots, so their swapped tiles are at most
    // 160 wide.
    const bool swap_small = mx ? (M <= 160 && N > M) : (M <= 256 && N > M);
    bool swap = swap_small || (!transA && !transB);
    if (tuning().orient == 1) swap = true;
    if (tuning().orient == 2 && !swap_small) swap = false;
    const int64_t Mp = swap ? N : M;
    const int64_t Nq = swap ? M : N;
    const bool p_mn = swap ? !transB : transA;
    const bool q_mn = swap ? transA : !transB;
    // fp8 operands are loaded K-contiguous only (A [M,K], B [N,K]).
    if (fp8 && (p_mn || q_mn))
        return fail(TPGEMM_ERR_PATH,
                    "fp8 A and B must both be K-contiguous: A stored [M,K] (transA = 0) and B "
                    "stored [N,K] (transB = 1)");
    // The CTA-pair MMA needs at least two 128-row P tiles.
    const bool pair_wanted = Mp > 128;
    // Block-scaled tiles are at most 224 wide: each accumulator half keeps the
    // columns past its tile for the scale slots (two 12-column slots per half
    // at 224, so a 4-deep ring; five at 192). Measured on GB300, 8192^3 e4m3:
    // 224 wide 491 us, 192 wide 570 us, 160 wide 654 us (4096^3 e5m2: 80 vs
    // 94 us at 192): the operand bytes per flop fall with the width and the
    // kernel is bound by operand delivery. TPGEMM_TC_BN (32..224, a multiple
    // of 32) overrides.
    const int mx_bn = (tuning().bn >= 32 && tuning().bn <= 224 && tuning().bn % 32 == 0)
                          ? tuning().bn
                          : 224;
    const int bn = swap_small ? int(Nq)
                   : mx       ? (Nq <= mx_bn ? int(((Nq + 15) / 16) * 16) : mx_bn)
                              : pick_bn(Mp, Nq, sms, pair_wanted);
    p.Mp = int(Mp);
    p.Nq = int(Nq);
    p.K = int(K);
    p.bn = bn;
    p.bp = 128;
    p.tiles_p = int((Mp + 127) / 128);
    p.tiles_q = int((Nq + bn - 1) / bn);
    p.num_tiles = p.tiles_p * p.tiles_q;
    p.bk = fp8 ? 128 : 64;  // one 128-byte swizzle row of K per stage
    p.fp8 = fp8 ? 1 : 0;
    p.k_blocks = int((K + p.bk - 1) / p.bk);
    p.p_mn = p_mn;
    p.q_mn = q_mn;
    p.beta = beta == 1.0f;
    // Tensor memory: two accumulators, each a power-of-two >= 32 columns wide
    // enough for the tile's 32-column epilogue chunks.
    int acc_cols = 32;
    while (acc_cols < 32 * ((bn + 31) / 32)) acc_cols *= 2;
    p.tmem_cols = 2 * acc_cols;
    // CTA-pair MMA: a pair of CTAs computes a 256 x bn tile with cta_group::2;
    // each loads its own 128 P rows and half of the Q tile (the MMA splits N
    // between the pair at bn / 2). A K-contiguous half must be whole 8-row
    // swizzle groups; an MN-contiguous half starts on a 16-row boundary and is
    // loaded as whole 64-row atoms (rows past the half are not read).
    const bool pair_ok = p.tiles_p >= 2 && (q_mn ? (bn % 32 == 0) : (bn % 16 == 0));
    // On by default where it applies (measured: 8192^3 1449 -> 1563 TFLOP/s,
    // 4096^3 1105 -> 1383, skinny 36.1 -> 33.5 us); TPGEMM_TC_PAIR=0 turns it off.
    p.pair = pair_ok ? 1 : 0;
    if (tuning().pair >= 0) p.pair = (tuning().pair != 0 && pair_ok) ? 1 : 0;
    const int q_rows = p.pair ? bn / 2 : bn;  // Q rows this CTA loads per stage
    p.idesc = mx ? tpg::idesc_mx_f32(format_code(dtype), p.pair ? 256 : 128, bn, 0, 0)
                 : tpg::idesc_f16_f32(format_code(dtype), p_mn, q_mn, p.pair ? 256 : 128, bn);
    p.mx = mx ? 1 : 0;
    if (mx) {
        // Scale slots: one per ring stage, in each accumulator half's columns
        // past its tile ([bn rounded to 32, 256) of the half).
        p.tmem_cols = 512;
        p.sf_q_chunks = (bn + 127) / 128;
        p.sf_q_rows = p.sf_q_chunks * tpg::mx_reps(bn);
        p.sf_cols = 4 + 4 * p.sf_q_chunks;
        p.sf_col0 = 32 * ((bn + 31) / 32);
        p.sf_spr = (256 - p.sf_col0) / p.sf_cols;
        p.sf_bytes = uint32_t(((512 * (1 + p.sf_q_rows)) + 1023) / 1024 * 1024);
        if (p.sf_spr < 1) return fail(TPGEMM_ERR_PATH, "internal: no room for scale slots");
    }
    p.p_bytes = stage_tile_bytes(128, p_mn);
    p.row_tx = dtype == TPGEMM_E2M1 ? 64u : 128u;
    p.p_tx = 128u * p.row_tx;
    p.q_bytes = stage_tile_bytes(q_rows, q_mn);
    p.tx_bytes = p.p_bytes + p.q_bytes;
    p.timeout_ns = wait_timeout_ns();
    p.test_stall = 0;  // set only by tpgemm_test_gemm_withhold_fill
    p.swap = swap;
    // L2 policies (set with the grid in choose_l2_policies); C and D stream
    // through once.
    p.l2_p = 2;
    p.l2_q = 2;
    p.l2_cd = 1;
    // Raster: runs of 8 P groups sweep all Q tiles (measured best at 8192^3:
    // fewer panel re-reads from HBM than 16 or 32, less power, higher clock).
    p.group = 8;
    if (tuning().group >= 0) p.group = std::max(1, tuning().group);
    p.snake = 1;
    if (tuning().snake >= 0) p.snake = tuning().snake != 0;
    // Every tile shares the one Q tile when all of Q fits it: spread the CTAs'
    // starting K blocks so they do not contend for the same lines of it.
    p.k_rotate = (p.tiles_q == 1 && p.tiles_p > 1) ? 1 : 0;
    // Shared memory: the deepest TMA ring with two staging tiles per lane
    // quadrant; with beta = 1, one staging tile per 32-column chunk instead
    // (all of C prefetched at tile start) when that still leaves a 4-deep ring.
    // When all of Q fits one tile (small M: P is streamed from memory once and
    // the kernel is bound by it) the ring is capped near 160 KB -- on
    // 144 x 16392 x 4104, 7 stages of 25 KB measured 1.4 us slower than 6 --
    // and the space left over stages more of C.
    auto fits = [&](int st, int eb) {
        if (mx && st > 2 * p.sf_spr) return false;
        return tpg::tc_smem_bytes(st, p.p_bytes + p.q_bytes + p.sf_bytes, eb) <=
               size_t(tpg::kTcMaxSmem);
    };
    auto deepest = [&](int eb) {
        int st = 8;
        while (st > 2 && !fits(st, eb)) --st;
        return fits(st, eb) ? st : 0;
    };
    int epi_bufs = 2;
    int stages = deepest(2);
    const int nchunks = (bn + 31) / 32;
    if (p.tiles_q == 1) {
        constexpr uint32_t kStreamRingBytes = 160 * 1024;
        stages = std::min(stages, std::max(2, int(kStreamRingBytes / (p.p_bytes + p.q_bytes))));
        if (p.beta)
            while (epi_bufs < std::min(nchunks, tpg::kTcMaxEpiBufs) && fits(stages, epi_bufs + 1))
                ++epi_bufs;
    } else if (p.beta && nchunks > 2 && nchunks <= tpg::kTcMaxEpiBufs && !mx) {
        // (Block-scaled stages hold 128 K per stage and carry scales: their
        // plans keep the deepest ring instead.)
        const int st = deepest(nchunks);
        if (st >= 4) {
            epi_bufs = nchunks;
            stages = st;
        }
    }
    // Tuning overrides (TPGEMM_TC_STAGES, TPGEMM_TC_EPI_BUFS, TPGEMM_TC_KROTATE),
    // used to sweep the ring depth, staging and K rotation on real problems.
    {
        const int v = tuning().epi_bufs;
        if (v >= 2 && v <= tpg::kTcMaxEpiBufs) {
            epi_bufs = v;
            stages = deepest(v);
        }
    }
    {
        const int v = tuning().stages;
        if (v >= 2 && v <= 8 && fits(v, epi_bufs)) stages = v;
    }
    if (tuning().krotate >= 0) p.k_rotate = tuning().krotate;
    // Clusters: a CTA pair is a cluster of two; every other plan runs one CTA
    // per cluster. No plan shares a tile between CTAs by TMA multicast.
    p.mc = p.pair ? 2 : 1;
    p.tiles_ps = (p.tiles_p + p.mc - 1) / p.mc;
    p.num_super = p.tiles_ps * p.tiles_q;
    // Work units before any tail split (set by apply_tail_split once the grid is known).
    p.full_units = p.num_super;
    p.tail_split = 1;
    p.num_units = p.num_super;
    p.idesc_tail = p.idesc;
    p.q_box_rows = p.pair ? bn / 2 : bn;
    if (stages == 0) return fail(TPGEMM_ERR_PATH, "tile does not fit in shared memory");
    p.stages = stages;
    p.producers = 1;  // set with the grid (choose_producers)
    p.epi_bufs = epi_bufs;
    p.epi_groups = 1;  // set with the grid (choose_epi_groups)
    // The epilogue stores 32-column boxes; a tile width that is not a multiple
    // of 32 is only used when it is the only tile along Q (the box overhang is
    // then past the end of the matrix and clipped by the TMA store).
    if (bn % 32 != 0 && p.tiles_q != 1)
        return fail(TPGEMM_ERR_PATH, "internal: tile width %d with %d tiles along Q", bn, p.tiles_q);
    out->kernel = Kernel::Tc;
    out->tc = p;
    out->grid = std::min(p.num_super, std::max(1, sms / p.mc)) * p.mc;
    out->max_grid = std::max(1, sms / p.mc) * p.mc;
    out->sms = sms;
    out->swap = swap;
    return TPGEMM_OK;
}

// The last wave of the persistent grid is partial when the work items do not
// divide evenly among the clusters. Its tiles are then split along Q into 2 or
// 4 narrower units (as many as still fit one wave), so the wave takes half or
// a quarter of the time. A unit stays a whole number of 32-column chunks and
// each CTA's share of it whole 8-row groups (K-contiguous Q) or 16-row steps.
// Stream-K flags: one epoch flag per epilogue warp of each CTA, sized for the
// largest grid.
constexpr int kSkMaxGrid = tpg::kTcMaxFlagSlots;
constexpr size_t kSkFlagBytes = kSkMaxGrid * tpg::kTcEpiWarps * sizeof(uint32_t);

// Balance the last, partial wave of the persistent grid. Stream-K: each
// leftover tile is split into two K halves on two clusters (when twice the
// leftover tiles fit the grid), the halves adding their accumulators into D
// with TMA reductions onto zeros written at kernel start. Measured on GB300,
// 4096^3 f16: 84.2 us against 88.5 with the tail split below (one box,
// interleaved). The tail split instead divides the leftover tiles along Q
// into 2 or 4 narrower units (as many as still fit one wave); a narrower MMA
// takes about as long per instruction, so a half-width unit takes about as
// long as a whole one (0.94 of it at 4096^3). A unit stays a whole number of
// 32-column chunks and each CTA's share of it whole 8-row groups (K-contiguous
// Q) or 16-row steps.
// *grid is the persistent grid (at most one cluster per work item); max_grid
// is every cluster the device holds at once. Stream-K runs on max_grid.
// Whether a plan may use stream-K: by default (TPGEMM_TC_SK=0 turns it off),
// always (the static flags of tpgemm_gemm_noalloc), or never.
enum class SkMode { Env, Force, Off };

bool stream_k_requested(SkMode m) {
    if (m != SkMode::Env) return m == SkMode::Force;
    return tuning().sk != 0;  // on unless TPGEMM_TC_SK=0
}

// Fewest K blocks per tile for the default stream-K plans: the first half's
// zero-fill, the flag and the reductions cost a few microseconds, which a
// short K loop would not win back. TPGEMM_TC_SK=1 and the static flags of
// tpgemm_gemm_noalloc take any split (two blocks at least).
constexpr int kSkMinKBlocks = 16;

void apply_tail_split(tpg::TcParams& p, int* grid, int max_grid, bool code1,
                      SkMode sk_mode = SkMode::Env) {
    p.sk = 0;
    p.sk_total = 0;
    p.sk_ncl = 1;
    // Block-scaled plans keep whole 128-wide units (their Q tiles start on the
    // packed scales' 128-row boundaries) and use no stream-K.
    if (p.mx) {
        p.full_units = p.num_super;
        p.tail_split = 1;
        p.num_units = p.num_super;
        p.idesc_tail = p.idesc;
        return;
    }
    const bool sk_on = stream_k_requested(sk_mode);
    {
        const int ncl = std::max(1, max_grid / p.mc);
        const int full = (p.num_super / ncl) * ncl;
        const int rem = p.num_super - full;
        const int min_kb = (sk_mode == SkMode::Env && tuning().sk < 0) ? kSkMinKBlocks : 2;
        if (sk_on && rem > 0 && 2 * rem <= ncl && max_grid <= kSkMaxGrid &&
            p.k_blocks >= min_kb) {
            *grid = ncl * p.mc;
            p.full_units = full;
            p.sk = 1;
            p.sk_total = rem * p.k_blocks;
            p.sk_ncl = 2 * rem;
            p.k_rotate = 0;
            p.tail_split = 1;
            p.num_units = p.full_units;
            p.idesc_tail = p.idesc;
            p.q_box_rows = p.pair ? p.bn / 2 : p.bn;
            return;
        }
    }
    const int ncl = std::max(1, *grid / p.mc);
    p.full_units = (p.num_super / ncl) * ncl;
    const int rem = p.num_super - p.full_units;
    int split = 1;
    const bool allowed = p.tiles_q > 1 && rem > 0;
    if (allowed) {
        for (int sp = 4; sp >= 2; sp /= 2) {
            const int w = p.bn / sp;
            const int share = p.pair ? w / 2 : w;
            if (p.bn % sp == 0 && w % 32 == 0 && share % 16 == 0 && rem * sp <= ncl) {
                split = sp;
                break;
            }
        }
    }
    if (tuning().tail == 0) split = 1;
    if (split == 1) p.full_units = p.num_super;
    p.tail_split = split;
    p.num_units = p.full_units + (p.num_super - p.full_units) * split;
    p.idesc_tail = tpg::idesc_f16_f32(code1, p.p_mn, p.q_mn, p.pair ? 256 : 128, p.bn / split);
    p.q_box_rows = p.pair ? p.bn / 2 : p.bn;
}

// P rows per tile. A single-wave plan whose tiles all share the one Q tile
// (small M, or small N in the swapped orientation) streams P from memory once
// and is bound by each streaming SM's load rate (measured on 144 x N x 4104 f16:
// 128 -> 152 SMs streaming the same bytes each took 33.9 -> 35.8 us for 19 %
// more data), so it gives each CTA fewer P rows and uses more SMs: the
// smallest bp of 64 .. 112 (steps of 16) whose tiles still fit one wave.
// TPGEMM_TC_BP (64 .. 128, a multiple of 16) overrides where it fits one wave.
void choose_p_rows(tpg::TcParams& p, int* grid, int max_grid) {
    if (p.tiles_q != 1 || p.bp != 128) return;
    const int avail = std::max(1, max_grid / p.mc);
    if (p.num_super > avail) return;
    auto supers = [&](int bp) {
        const int tiles = int((int64_t(p.Mp) + bp - 1) / bp);
        return (tiles + p.mc - 1) / p.mc;
    };
    auto fits = [&](int bp) {
        const int tiles = int((int64_t(p.Mp) + bp - 1) / bp);
        return supers(bp) <= avail && (!p.pair || tiles >= 2);
    };
    int bp = 128;
    for (int c = 64; c < 128; c += 16)
        if (fits(c)) {
            bp = c;
            break;
        }
    {
        const int v = tuning().bp;
        if (v >= 64 && v <= 128 && v % 16 == 0 && fits(v)) bp = v;
    }
    if (bp == 128) return;
    p.bp = bp;
    p.p_tx = uint32_t(bp) * p.row_tx;
    p.tx_bytes = p.p_tx + p.q_bytes;
    p.tiles_p = int((int64_t(p.Mp) + bp - 1) / bp);
    p.num_tiles = p.tiles_p * p.tiles_q;
    p.tiles_ps = supers(bp);
    p.num_super = p.tiles_ps * p.tiles_q;
    p.full_units = p.num_super;
    p.num_units = p.num_super;
    *grid = p.num_super * p.mc;
}

// Epilogue warpgroups. With at most one work unit per cluster (a single wave)
// no later tile's MMAs run under the epilogue, so both warpgroups drain it;
// with more, one group keeps up and the second only competes with the MMA and
// producer warps for issue slots and shared memory. TPGEMM_TC_EPI_GROUPS
// overrides.
void choose_epi_groups(tpg::TcParams& p, int grid) {
    const int ncl = std::max(1, grid / p.mc);
    p.epi_groups = (!p.sk && p.num_units <= ncl) ? 2 : 1;
    {
        const int v = tuning().epi_groups;
        if (v == 1 || v == 2) p.epi_groups = v;
    }
    // One-group plans: the second warpgroup's warps (TMA issuers or idle
    // until then) share the epilogue of each CTA's last segment, which no
    // later MMA hides, staging through the idle TMA ring.
    p.epi_help = (p.epi_groups == 1 && tpg::tc_epi_help_fits(p)) ? 1 : 0;
    if (tuning().epi_help == 0) p.epi_help = 0;
}

// TMA-issuing threads: warp 0, and with more than one producer warps 6, 7, 8,
// fill g going to producer g % producers. One issuing thread puts its own
// wake-up and issue latency on the path of every fill; two halve that and
// issue the first ring fill twice as fast. Measured on GB300 against one
// producer: 144 x 16392 x 4104 32.9 -> 32.7 us, 4096^3 105 -> 98.8 us, and,
// interleaved on one box with the current kernel, 8192^3 bf16 589 -> 584 us,
// e4m3 320 -> 317 us, block-scaled e4m3 499 -> 485 us (a third producer gained
// nothing at 4096^3).
// Warps 6, 7, 8 belong to the second epilogue warpgroup; when that group is
// active they issue their fills before their epilogue work, which is only
// safe when the cluster has a single work unit (with more, the MMA of a third
// unit would wait for an epilogue they have not reached).
// TPGEMM_TC_PRODUCERS (1..4) overrides within those limits.
void choose_producers(tpg::TcParams& p, int grid) {
    const int ncl = std::max(1, grid / p.mc);
    int n = std::min(2, p.stages);
    {
        const int v = tuning().producers;
        if (v >= 1 && v <= 4) n = std::min(v, p.stages);
    }
    if (p.epi_groups == 2 && (p.sk || p.num_units > ncl)) n = 1;
    p.producers = n;
    // Early start: each thread waits for the previous grid just before its
    // first global access (measured on GB300: 144 x 16392 x 4104 32.9 -> 31.9
    // us, 4096^3 96.5 -> 96.0 us, 8192^3 unchanged). TPGEMM_TC_DEP_EARLY=0
    // makes every thread wait after set-up.
    p.dep_early = 1;
    if (tuning().dep_early >= 0) p.dep_early = tuning().dep_early != 0;
}

// L2 eviction priorities of the TMA traffic. C and D are read / written once
// (evict first). Operand panels that later tiles reuse are kept (evict last):
// on 8192^3 bf16, measured on one box interleaved, 645 -> 630 us burst and
// 722 -> 702 us sustained against normal priority for all (evict first on C
// and D alone changed nothing). A single-wave plan whose tiles share the one
// Q tile streams P once: P evict first, the shared Q tile evict last (on
// 144 x 16392 x 4104, back to back: P normal 37.9 us, evict last 32.3, evict
// first 31.4). TPGEMM_TC_L2_P / _Q / _CD (0 normal, 1 evict first, 2 evict
// last) override.
void choose_l2_policies(tpg::TcParams& p, int grid) {
    const int ncl = std::max(1, grid / p.mc);
    const bool streamed_p = p.tiles_q == 1 && p.num_units <= ncl;
    p.l2_p = streamed_p ? 1 : 2;
    p.l2_q = 2;
    p.l2_cd = 1;
    auto pick = [](int v, int* dst) {
        if (v >= 0 && v <= 2) *dst = v;
    };
    pick(tuning().l2_p, &p.l2_p);
    pick(tuning().l2_q, &p.l2_q);
    pick(tuning().l2_cd, &p.l2_cd);
}

// Stream-K scratch per (device, stream): allocated on first use, kept until
// exit, flags zeroed once; launches on one stream are ordered, so each takes
// the next epoch and never sees an earlier launch's flags as its own.
struct SkWorkspace {
    void* base = nullptr;
    uint32_t epoch = 0;
};
std::mutex g_sk_mutex;
std::map<std::pair<int, cudaStream_t>, SkWorkspace> g_sk;

tpgemm_status stream_k_workspace(cudaStream_t st, uint32_t** flags, uint32_t* epoch) {
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lock(g_sk_mutex);
    SkWorkspace& w = g_sk[std::make_pair(dev, st)];
    if (!w.base) {
        void* b = nullptr;
        cudaError_t e = cudaMalloc(&b, kSkFlagBytes);
        if (e != cudaSuccess)
            return fail(TPGEMM_ERR_LAUNCH, "stream-K flag allocation: %s", cudaGetErrorString(e));
        e = cudaMemset(b, 0, kSkFlagBytes);
        if (e != cudaSuccess)
            return fail(TPGEMM_ERR_LAUNCH, "stream-K flag init: %s", cudaGetErrorString(e));
        w.base = b;
    }
    *flags = static_cast<uint32_t*>(w.base);
    *epoch = ++w.epoch;
    if (w.epoch == 0) *epoch = ++w.epoch;  // 0 is the flags' initial value
    return TPGEMM_OK;
}

// Persistent grid: no more clusters than fit the device at once (clusters are
// placed within GPCs, so CTA pairs can be fewer than SMs / 2).
// Tuning override: at most TPGEMM_TC_MAX_CLUSTERS clusters in the persistent
// grid (used to measure fewer, longer-lived CTAs).
int cluster_cap(int n) {
    if (tuning().max_clusters >= 1) return std::min(n, tuning().max_clusters);
    return n;
}

tpgemm_status fit_grid(Plan* plan) {
    tpg::TcParams& p = plan->tc;
    if (p.mc == 1) {
        const int n = cluster_cap(plan->sms);
        plan->grid = std::min(p.num_super, n);
        plan->max_grid = n;
        return TPGEMM_OK;
    }
    static std::mutex m;
    static int cache[2] = {};  // [swap] of a pair plan: 0 = unknown
    std::lock_guard<std::mutex> lock(m);
    int& n = cache[p.swap ? 1 : 0];
    if (n == 0) {
        int v = 0;
        cudaError_t e = tpg::tc_max_active_clusters(p, &v);
        if (e != cudaSuccess || v <= 0)
            return fail(TPGEMM_ERR_LAUNCH, "cluster occupancy query failed: %s",
                        cudaGetErrorString(e));
        n = v;
    }
    const int avail = cluster_cap(n);
    plan->grid = std::min(p.num_super, avail) * p.mc;
    plan->max_grid = avail * p.mc;
    return TPGEMM_OK;
}

tpgemm_status make_plan(int64_t M, int64_t N, int64_t K, bool transA, bool transB,
                        tpgemm_dtype dtype, float beta, tpgemm_path path, int sms, Plan* out) {
    if (is_f8f6f4(dtype)) {
        // fp8 runs on the tcgen05 kernel only (kind::f8f6f4).
        if (path == TPGEMM_PATH_MMA_SYNC)
            return fail(TPGEMM_ERR_PATH, "the mma.sync kernel takes f16 / bf16 only");
        if (path != TPGEMM_PATH_AUTO && path != TPGEMM_PATH_TCGEN05)
            return fail(TPGEMM_ERR_PATH, "unknown path %d", int(path));
        return plan_tc(M, N, K, transA, transB, dtype, beta, sms, out);
    }
    if (path == TPGEMM_PATH_MMA_SYNC) {
        out->kernel = Kernel::MmaSync;
        return TPGEMM_OK;
    }
    if (path == TPGEMM_PATH_AUTO) {
        // Tiny problems finish faster on the mma.sync kernel (no TMA / TMEM
        // set-up, more CTAs than 128-row tiles would give).
        const double flops = 2.0 * double(M) * double(N) * double(K);
        if (flops <= double(1 << 26)) {
            out->kernel = Kernel::MmaSync;
            return TPGEMM_OK;
        }
    } else if (path != TPGEMM_PATH_TCGEN05) {
        return fail(TPGEMM_ERR_PATH, "unknown path %d", int(path));
    }
    return plan_tc(M, N, K, transA, transB, dtype, beta, sms, out);
}

// ---------------------------------------------------------- tensor maps
tpgemm_status encode_2d(PFN_cuTensorMapEncodeTiled_v12000 enc, CUtensorMap* map, const void* base,
                        CUtensorMapDataType type, int elem_bits, uint64_t inner, uint64_t outer,
                        uint32_t box_inner, uint32_t box_outer, const char* what) {
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner * uint64_t(elem_bits) / 8};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, type, 2, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(TPGEMM_ERR_LAUNCH, "cuTensorMapEncodeTiled(%s) failed with CUresult %d", what,
                    int(r));
    return TPGEMM_OK;
}

// Packed block scales: rows of 128 32-bit words (one 512-byte chunk each),
// boxes of box_rows whole chunks, no swizzle.
tpgemm_status encode_u32_rows(PFN_cuTensorMapEncodeTiled_v12000 enc, CUtensorMap* map,
                              const void* base, uint64_t rows, uint32_t box_rows,
                              const char* what) {
    cuuint64_t dims[2] = {128, rows};
    cuuint64_t strides[1] = {512};
    cuuint32_t box[2] = {128, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void*>(base), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(TPGEMM_ERR_LAUNCH, "cuTensorMapEncodeTiled(%s) failed with CUresult %d", what,
                    int(r));
    return TPGEMM_OK;
}

// Map of a K x rows operand: K-contiguous -> dims {K, rows}, box {64, box_rows};
// MN-contiguous -> dims {rows, K}, box {64, 64}.
// fp4 is loaded with the TMA's 4-bit type that writes each 16-element group
// (8 packed bytes) into 16 bytes of shared memory, the 8 bytes of padding the
// kind::f8f6f4 MMA expects for 4-bit operands: a 128-element box fills one
// 128-byte swizzle row, as 128 fp8 elements do.
CUtensorMapDataType operand_type(tpgemm_dtype dtype) {
    return dtype == TPGEMM_E2M1   ? CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B
           : is_f8f6f4(dtype)     ? CU_TENSOR_MAP_DATA_TYPE_UINT8
           : dtype == TPGEMM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                  : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
}

// mn_box: MN-contiguous box width along MN (default: the whole 64-row atom).
// A box narrower than the 128-byte swizzle row fills the leading 16-byte
// units of each row, in the same swizzled positions as a full box (measured
// on GB300), so it is the leading part of the atom.
tpgemm_status encode_operand(PFN_cuTensorMapEncodeTiled_v12000 enc, CUtensorMap* map,
                             const void* base, tpgemm_dtype dtype, int64_t rows, int64_t K, bool mn,
                             int box_rows, const char* what, int mn_box = 0) {
    const CUtensorMapDataType t = operand_type(dtype);
    const int bits = elem_bits(dtype);
    // Elements of one 128-byte swizzle row of shared memory (fp4 unpacked).
    const uint32_t row_elems = dtype == TPGEMM_E2M1 ? 128u : uint32_t(1024 / bits);
    if (mn)
        return encode_2d(enc, map, base, t, bits, uint64_t(rows), uint64_t(K),
                         mn_box > 0 ? uint32_t(mn_box) : row_elems, 64, what);
    return encode_2d(enc, map, base, t, bits, uint64_t(K), uint64_t(rows), row_elems,
                     uint32_t(box_rows), what);
}

// Where a stream-K launch finds its scratch: a per-stream buffer the library
// allocates on first use, or the static array of tpgemm_gemm_noalloc.
enum class Scratch { Allocated, Static };

// K direction. With eight or more waves of 16-bit tiles, a cluster's second,
// fourth, ... unit walks K backwards, so each wave starts on the operand
// slices the wave before it read last, while they are still in L2: 8192^3 bf16
// DRAM reads 1.37 -> 1.18 GB and 1 % faster, interleaved on one box. fp8 and
// block-scaled 8192^3 and the 3.4 waves of 4096^3 f16 measured no gain (0 to
// 0.5 % slower), so they keep one direction.
void choose_k_order(tpg::TcParams& p, int grid) {
    const int ncl = std::max(1, grid / p.mc);
    p.k_reverse = (!p.fp8 && !p.mx && p.k_rotate == 0 && p.num_super >= 8 * ncl) ? 1 : 0;
    if (tuning().krev >= 0) p.k_reverse = tuning().krev != 0;
}

// The grid-dependent part of a tcgen05 plan: persistent grid, P rows per
// tile, tail split or stream-K, epilogue groups and producers. Pure host work.
tpgemm_status finish_tc_plan(Plan* plan, tpgemm_dtype dtype, SkMode sk_mode) {
    if (plan->kernel != Kernel::Tc) return TPGEMM_OK;
    tpgemm_status s = fit_grid(plan);
    if (s != TPGEMM_OK) return s;
    choose_p_rows(plan->tc, &plan->grid, plan->max_grid);
    apply_tail_split(plan->tc, &plan->grid, plan->max_grid, format_code(dtype), sk_mode);
    choose_epi_groups(plan->tc, plan->grid);
    choose_producers(plan->tc, plan->grid);
    choose_l2_policies(plan->tc, plan->grid);
    choose_k_order(plan->tc, plan->grid);
    return TPGEMM_OK;
}

// Bytes of the static array a stream-K plan uses: one flag per epilogue warp
// of each CTA. Plans with more CTAs than the array has rows for never fit.
size_t static_scratch_need(const Plan& plan) {
    if (plan.grid > tpg::kTcMaxFlagSlots) return ~size_t(0);
    return size_t(plan.grid) * tpg::kTcEpiWarps * sizeof(uint32_t);
}

// The calling thread's last launched plan (tpgemm_last_plan).
struct LastPlan {
    bool valid = false;
    Plan plan;
    int64_t M = 0, N = 0, K = 0;
    const char* scratch = "none";
};
thread_local LastPlan g_last;

void record_last_plan(const Plan& plan, int64_t M, int64_t N, int64_t K, const char* scratch) {
    g_last.valid = true;
    g_last.plan = plan;
    g_last.M = M;
    g_last.N = N;
    g_last.K = K;
    g_last.scratch = scratch;
}

// One line of text describing a plan (tpgemm_describe_plan, tpgemm_last_plan).
void format_plan(const Plan& plan, int64_t M, int64_t N, int64_t K, const char* scratch,
                 char* text, size_t len) {
    if (plan.kernel == Kernel::MmaSync) {
        snprintf(text, len, "path=mma_sync tile=%dx%dx32 grid=%lldx%lld warps=4 k_inst=%s",
                 tpg::kMmaTileM, tpg::kMmaTileN, (long long)((N + 63) / 64),
                 (long long)((M + 63) / 64), (K % 16) ? "m16n8k16+m16n8k8" : "m16n8k16");
        return;
    }
    const tpg::TcParams& p = plan.tc;
    snprintf(text, len,
             "path=tcgen05 orientation=%s tile=%dx%dx%d umma=%dx%dx%d kind=%s stages=%d "
             "epi_bufs=%d epi_groups=%d epi_help=%d producers=%d dep_early=%d k_rotate=%d k_reverse=%d cluster=%d pair=%d "
             "tmem=%d tiles=%dx%d grid=%d units=%d+%dx%d stream_k=%d scratch=%s p_major=%s "
             "q_major=%s l2=%d%d%d snake=%d smem=%zu sk_clusters=%d",
             plan.swap ? "swapped" : "normal", p.bp, p.bn, p.bk, p.pair ? 256 : 128, p.bn,
             p.fp8 ? 32 : 16, p.mx ? "mxf8f6f4" : (p.fp8 ? "f8f6f4" : "f16"), p.stages,
             p.epi_bufs, p.epi_groups, p.epi_help,
             p.producers, p.dep_early, p.k_rotate, p.k_reverse, p.mc, p.pair, p.tmem_cols, p.tiles_p,
             p.tiles_q, plan.grid, p.full_units, p.num_super - p.full_units, p.tail_split, p.sk,
             scratch, p.p_mn ? "mn" : "k", p.q_mn ? "mn" : "k", p.l2_p, p.l2_q, p.l2_cd, p.snake,
             tpg::tc_smem_bytes(p.stages, p.p_bytes + p.q_bytes + p.sf_bytes, p.epi_bufs),
             p.sk ? p.sk_ncl : 0);
}

void copy_text(const char* text, char* buf, int buflen) {
    if (buf && buflen > 0) {
        strncpy(buf, text, size_t(buflen) - 1);
        buf[buflen - 1] = '\0';
    }
}

// Block-scaled operands of tpgemm_gemm_mx: E8M0 scales and the caller's
// workspace for their packed form.
struct MxArgs {
    const uint8_t* SFA;
    const uint8_t* SFB;
    void* ws;
    size_t ws_bytes;
};

// Workspace of tpgemm_gemm_mx: the packed scales of A, then (256-byte aligned)
// those of B, each sized for any tile height a plan may use.
size_t mx_ws_b_offset(int64_t M, int64_t K) {
    return (tpg::mx_packed_bytes_bound(M, K) + 255) / 256 * 256;
}
size_t mx_ws_bytes(int64_t M, int64_t N, int64_t K) {
    return mx_ws_b_offset(M, K) + tpg::mx_packed_bytes_bound(N, K);
}

// Per-device epoch counter of the static scratch (all its calls share it).
std::mutex g_static_epoch_mutex;
uint32_t g_static_epoch[tpg::kMaxStaticScratchDevices] = {};

tpgemm_status run(float* D, const void* A, const void* B, const float* C, int64_t M, int64_t N,
                  int64_t K, int transA, int transB, tpgemm_dtype dtype, float beta, void* stream,
                  tpgemm_path path, Scratch scratch = Scratch::Allocated,
                  bool withhold_fill = false, const MxArgs* mx = nullptr) {
    g_detail.clear();
    tpgemm_status s = check_shape(M, N, K, dtype, beta);
    if (s != TPGEMM_OK) return s;
    s = check_pointers(D, A, B, C, M, N, K, beta, dtype);
    if (s != TPGEMM_OK) return s;
    if (mx) {
        if (!is_f8f6f4(dtype))
            return fail(TPGEMM_ERR_DTYPE,
                        "block-scaled A and B must be TPGEMM_E4M3 or TPGEMM_E5M2 (dtype %d)",
                        int(dtype));
        if (!mx->SFA) return fail(TPGEMM_ERR_NULL, "SFA is NULL");
        if (!mx->SFB) return fail(TPGEMM_ERR_NULL, "SFB is NULL");
        if (!mx->ws) return fail(TPGEMM_ERR_NULL, "workspace is NULL");
        if (reinterpret_cast<uintptr_t>(mx->ws) % 256)
            return fail(TPGEMM_ERR_ALIGN, "workspace=%p is not 256-byte aligned", mx->ws);
        const size_t need = mx_ws_bytes(M, N, K);
        if (mx->ws_bytes < need)
            return fail(TPGEMM_ERR_NULL, "workspace of %zu bytes; %zu needed", mx->ws_bytes, need);
        const int64_t kb = (K + tpg::kMxBlock - 1) / tpg::kMxBlock;
        const size_t dn = size_t(M) * size_t(N) * 4;
        if (overlaps(D, dn, mx->SFA, size_t(M) * size_t(kb)) ||
            overlaps(D, dn, mx->SFB, size_t(N) * size_t(kb)))
            return fail(TPGEMM_ERR_ALIAS, "D overlaps a scale matrix");
        const void* ops[5] = {D, A, B, mx->SFA, mx->SFB};
        const size_t lens[5] = {dn, operand_bytes(dtype, M * K), operand_bytes(dtype, K * N),
                                size_t(M) * size_t(kb), size_t(N) * size_t(kb)};
        for (int i = 0; i < 5; ++i)
            if (overlaps(mx->ws, need, ops[i], lens[i]))
                return fail(TPGEMM_ERR_ALIAS, "the workspace overlaps an operand");
        if (beta == 1.0f && overlaps(mx->ws, need, C, dn))
            return fail(TPGEMM_ERR_ALIAS, "the workspace overlaps C");
    }
    DeviceInfo dev;
    s = device_info(&dev);
    if (s != TPGEMM_OK) return s;
    if (!(dev.major == 10 && dev.minor == 3))
        return fail(TPGEMM_ERR_ARCH, "device is compute capability %d.%d; this build targets sm_103a",
                    dev.major, dev.minor);
    const bool bf16 = dtype == TPGEMM_BF16;
    Plan plan;
    if (mx) {
        s = plan_tc(M, N, K, transA != 0, transB != 0, dtype, beta, dev.sms, &plan, true);
    } else {
        s = make_plan(M, N, K, transA != 0, transB != 0, dtype, beta, path, dev.sms, &plan);
    }
    if (s != TPGEMM_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    if (plan.kernel == Kernel::MmaSync) {
        tpg::MmaSyncArgs a{D, A, B, beta == 1.0f ? C : nullptr, int(M), int(N), int(K),
                           transA != 0, transB != 0, bf16, beta == 1.0f};
        cudaError_t e = tpg::launch_mma_sync(a, st);
        if (e != cudaSuccess)
            return fail(TPGEMM_ERR_LAUNCH, "mma.sync kernel launch: %s", cudaGetErrorString(e));
        record_last_plan(plan, M, N, K, "none");
        return TPGEMM_OK;
    }

    PFN_cuTensorMapEncodeTiled_v12000 enc;
    s = get_encoder(&enc);
    if (s != TPGEMM_OK) return s;
    const tpg::TcParams& p = plan.tc;
    tpg::TcMaps maps;
    std::memset(&maps, 0, sizeof(maps));
    // In place (D == C with beta = 1): stream-K's first half zeroes its tile
    // of D at kernel start, which here would erase C before it is read, so
    // those calls take the split along N. So do calls on a stream being
    // captured into a graph: a captured launch keeps its flag epoch, and a
    // replay would find the flags already at that value (and the first
    // stream-K call on a stream allocates its flags).
    const bool in_place = beta == 1.0f && static_cast<const void*>(D) == static_cast<const void*>(C);
    cudaStreamCaptureStatus capture = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(static_cast<cudaStream_t>(stream), &capture) != cudaSuccess) {
        (void)cudaGetLastError();
        capture = cudaStreamCaptureStatusActive;  // unknown: plan as if captured
    }
    const bool capturing = capture != cudaStreamCaptureStatusNone;
    const SkMode sk_mode = (in_place || capturing)
                               ? SkMode::Off
                               : (scratch == Scratch::Static ? SkMode::Force : SkMode::Env);
    s = finish_tc_plan(&plan, dtype, sk_mode);
    if (s != TPGEMM_OK) return s;
    if (scratch == Scratch::Static && plan.tc.sk && static_scratch_need(plan) > tpg::kStaticScratchBytes) {
        // The stream-K scratch would not fit the static array: plan again
        // without stream-K. The tail split needs no scratch at all.
        s = make_plan(M, N, K, transA != 0, transB != 0, dtype, beta, path, dev.sms, &plan);
        if (s != TPGEMM_OK) return s;
        s = finish_tc_plan(&plan, dtype, SkMode::Off);
        if (s != TPGEMM_OK) return s;
    }
    plan.tc.test_stall = withhold_fill ? 1 : 0;
#ifdef TPGEMM_DEBUG
    plan.tc.debug_plant = tuning().debug_plant > 0 ? 1 : 0;
#endif
    // P / Q operands: normal P = A (rows M), Q = B^T (rows N); swapped P = B^T, Q = A.
    const void* pp = plan.swap ? B : A;
    const void* qq = plan.swap ? A : B;
    // P: K-contiguous, one box of bp rows; MN-contiguous, a 64-row atom from
    // maps.P and rows 64 .. bp - 1 from maps.Ph.
    s = encode_operand(enc, &maps.P, pp, dtype, p.Mp, K, p.p_mn, p.bp, "P operand");
    if (s != TPGEMM_OK) return s;
    if (p.p_mn && p.bp > 64) {
        s = encode_operand(enc, &maps.Ph, pp, dtype, p.Mp, K, true, 0,
                           "P operand (rows 64 .. bp of a tile)", p.bp - 64);
        if (s != TPGEMM_OK) return s;
    } else {
        maps.Ph = maps.P;
    }
    s = encode_operand(enc, &maps.Q, qq, dtype, p.Nq, K, p.q_mn, p.q_box_rows, "Q operand");
    if (s != TPGEMM_OK) return s;
    if (p.tail_split > 1) {
        s = encode_operand(enc, &maps.Qt, qq, dtype, p.Nq, K, p.q_mn, p.q_box_rows / p.tail_split,
                           "Q operand (tail units)");
        if (s != TPGEMM_OK) return s;
    }
    if (p.sk) {
        // The epoch flags of the first segments' zero-fills.
        if (scratch == Scratch::Static) {
            // No allocation: the static flag array; the plan must fit, else
            // the call is refused.
            const size_t need = static_scratch_need(plan);
            if (need > tpg::kStaticScratchBytes)
                return fail(TPGEMM_ERR_SHAPE,
                            "internal: stream-K flags for this plan need %zu bytes; the static "
                            "array holds %zu",
                            need, tpg::kStaticScratchBytes);
            void* base = nullptr;
            cudaError_t e = tpg::tc_static_scratch(&base);
            if (e != cudaSuccess)
                return fail(TPGEMM_ERR_LAUNCH, "static scratch set-up: %s", cudaGetErrorString(e));
            int dev = 0;
            cudaGetDevice(&dev);
            uint32_t epoch;
            {
                std::lock_guard<std::mutex> lock(g_static_epoch_mutex);
                epoch = ++g_static_epoch[dev];
                if (epoch == 0) epoch = ++g_static_epoch[dev];
            }
            plan.tc.sk_flags = static_cast<uint32_t*>(base);
            plan.tc.sk_epoch = epoch;
        } else {
            s = stream_k_workspace(st, &plan.tc.sk_flags, &plan.tc.sk_epoch);
            if (s != TPGEMM_OK) return s;
        }
    }
    s = encode_2d(enc, &maps.D, D, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 32, uint64_t(N), uint64_t(M), 32,
                  32, "D");
    if (s != TPGEMM_OK) return s;
    if (p.beta) {
        s = encode_2d(enc, &maps.C, C, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 32, uint64_t(N), uint64_t(M),
                      32, 32, "C");
        if (s != TPGEMM_OK) return s;
    }
    // Half-quadrant boxes (16 tensor-memory lanes = 16 P rows): 16 rows of D
    // (normal) or 16 columns (swapped), read from the same swizzled staging tile.
    maps.Dh = maps.D;
    maps.Ch = maps.C;
    if (p.bp % 32) {
        const uint32_t hx = plan.swap ? 16 : 32, hy = plan.swap ? 32 : 16;
        s = encode_2d(enc, &maps.Dh, D, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 32, uint64_t(N),
                      uint64_t(M), hx, hy, "D (half-quadrant box)");
        if (s != TPGEMM_OK) return s;
        if (p.beta) {
            s = encode_2d(enc, &maps.Ch, C, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 32, uint64_t(N),
                          uint64_t(M), hx, hy, "C (half-quadrant box)");
            if (s != TPGEMM_OK) return s;
        }
    }
    if (mx) {
        // Pack both scale matrices into the workspace (ordered before the GEMM
        // on the same stream): P's in tiles of bp rows (one chunk, rows past bp
        // padded), Q's in tiles of bn rows.
        // P's scales are A's in the normal orientation.
        uint32_t* wa = static_cast<uint32_t*>(mx->ws);
        uint32_t* wb = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(mx->ws) +
                                                   mx_ws_b_offset(M, K));
        const int rows_a = plan.swap ? p.bn : p.bp, rows_b = plan.swap ? p.bp : p.bn;
        cudaError_t e =
            tpg::launch_mx_pack_scales(mx->SFA, M, rows_a, wa, mx->SFB, N, rows_b, wb, K, st);
        if (e != cudaSuccess)
            return fail(TPGEMM_ERR_LAUNCH, "scale packing launch: %s", cudaGetErrorString(e));
        const uint32_t* sp = plan.swap ? wb : wa;
        const uint32_t* sq = plan.swap ? wa : wb;
        const uint64_t chunk_rows_p = tpg::mx_packed_bytes(p.Mp, K, p.bp) / 512;
        const uint64_t chunk_rows_q = tpg::mx_packed_bytes(p.Nq, K, p.bn) / 512;
        s = encode_u32_rows(enc, &maps.SP, sp, chunk_rows_p, 1, "P scales");
        if (s != TPGEMM_OK) return s;
        s = encode_u32_rows(enc, &maps.SQ, sq, chunk_rows_q, uint32_t(p.sf_q_rows), "Q scales");
        if (s != TPGEMM_OK) return s;
    }
    cudaError_t e = tpg::launch_tc(maps, p, plan.grid, st);
    if (e != cudaSuccess)
        return fail(TPGEMM_ERR_LAUNCH, "tcgen05 kernel launch: %s", cudaGetErrorString(e));
    record_last_plan(plan, M, N, K,
                     !p.sk ? "none" : (scratch == Scratch::Static ? "static" : "allocated"));
    return TPGEMM_OK;
}

// ------------------------------------------------------ host-buffer path
constexpr size_t kWsAlign = 256;

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Rows of the first and last row block of the host-buffer path (large M).
// 8192^3 bf16, alternating on one box: equal blocks 3.075 ms per call, edges
// of 256 rows 3.092 ms, of 512 rows 3.066 ms.
constexpr int64_t kHostEdgeRows = 512;

struct HostWsLayout {
    size_t a, b, c, d, total;  // byte offsets in the workspace, and its size
};

HostWsLayout host_ws_layout(int64_t M, int64_t N, int64_t K, bool beta, int eb) {
    HostWsLayout L;
    size_t off = 0;
    L.a = off;
    off = align_up(off + size_t(M) * size_t(K) * size_t(eb), kWsAlign);
    L.b = off;
    off = align_up(off + size_t(K) * size_t(N) * size_t(eb), kWsAlign);
    L.c = off;
    if (beta) off = align_up(off + size_t(M) * size_t(N) * 4, kWsAlign);
    L.d = off;
    off = align_up(off + size_t(M) * size_t(N) * 4, kWsAlign);
    L.total = off;
    return L;
}

// Per-device helper streams and events of the host-buffer path (created once).
struct HostPipe {
    bool ready = false;
    cudaStream_t in = nullptr, out = nullptr;
    static constexpr int kEvents = 40;
    cudaEvent_t ev[kEvents] = {};
};
HostPipe g_pipes[kMaxDevices];
std::mutex g_pipe_mutex;

tpgemm_status host_pipe(int dev, HostPipe** out) {
    HostPipe& hp = g_pipes[dev];
    if (!hp.ready) {
        if (cudaStreamCreateWithFlags(&hp.in, cudaStreamNonBlocking) != cudaSuccess ||
            cudaStreamCreateWithFlags(&hp.out, cudaStreamNonBlocking) != cudaSuccess)
            return fail(TPGEMM_ERR_LAUNCH, "cannot create the copy streams");
        for (int i = 0; i < HostPipe::kEvents; ++i)
            if (cudaEventCreateWithFlags(&hp.ev[i], cudaEventDisableTiming) != cudaSuccess)
                return fail(TPGEMM_ERR_LAUNCH, "cannot create the copy events");
        hp.ready = true;
    }
    *out = &hp;
    return TPGEMM_OK;
}

tpgemm_status run_host(float* Dh, const void* Ah, const void* Bh, const float* Ch, int64_t M,
                       int64_t N, int64_t K, int transA, int transB, tpgemm_dtype dtype,
                       float beta, void* ws, size_t ws_bytes, void* stream) {
    g_detail.clear();
    tpgemm_status s = check_shape(M, N, K, dtype, beta);
    if (s != TPGEMM_OK) return s;
    if (!Dh || !Ah || !Bh || (beta == 1.0f && !Ch))
        return fail(TPGEMM_ERR_NULL, "a host operand is NULL");
    if (!ws) return fail(TPGEMM_ERR_NULL, "workspace is NULL");
    if (reinterpret_cast<uintptr_t>(ws) % kWsAlign)
        return fail(TPGEMM_ERR_ALIGN, "workspace is not 256-byte aligned");
    if (dtype == TPGEMM_E2M1)
        return fail(TPGEMM_ERR_DTYPE, "the host-buffer path takes f16, bf16 and fp8 operands");
    const bool use_c = beta == 1.0f;
    const size_t eb = size_t(elem_bits(dtype) / 8);
    const HostWsLayout L = host_ws_layout(M, N, K, use_c, int(eb));
    if (ws_bytes < L.total)
        return fail(TPGEMM_ERR_NULL, "workspace of %zu bytes; %zu needed", ws_bytes, L.total);
    DeviceInfo dev;
    s = device_info(&dev);
    if (s != TPGEMM_OK) return s;
    int dev_id = 0;
    cudaGetDevice(&dev_id);
    uint8_t* w = static_cast<uint8_t*>(ws);
    uint8_t* dA = w + L.a;
    uint8_t* dB = w + L.b;
    float* dC = reinterpret_cast<float*>(w + L.c);
    float* dD = reinterpret_cast<float*>(w + L.d);
    const uint8_t* hA = static_cast<const uint8_t*>(Ah);
    const uint8_t* hB = static_cast<const uint8_t*>(Bh);

    // Row blocks of M, multiples of 16 (of 256 when large), about 12 of them
    // for large M: 8192^3 bf16 took 3.14 ms with 8 blocks, 3.08 with 12 and 3.12
    // with 16 (TPGEMM_HOST_BLOCKS, 1..16, overrides the count).
    int64_t blk = M;
    int want = 12;
    if (tuning().host_blocks >= 0) want = std::min(16, std::max(1, tuning().host_blocks));
    if (M >= 2048) blk = ((M / want + 255) / 256) * 256;
    else if (M >= 512) blk = ((M / 4 + 15) / 16) * 16;
    // Edge blocks (TPGEMM_HOST_EDGE rows, a multiple of 16; 0 = none): a large
    // M gets a short first block, so that D starts back across the link while
    // the inputs are still coming in, and a short last block, so that little of
    // D is left to copy out once every input is in.
    int64_t edge = M >= 2048 ? kHostEdgeRows : 0;
    if (tuning().host_edge >= 0) edge = (int64_t(tuning().host_edge) / 16) * 16;
    if (edge > 0 && M < 2 * edge + 2 * blk) edge = 0;
    int64_t starts[HostPipe::kEvents];
    int nblk = 0;
    if (edge > 0) starts[nblk++] = 0;
    for (int64_t m = edge; m < M - edge && nblk < HostPipe::kEvents; m += blk) starts[nblk++] = m;
    if (edge > 0 && nblk < HostPipe::kEvents) starts[nblk++] = M - edge;
    auto block_end = [&](int i) { return i + 1 < nblk ? starts[i + 1] : M; };

    std::lock_guard<std::mutex> lock(g_pipe_mutex);
    HostPipe* hp = nullptr;
    s = host_pipe(dev_id, &hp);
    if (s != TPGEMM_OK) return s;
    if (2 * nblk + 2 > HostPipe::kEvents) return fail(TPGEMM_ERR_LAUNCH, "too many row blocks");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaEvent_t start = hp->ev[0], done = hp->ev[1];
    auto ev_in = [&](int i) { return hp->ev[2 + 2 * i]; };
    auto ev_mm = [&](int i) { return hp->ev[3 + 2 * i]; };
    auto ck = [&](cudaError_t e, const char* what) -> tpgemm_status {
        if (e != cudaSuccess)
            return fail(TPGEMM_ERR_LAUNCH, "%s: %s", what, cudaGetErrorString(e));
        return TPGEMM_OK;
    };
#define TPG_CK(expr, what)                 \
    do {                                   \
        tpgemm_status r_ = ck((expr), what); \
        if (r_ != TPGEMM_OK) return r_;    \
    } while (0)
    TPG_CK(cudaEventRecord(start, st), "event");
    TPG_CK(cudaStreamWaitEvent(hp->in, start, 0), "stream wait");
    TPG_CK(cudaStreamWaitEvent(hp->out, start, 0), "stream wait");
    TPG_CK(cudaMemcpyAsync(dB, hB, size_t(K) * size_t(N) * eb, cudaMemcpyHostToDevice, hp->in),
           "copy of B");
    // A block i: rows [m0, m1) of the logical A, packed densely in the
    // workspace (for transA a column block of the stored [K, M] matrix).
    size_t a_off = 0;
    for (int i = 0; i < nblk; ++i) {
        const int64_t m0 = starts[i];
        const int64_t mb = block_end(i) - m0;
        uint8_t* dAi = dA + a_off;
        if (!transA) {
            TPG_CK(cudaMemcpyAsync(dAi, hA + size_t(m0) * size_t(K) * eb,
                                   size_t(mb) * size_t(K) * eb, cudaMemcpyHostToDevice, hp->in),
                   "copy of A");
        } else {
            TPG_CK(cudaMemcpy2DAsync(dAi, size_t(mb) * eb, hA + size_t(m0) * eb, size_t(M) * eb,
                                     size_t(mb) * eb, size_t(K), cudaMemcpyHostToDevice, hp->in),
                   "copy of A");
        }
        if (use_c)
            TPG_CK(cudaMemcpyAsync(dC + size_t(m0) * size_t(N), Ch + size_t(m0) * size_t(N),
                                   size_t(mb) * size_t(N) * 4, cudaMemcpyHostToDevice, hp->in),
                   "copy of C");
        TPG_CK(cudaEventRecord(ev_in(i), hp->in), "event");
        TPG_CK(cudaStreamWaitEvent(st, ev_in(i), 0), "stream wait");
        s = run(dD + size_t(m0) * size_t(N), dAi, dB, use_c ? dC + size_t(m0) * size_t(N) : nullptr,
                mb, N, K, transA, transB, dtype, beta, st, TPGEMM_PATH_AUTO);
        if (s != TPGEMM_OK) return s;
        TPG_CK(cudaEventRecord(ev_mm(i), st), "event");
        TPG_CK(cudaStreamWaitEvent(hp->out, ev_mm(i), 0), "stream wait");
        TPG_CK(cudaMemcpyAsync(Dh + size_t(m0) * size_t(N), dD + size_t(m0) * size_t(N),
                               size_t(mb) * size_t(N) * 4, cudaMemcpyDeviceToHost, hp->out),
               "copy of D");
        a_off += size_t(mb) * size_t(K) * eb;
    }
    TPG_CK(cudaEventRecord(done, hp->out), "event");
    TPG_CK(cudaStreamWaitEvent(st, done, 0), "stream wait");
#undef TPG_CK
    return TPGEMM_OK;
}

}  // namespace

namespace tpg {
void set_error_detail(const char* text) { g_detail = text ? text : ""; }

uint64_t wait_timeout_ns() {
    long long ms = tuning().wait_ms;
    if (ms <= 0) ms = 2000;
    return uint64_t(ms) * 1000000ull;
}
}  // namespace tpg

extern "C" {

size_t tpgemm_gemm_host_workspace_bytes(int64_t M, int64_t N, int64_t K, tpgemm_dtype dtype,
                                        float beta) {
    const std::string keep = g_detail;
    const bool ok = check_shape(M, N, K, dtype, beta) == TPGEMM_OK;
    g_detail = keep;
    if (!ok) return 0;
    if (dtype == TPGEMM_E2M1) return 0;
    return host_ws_layout(M, N, K, beta == 1.0f, elem_bits(dtype) / 8).total;
}

tpgemm_status tpgemm_gemm_host(float* D_host, const void* A_host, const void* B_host,
                               const float* C_host, int64_t M, int64_t N, int64_t K, int transA,
                               int transB, tpgemm_dtype dtype, float beta, void* workspace,
                               size_t workspace_bytes, void* stream) {
    return run_host(D_host, A_host, B_host, C_host, M, N, K, transA, transB, dtype, beta,
                    workspace, workspace_bytes, stream);
}

tpgemm_status tpgemm_gemm(float* D, const void* A, const void* B, const float* C, int64_t M,
                          int64_t N, int64_t K, int transA, int transB, tpgemm_dtype dtype,
                          float beta, void* stream) {
    return run(D, A, B, C, M, N, K, transA, transB, dtype, beta, stream, TPGEMM_PATH_AUTO);
}

tpgemm_status tpgemm_gemm_path(float* D, const void* A, const void* B, const float* C, int64_t M,
                               int64_t N, int64_t K, int transA, int transB, tpgemm_dtype dtype,
                               float beta, void* stream, tpgemm_path path) {
    return run(D, A, B, C, M, N, K, transA, transB, dtype, beta, stream, path);
}

// The stream-K variant for callers that must not allocate device memory: its
// scratch is the static array in tc_gemm.cu, never cudaMalloc.
tpgemm_status tpgemm_gemm_noalloc(float* D, const void* A, const void* B, const float* C,
                                  int64_t M, int64_t N, int64_t K, int transA, int transB,
                                  tpgemm_dtype dtype, float beta, void* stream) {
    return run(D, A, B, C, M, N, K, transA, transB, dtype, beta, stream, TPGEMM_PATH_AUTO,
               Scratch::Static);
}

size_t tpgemm_gemm_mx_workspace_bytes(int64_t M, int64_t N, int64_t K) {
    if (M <= 0 || N <= 0 || K <= 0 || M >= (int64_t(1) << 30) || N >= (int64_t(1) << 30) ||
        K >= (int64_t(1) << 30))
        return 0;
    return mx_ws_bytes(M, N, K);
}

tpgemm_status tpgemm_gemm_mx(float* D, const void* A, const void* B, const float* C,
                             const uint8_t* SFA, const uint8_t* SFB, int64_t M, int64_t N,
                             int64_t K, tpgemm_dtype dtype, float beta, void* workspace,
                             size_t workspace_bytes, void* stream) {
    const MxArgs mx{SFA, SFB, workspace, workspace_bytes};
    return run(D, A, B, C, M, N, K, 0, 1, dtype, beta, stream, TPGEMM_PATH_TCGEN05,
               Scratch::Allocated, false, &mx);
}

tpgemm_status tpgemm_test_gemm_withhold_fill(float* D, const void* A, const void* B,
                                             const float* C, int64_t M, int64_t N, int64_t K,
                                             int transA, int transB, tpgemm_dtype dtype, float beta,
                                             void* stream) {
    return run(D, A, B, C, M, N, K, transA, transB, dtype, beta, stream, TPGEMM_PATH_TCGEN05,
               Scratch::Allocated, true);
}

void tpgemm_reload_tuning(void) {
    std::lock_guard<std::mutex> lock(g_tuning_mutex);
    g_tuning.store(new Tuning(read_tuning()), std::memory_order_release);
}

const char* tpgemm_status_string(tpgemm_status s) {
    switch (s) {
        case TPGEMM_OK: return "ok";
        case TPGEMM_ERR_SHAPE: return "invalid shape";
        case TPGEMM_ERR_DTYPE: return "unsupported dtype";
        case TPGEMM_ERR_BETA: return "unsupported beta";
        case TPGEMM_ERR_NULL: return "null pointer";
        case TPGEMM_ERR_ALIGN: return "misaligned pointer";
        case TPGEMM_ERR_ALIAS: return "overlapping operands";
        case TPGEMM_ERR_ARCH: return "unsupported device";
        case TPGEMM_ERR_LAUNCH: return "launch failed";
        case TPGEMM_ERR_TIMEOUT: return "device wait timed out";
        case TPGEMM_ERR_PATH: return "kernel path cannot run this problem";
        case TPGEMM_ERR_BOUNDS: return "debug bounds check failed";
    }
    return "unknown status";
}

const char* tpgemm_last_error_detail(void) { return g_detail.c_str(); }

tpgemm_status tpgemm_last_device_error(void) {
    g_detail.clear();
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess)
        return fail(TPGEMM_ERR_LAUNCH, "device synchronize: %s", cudaGetErrorString(e));
    int st = 0, st_cp = 0, site = 0;
    e = tpg::tc_read_and_clear_device_status(&st, &site);
    if (e == cudaSuccess) e = tpg::cp_read_and_clear_device_status(&st_cp);
    if (e != cudaSuccess)
        return fail(TPGEMM_ERR_LAUNCH, "reading device status: %s", cudaGetErrorString(e));
    if (st == tpg::kStatusTimeout)
        return fail(TPGEMM_ERR_TIMEOUT, "a tcgen05 kernel wait exceeded its bound");
    if (st == tpg::kStatusBounds) {
        static const char* kSites[] = {"?", "epilogue tensor-memory load", "MMA accumulator",
                                       "block-scale slot", "TMA store coordinate",
                                       "TMA load coordinate", "stream-K flag index",
                                       "helper staging"};
        return fail(TPGEMM_ERR_BOUNDS,
                    "a debug bounds check failed at site %d (%s); the access was skipped", site,
                    kSites[site >= 0 && site <= 7 ? site : 0]);
    }
    if (st_cp == tpg::kStatusTimeout)
        return fail(TPGEMM_ERR_TIMEOUT, "a tensor-memory copy kernel wait exceeded its bound");
    return TPGEMM_OK;
}

tpgemm_status tpgemm_describe_plan(int64_t M, int64_t N, int64_t K, int transA, int transB,
                                   tpgemm_dtype dtype, float beta, tpgemm_path path, char* buf,
                                   int buflen) {
    g_detail.clear();
    tpgemm_status s = check_shape(M, N, K, dtype, beta);
    if (s != TPGEMM_OK) return s;
    int sms = 152;  // GB300; replaced by the live count when a device is present
    int dev = 0;
    int v = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0)
        sms = v;
    else
        cudaGetLastError();
    Plan plan;
    s = make_plan(M, N, K, transA != 0, transB != 0, dtype, beta, path, sms, &plan);
    if (s != TPGEMM_OK) return s;
    if (plan.kernel == Kernel::Tc) {
        // As tpgemm_gemm plans it, except that the grid is one CTA (pair) per
        // SM without the device's cluster-occupancy query (the cluster cap
        // override still applies).
        const int avail = cluster_cap(std::max(1, sms / plan.tc.mc));
        plan.grid = std::min(plan.tc.num_super, avail) * plan.tc.mc;
        plan.max_grid = avail * plan.tc.mc;
        choose_p_rows(plan.tc, &plan.grid, plan.max_grid);
        apply_tail_split(plan.tc, &plan.grid, plan.max_grid, format_code(dtype));
        choose_epi_groups(plan.tc, plan.grid);
        choose_producers(plan.tc, plan.grid);
        choose_l2_policies(plan.tc, plan.grid);
        choose_k_order(plan.tc, plan.grid);
    }
    char text[640];
    format_plan(plan, M, N, K, plan.tc.sk ? "allocated" : "none", text, sizeof(text));
    copy_text(text, buf, buflen);
    return TPGEMM_OK;
}

tpgemm_status tpgemm_last_plan(char* buf, int buflen) {
    if (!g_last.valid) {
        copy_text("", buf, buflen);
        return fail(TPGEMM_ERR_NULL, "no GEMM has been enqueued on this thread");
    }
    char text[640];
    format_plan(g_last.plan, g_last.M, g_last.N, g_last.K, g_last.scratch, text, sizeof(text));
    copy_text(text, buf, buflen);
    return TPGEMM_OK;
}

uint64_t tpgemm_encode_smem_desc(uint32_t start_addr, uint32_t lbo_bytes, uint32_t sbo_bytes,
                                 tpgemm_cp_swizzle swizzle) {
    uint32_t layout = tpg::kDescLayoutNone;
    switch (swizzle) {
        case TPGEMM_CP_SWIZZLE_32B: layout = tpg::kDescLayoutSw32; break;
        case TPGEMM_CP_SWIZZLE_64B: layout = tpg::kDescLayoutSw64; break;
        case TPGEMM_CP_SWIZZLE_128B: layout = tpg::kDescLayoutSw128; break;
        default: break;
    }
    return tpg::smem_desc_with_addr(tpg::smem_desc_template(lbo_bytes, sbo_bytes, layout),
                                    start_addr);
}

uint32_t tpgemm_encode_idesc_mx(tpgemm_dtype dtype, int m, int n, int a_sf_id, int b_sf_id) {
    if (!is_f8f6f4(dtype)) return 0;
    return tpg::idesc_mx_f32(format_code(dtype), m, n, uint32_t(a_sf_id), uint32_t(b_sf_id));
}

uint32_t tpgemm_encode_idesc(tpgemm_dtype dtype, int a_mn_major, int b_mn_major, int m, int n) {
    if (dtype != TPGEMM_F16 && dtype != TPGEMM_BF16 && !is_f8f6f4(dtype)) return 0;
    return tpg::idesc_f16_f32(format_code(dtype), a_mn_major != 0, b_mn_major != 0, m, n);
}

const char* tpgemm_version(void) {
#ifdef TPGEMM_DEBUG
    return "0.2.0-debug";
#else
    return "0.2.0";
#endif
}

}  // extern "C"
