// tcgen05 GEMM for sm_103a:  X = P . Q^T (+ C), f16/bf16 (or e4m3/e5m2) in, f32
// accumulate and out.
//
// Persistent, warp-specialised CTA of 10 warps, one CTA per SM (or per SM of
// a CTA pair); a tile has bp <= 128 P rows, one per tensor-memory lane:
//   warp 0      TMA producer: one thread fills a ring of shared-memory stages
//               with 128-byte-swizzled P and Q tiles (cp.async.bulk.tensor);
//               with the plan's producers > 1, lane 0 of warps 6, 7, 8 issues
//               every producers-th fill as well.
//   warp 1      owns tensor memory (tcgen05.alloc / dealloc, whole warp) and
//               one thread issues tcgen05.mma for every 16-deep K step into a
//               double-buffered accumulator, committing stage releases and
//               "accumulator full" to mbarriers (tcgen05.commit).
//   warps 2..9  one or two epilogue warpgroups (the plan's epi_groups; the
//               second sits idle when 1): tcgen05.ld 32x32b of the warp's
//               32-lane quadrant (with two groups, warps w and w + 4 share
//               one and take alternate 32-column chunks), + beta.C (TMA-loaded
//               into a swizzled staging tile), and a TMA store of D from the
//               same staging tile.
//
// This follows the single-thread issue, commit-to-mbarrier and
// alloc / relinquish / dealloc protocol of the tcgen05 copy page ("TVM
// Blackwell tcgen05.cp 全解析", section 演示程序), the encode-once descriptor
// with a patched 14-bit start address (same page, 调度算法四步 第3步/第4步), the
// warpgroup .32x32b tensor-memory load of the tcgen05_ldst page (Algorithm,
// Generated CUDA), and the gemm semantics of the synchronous gemm page
// (语义定义, 二: D = A.B + beta.C, beta in {0,1}). Every mbarrier wait is bounded
// in time; on expiry the kernel records a status word, stops every role, waits
// for its own copies and MMAs in flight, frees tensor memory and returns.
#include <mutex>
#include <type_traits>

#include "ptx.cuh"
#include "tpgemm_internal.h"

namespace tpg {

__device__ int g_tc_status;  // 0 = ok, kStatusTimeout after an expired wait
__device__ int g_tc_bounds_site;  // debug builds: the site of the last failed bounds check

// Sites of the debug bounds checks (reported with TPGEMM_ERR_BOUNDS).
enum BoundsSite : int {
    kSiteEpilogueLoad = 1,   // a tcgen05.ld column past the accumulator's buffer
    kSiteMmaAccumulator = 2, // an accumulator buffer past the tensor-memory allocation
    kSiteScaleSlot = 3,      // a block-scale slot past the allocation
    kSiteStore = 4,          // a TMA store coordinate negative or not 16-byte aligned
    kSiteLoadC = 5,          // a TMA load coordinate of C or a partial tile not aligned
    kSiteFlag = 6,           // a stream-K flag index past the flag area
    kSiteHelperStaging = 7,  // a helper warp's chunks do not fit its share of the TMA ring
};

// Debug builds (-DTPGEMM_DEBUG): a computed tensor-memory column, TMA
// coordinate or stream-K flag index outside its range records kStatusBounds
// and the site (read by tpgemm_last_device_error) and the caller skips the
// access: nothing traps. Release builds compile every check away.
__device__ __forceinline__ bool in_bounds(bool ok, int site) {
#ifdef TPGEMM_DEBUG
    if (!ok) {
        atomicExch(&g_tc_status, kStatusBounds);
        atomicExch(&g_tc_bounds_site, site);
    }
    return ok;
#else
    (void)ok;
    (void)site;
    return true;
#endif
}

// Stream-K flags of tpgemm_gemm_noalloc (one epoch flag per epilogue warp of
// each CTA). Every GPU that loads the library holds it until exit; all calls
// of that entry point on a device share it.
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

namespace {

constexpr int kBK = 64;            // 16-bit K elements per stage: one 128-byte swizzle row
constexpr int kUmmaK = 16;         // 16-bit K per tcgen05.mma (kind::f16); 32 for fp8
constexpr int kEpiWarps = kTcEpiWarps;  // two per lane quadrant
constexpr int kEpiQuads = 4;
constexpr int kEpiBufFloats = 32 * 32;  // one 32 x 32 f32 staging tile (4 KB)
constexpr int kAtomBytes = 8192;   // MN-major atom: 64 K rows x 128 bytes

struct Smem {
    uint8_t* stages;
    float* epi;            // [4 quadrants][epi_bufs][32*32]
    uint64_t* full;        // [stages]
    uint64_t* empty;       // [stages]
    uint64_t* acc_full;    // [2]
    uint64_t* acc_empty;   // [2]
    uint64_t* cbar;        // [4 quadrants][kTcMaxEpiBufs]
    uint64_t* drain;       // [1]
    uint64_t* last_full;   // [1] the CTA's last accumulator is complete (epi_help)
    uint64_t* hbar;        // [4 quadrants] C fills of the last segment's helper warps
    uint32_t* tmem_base;
    volatile int* abort;
};

__device__ __forceinline__ Smem carve(uint8_t* raw, const TcParams& p) {
    Smem s;
    uintptr_t a = (reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023);
    uint8_t* b = reinterpret_cast<uint8_t*>(a);
    s.stages = b;
    b += size_t(p.stages) * (p.p_bytes + p.q_bytes + p.sf_bytes);
    s.epi = reinterpret_cast<float*>(b);
    b += size_t(kEpiQuads) * p.epi_bufs * kEpiBufFloats * sizeof(float);
    uint64_t* bars = reinterpret_cast<uint64_t*>(b);
    s.full = bars;
    s.empty = bars + p.stages;
    s.acc_full = bars + 2 * p.stages;
    s.acc_empty = s.acc_full + 2;
    s.cbar = s.acc_empty + 2;
    s.drain = s.cbar + kTcMaxEpiBufs * kEpiQuads;
    s.last_full = s.drain + 1;
    s.hbar = s.last_full + 1;
    s.tmem_base = reinterpret_cast<uint32_t*>(s.hbar + kEpiQuads);
    s.abort = reinterpret_cast<volatile int*>(s.tmem_base + 1);
    return s;
}

// An epilogue warp's share of its quadrant's staging tiles: active epilogue
// warp ew (0 .. 4 epi_groups - 1) reads lane quadrant (ew + 2) % 4 and, of the
// quadrant's 32-column chunks, those with c % epi_groups == ew / 4. The
// quadrant's epi_bufs staging tiles (and their C-fill barriers) are split
// between its active warps, the first ones taking any remainder.
struct EpiShare {
    int g;          // this warp's group: it takes chunks c = groups * j + g
    int nbw;        // staging tiles of this warp (>= 1)
    float* bufs;    // its first staging tile
    uint64_t* cb;   // its first C-fill barrier
};

__device__ __forceinline__ EpiShare epi_share(const Smem& s, const TcParams& p, int ew) {
    const int qs = ew & 3;
    const int g = ew >> 2;
    const int base = p.epi_bufs / p.epi_groups;
    const int extra = p.epi_bufs % p.epi_groups;
    const int first = g * base + min(g, extra);
    return {g, base + (g < extra ? 1 : 0),
            s.epi + (size_t(qs) * p.epi_bufs + first) * kEpiBufFloats,
            s.cbar + kTcMaxEpiBufs * qs + first};
}

// Bounded wait on one mbarrier phase. False if the bound expired or (unless
// draining) another role already gave up. A drain wait ignores the abort flag:
// it is how a role lets its own copies or MMAs in flight finish before exit.
__device__ __forceinline__ bool wait_phase(uint64_t* bar, uint32_t parity, volatile int* abort,
                                           uint64_t timeout_ns, bool drain = false) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (!drain && *abort) return false;
        if (globaltimer_ns() - t0 > timeout_ns) {
            *abort = 1;
            atomicExch(&g_tc_status, kStatusTimeout);
            return false;
        }
    }
}

// Work item T of a cluster -> (group of mc P tiles, Q tile); runs of `group`
// P groups sweep all Q tiles so one wave of clusters shares a few P and Q
// panels in L2. With p.snake, odd runs sweep Q backwards, so a run starts on
// the Q panels the previous run used last (still in L2). The CTA of cluster
// rank r then owns P tile tps * mc + r.
__device__ __forceinline__ void tile_coords(int T, const TcParams& p, int& tps, int& tq) {
    const int per_group = p.group * p.tiles_q;
    const int g = T / per_group;
    const int first = g * p.group;
    const int gsz = min(p.tiles_ps - first, p.group);
    const int r = T - g * per_group;
    tps = first + r % gsz;
    tq = r / gsz;
    if (p.snake && (g & 1)) tq = p.tiles_q - 1 - tq;
}

// First K block of tile t. With rotation, groups of k_rotate consecutive tiles
// start at evenly spread blocks and wrap around, so CTAs that share an operand
// tile (every CTA, when all of M fits one tile) do not all read the same K
// slice of it at the same time.
__device__ __forceinline__ int first_k_block(int t, const TcParams& p) {
    if (!p.k_rotate) return 0;
    const int g = t / p.k_rotate;
    const int groups = (p.num_super + p.k_rotate - 1) / p.k_rotate;
    return int((int64_t(g) * p.k_blocks) / groups) % p.k_blocks;
}

// Work unit U -> work item T, offset of its Q columns inside the tile, width.
struct Unit {
    int T, q_off, width;
};

__device__ __forceinline__ Unit unit_of(int U, const TcParams& p) {
    if (U < p.full_units) return {U, 0, p.bn};
    const int r = U - p.full_units;
    const int w = p.bn / p.tail_split;
    return {p.full_units + r / p.tail_split, (r % p.tail_split) * w, w};
}

// One cluster's piece of work: work item T (columns q_off .. q_off + width of
// its Q tile) over K blocks [kb0, kb1). Whole tiles have owner = 1 and
// has_next = 0. Stream-K segments: owner = the segment holds K block 0 (it
// writes D); has_next = a later segment of the same tile exists, in the next
// cluster, whose partial this segment adds. rev: the producer walks the K
// blocks backwards.
struct Seg {
    int T, q_off, width, kb0, kb1, owner, has_next, rev;
};

// First stream-K K block of cluster c: the first p.sk_ncl clusters share them
// evenly; the others get none.
__device__ __forceinline__ int sk_begin(int c, const TcParams& p) {
    return c >= p.sk_ncl ? p.sk_total : int((int64_t(p.sk_total) * c) / p.sk_ncl);
}

// This cluster's segments in order: its whole work units first (U = cid,
// cid + ncl, ...), then its contiguous share of the stream-K K blocks.
struct SegIter {
    int U, u, ub, odd;
    __device__ __forceinline__ SegIter(int cid, int ncl, const TcParams& p)
        : U(cid), u(p.sk ? sk_begin(cid, p) : 0), ub(p.sk ? sk_begin(cid + 1, p) : 0), odd(0) {}
    __device__ __forceinline__ bool next(int ncl, const TcParams& p, Seg& s) {
        if (U < p.num_units) {
            const Unit un = unit_of(U, p);
            s = {un.T, un.q_off, un.width, 0, p.k_blocks, 1, 0, odd & p.k_reverse};
            U += ncl;
            odd ^= 1;
            return true;
        }
        if (u < ub) {
            const int t = u / p.k_blocks;
            const int k0 = u - t * p.k_blocks;
            const int k1 = min(p.k_blocks, k0 + (ub - u));
            s = {p.full_units + t, 0, p.bn, k0, k1, k0 == 0, k1 < p.k_blocks, 0};
            u += k1 - k0;
            return true;
        }
        return false;
    }
    // Whether a later call of next() would return a segment.
    __device__ __forceinline__ bool more(const TcParams& p) const {
        return U < p.num_units || u < ub;
    }
};

// The cluster whose stream-K share holds K block 0 of leftover tile t (the
// tile's first segment).
__device__ __forceinline__ int sk_owner_cluster(int t, const TcParams& p) {
    const int u0 = t * p.k_blocks;
    int c = int((int64_t(u0) * p.sk_ncl) / max(1, p.sk_total));
    while (c + 1 < p.sk_ncl && sk_begin(c + 1, p) <= u0) ++c;
    while (c > 0 && sk_begin(c, p) > u0) --c;
    return c;
}

// Bounded wait for a stream-K flag to reach this launch's epoch.
__device__ __forceinline__ bool wait_flag(const uint32_t* f, uint32_t v, volatile int* abort,
                                          uint64_t timeout_ns) {
    if (ld_acquire_gpu(f) == v) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (ld_acquire_gpu(f) == v) return true;
        if (*abort) return false;
        if (globaltimer_ns() - t0 > timeout_ns) {
            *abort = 1;
            atomicExch(&g_tc_status, kStatusTimeout);
            return false;
        }
    }
}

template <bool SWAP, bool PAIR, bool EARLY, bool MX>
__global__ void __launch_bounds__(kTcThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap mapP, const __grid_constant__ CUtensorMap mapQ,
                   const __grid_constant__ CUtensorMap mapC, const __grid_constant__ CUtensorMap mapD,
                   const __grid_constant__ CUtensorMap mapQt,
                   const __grid_constant__ CUtensorMap mapPh, const __grid_constant__ CUtensorMap mapCh,
                   const __grid_constant__ CUtensorMap mapDh, const __grid_constant__ CUtensorMap mapSP,
                   const __grid_constant__ CUtensorMap mapSQ, const TcParams p) {
    extern __shared__ uint8_t smem_raw[];
    const Smem s = carve(smem_raw, p);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // A CTA pair is a cluster of two; otherwise every CTA is its own cluster.
    // Rank within the cluster, which cluster, and how many clusters the
    // persistent grid has.
    constexpr int MC = PAIR ? 2 : 1;
    const int rank = PAIR ? int(cluster_ctarank()) : 0;
    const int cid = blockIdx.x / MC;
    const int ncl = gridDim.x / MC;
    constexpr uint16_t pair_mask = 3;
    constexpr int CG = PAIR ? 2 : 1;
    // Accumulator buffer b starts at column b * acc_stride.
    const int acc_stride = p.tmem_cols / 2;

    // ---------------------------------------------------------------- set-up
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&mapP);
        if (p.p_mn) prefetch_tensormap(&mapPh);
        prefetch_tensormap(&mapQ);
        if (p.tail_split > 1) prefetch_tensormap(&mapQt);
        if (MX) {
            prefetch_tensormap(&mapSP);
            prefetch_tensormap(&mapSQ);
        }
        if (p.beta) prefetch_tensormap(&mapC);
        prefetch_tensormap(&mapD);
        if (p.bp % 32) {
            if (p.beta) prefetch_tensormap(&mapCh);
            prefetch_tensormap(&mapDh);
        }
        for (int i = 0; i < p.stages; ++i) {
            mbar_init(&s.full[i], 1);
            // Freed by one commit of the MMA thread (in pair mode the leader's,
            // arriving on the barriers of both CTAs).
            mbar_init(&s.empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s.acc_full[i], 1);
            // Pair mode: the leader's accumulator barrier collects the
            // epilogue warps of both CTAs.
            mbar_init(&s.acc_empty[i], (PAIR ? 2 : 1) * kEpiQuads * p.epi_groups);
        }
        for (int i = 0; i < kTcMaxEpiBufs * kEpiQuads; ++i) mbar_init(&s.cbar[i], 1);
        mbar_init(s.drain, 1);
        mbar_init(s.last_full, 1);
        for (int i = 0; i < kEpiQuads; ++i) mbar_init(&s.hbar[i], 1);
        *s.abort = 0;
        fence_mbarrier_init();
    }
    if (warp == 1) {
        tmem_alloc<CG>(s.tmem_base, uint32_t(p.tmem_cols));
        tmem_relinquish_alloc_permit<CG>();
    }
    tc_fence_before_sync();
    // In a pair, no CTA may complete bytes on or arrive at a peer's barrier
    // before the peer's barriers exist: the set-up sync spans the pair.
    if constexpr (PAIR)
        cluster_sync();
    else
        __syncthreads();
    tc_fence_after_sync();
    // Launched with a programmatic dependency, this grid starts while the
    // previous one drains; griddepcontrol.wait then holds each thread that
    // calls it until that grid has finished and its writes are visible. With
    // EARLY (p.dep_early), only the threads that touch global memory wait, each just
    // before its first access: a producer before its first K loop, an
    // epilogue warp before its first C load or D store. Until then the
    // producers run their first work unit's bookkeeping, whose instruction
    // fetch otherwise costs about 1 us after the wait on a 144 x 16392 x 4104
    // step (measured on GB300); the MMA warp (shared and tensor memory only)
    // never waits. Otherwise every thread waits here.
    grid_launch_dependents();
    if constexpr (!EARLY) grid_dependency_wait();
    const uint32_t tmem = *s.tmem_base;
    const uint64_t tmo = p.timeout_ns;
    // In-flight bookkeeping kept to teardown, where an aborted CTA drains it.
    uint32_t issued_parity = 0;  // producer: bit i = parity of the last fill of stage i
    uint32_t issued_any = 0;     // producer: bit i = stage i was ever filled
    uint32_t cphase = 0;         // epilogue: bit i = parity of the next C fill of buffer i
    uint32_t cpend = 0;          // epilogue: bit i = a C fill into staging buffer i in flight
    bool hpend = false;          // helper warp: its C fill of the last segment is in flight

    // ---------------------------------------------------------- TMA producers
    // Lane 0 of warp 0 and, with p.producers > 1, of warps 6, 7, 8 (the second
    // epilogue warpgroup, which has no epilogue work before an accumulator is
    // ready, and none at all in one-group plans). Producer r issues the fills
    // of ring iterations g = r, r + P, r + 2P, ..., so one thread's wake-up and
    // issue latency sits on the path of only every P-th fill. With P no larger
    // than the ring, a producer waiting on a stage's empty barrier is never
    // more than one phase behind it.
    const int prod_r = warp == 0 ? 0 : ((warp >= 6 && warp - 5 < p.producers) ? warp - 5 : -1);
    // The producer's body is inline (not a lambda): kernel parameters are then
    // read from parameter space, not through a generic reference, which the
    // TMA issue's memory clobbers would reload on every fill.
    if (prod_r >= 0) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            // Whose fill the current ring iteration is: producer `turn`, cycling
            // through 0 .. producers - 1 over every fill of the CTA.
            int turn = 0;
            const int nprod = p.producers;
            const uint64_t pol_p = l2_policy(p.l2_p);
            const uint64_t pol_q = l2_policy(p.l2_q);
            bool ok = true;
            SegIter iter(cid, ncl, p);
            Seg u;
            bool first_seg = true;
            for (; ok && iter.next(ncl, p, u); first_seg = false) {
                int tps, tq;
                tile_coords(u.T, p, tps, tq);
                const int p0 = (tps * MC + rank) * p.bp;
                const int q0 = tq * p.bn + u.q_off;
                // Q rows this CTA loads per stage, and the bytes they fill.
                const int q_rows = PAIR ? u.width / 2 : u.width;
                const int q_atoms = (q_rows + 63) / 64;
                // K-contiguous Q: one box per stage, from the map whose box
                // height is this unit's share (whole tile or tail unit).
                const CUtensorMap* mq = u.width == p.bn ? &mapQ : &mapQt;
                const uint32_t tx = p.p_tx +
                                    (p.q_mn ? uint32_t(q_atoms) * kAtomBytes
                                            : uint32_t(q_rows) * p.row_tx) +
                                    (MX ? 512u * uint32_t(1 + p.sf_q_rows) : 0u);
                const int nk = u.kb1 - u.kb0;
                int kb = nk == p.k_blocks ? first_k_block(u.T, p) : u.kb0;
                // Backwards: the same blocks in the opposite order, ending on
                // the block a forward walk starts on.
                if (u.rev) kb = (kb == 0 ? p.k_blocks : kb) - 1;
                if constexpr (EARLY) {
                    if (first_seg) {
                        // Before waiting for the previous grid, ask L2 for the
                        // operand boxes of this producer's first ring of fills.
                        // L2 is where the previous grid's writes land, so a line
                        // prefetched early is never stale; the fills themselves
                        // still come after the wait.
                        for (int i = prod_r; i < nk && i < p.stages; i += nprod) {
                            const int k0 = ((kb + i) % p.k_blocks) * p.bk;
                            if (p.p_mn) {
                                tma_prefetch_2d(&mapP, p0, k0);
                                if (p.bp > 64) tma_prefetch_2d(&mapPh, p0 + 64, k0);
                            } else {
                                tma_prefetch_2d(&mapP, k0, p0);
                            }
                            const int qh = q0 + (PAIR ? rank * q_rows : 0);
                            if (p.q_mn) {
                                for (int a = 0; a < q_atoms; ++a)
                                    tma_prefetch_2d(&mapQ, qh + 64 * a, k0);
                            } else {
                                tma_prefetch_2d(mq, k0, qh);
                            }
                        }
                        grid_dependency_wait();
                    }
                }
                for (int i = 0; i < nk;
                     ++i, turn = (turn + 1 == nprod) ? 0 : turn + 1,
                     kb = u.rev ? (kb == 0 ? p.k_blocks : kb) - 1
                                : (kb + 1 == p.k_blocks ? 0 : kb + 1)) {
                    if (turn != prod_r) {  // another producer's fill
                        if (++stage == p.stages) {
                            stage = 0;
                            phase ^= 1u;
                        }
                        continue;
                    }
                    if (!wait_phase(&s.empty[stage], phase ^ 1u, s.abort, tmo)) {
                        ok = false;
                        break;
                    }
                    uint8_t* sp = s.stages + size_t(stage) * (p.p_bytes + p.q_bytes + p.sf_bytes);
                    uint8_t* sq = sp + p.p_bytes;
                    const int k0 = kb * p.bk;
                    if (p.test_stall && blockIdx.x == 0 && first_seg && i == 0) {
                        // Failure-detection test: expect the stage's bytes but
                        // load nothing, so this stage never fills.
                        mbar_arrive_expect_tx(&s.full[stage], PAIR ? 2 * tx : tx);
                        if (++stage == p.stages) {
                            stage = 0;
                            phase ^= 1u;
                        }
                        continue;
                    }
                    if (PAIR) {
                        // Both CTAs' fills complete on the leader's full barrier;
                        // the leader expects the bytes of both.
                        const uint32_t fb = mapa_shared(smem_u32(&s.full[stage]), 0);
                        if (rank == 0) mbar_arrive_expect_tx(&s.full[stage], 2 * tx);
                        if (p.p_mn) {
                            tma_load_2d_pair_hint(sp, &mapP, fb, p0, k0, pol_p);
                            if (p.bp > 64)
                                tma_load_2d_pair_hint(sp + kAtomBytes, &mapPh, fb, p0 + 64, k0,
                                                      pol_p);
                        } else {
                            tma_load_2d_pair_hint(sp, &mapP, fb, k0, p0, pol_p);
                        }
                        const int qh = q0 + rank * q_rows;  // this CTA's half of the unit's Q
                        if (p.q_mn) {
                            for (int a = 0; a < q_atoms; ++a)
                                tma_load_2d_pair_hint(sq + a * kAtomBytes, &mapQ, fb, qh + 64 * a,
                                                      k0, pol_q);
                        } else {
                            tma_load_2d_pair_hint(sq, mq, fb, k0, qh, pol_q);
                        }
                        if constexpr (MX) {
                            // This CTA's P chunk and all of the tile's Q chunks.
                            uint8_t* sf = sq + p.q_bytes;
                            tma_load_2d_pair(sf, &mapSP, fb, 0, (p0 / p.bp) * p.k_blocks + kb);
                            tma_load_2d_pair(sf + 512, &mapSQ, fb, 0,
                                             (tq * p.k_blocks + kb) * p.sf_q_rows);
                        }
                        issued_any |= 1u << stage;
                        issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                        if (++stage == p.stages) {
                            stage = 0;
                            phase ^= 1u;
                        }
                        continue;
                    }
                    mbar_arrive_expect_tx(&s.full[stage], tx);
                    if (p.p_mn) {
                        tma_load_2d_hint(sp, &mapP, &s.full[stage], p0, k0, pol_p);
                        if (p.bp > 64)
                            tma_load_2d_hint(sp + kAtomBytes, &mapPh, &s.full[stage], p0 + 64, k0,
                                             pol_p);
                    } else {
                        tma_load_2d_hint(sp, &mapP, &s.full[stage], k0, p0, pol_p);
                    }
                    if (p.q_mn) {
                        for (int a = 0; a < q_atoms; ++a)
                            tma_load_2d_hint(sq + a * kAtomBytes, &mapQ, &s.full[stage],
                                             q0 + 64 * a, k0, pol_q);
                    } else {
                        tma_load_2d_hint(sq, mq, &s.full[stage], k0, q0, pol_q);
                    }
                    if constexpr (MX) {
                        // This stage's packed scales: the P tile's chunk, then
                        // the Q tile's chunks.
                        uint8_t* sf = sq + p.q_bytes;
                        tma_load_2d(sf, &mapSP, &s.full[stage], 0, (p0 / p.bp) * p.k_blocks + kb);
                        tma_load_2d(sf + 512, &mapSQ, &s.full[stage], 0,
                                    (tq * p.k_blocks + kb) * p.sf_q_rows);
                    }
                    issued_any |= 1u << stage;
                    issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == p.stages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        }
        if (warp != 0) __syncwarp();  // a second-group warp goes on to its epilogue
    }
    if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        // (in pair mode only the leader CTA issues, for both CTAs)
        if (lane == 0 && (!PAIR || rank == 0)) {
            // Descriptor templates, encoded once; each issue patches the start address.
            const uint64_t dP = p.p_mn ? smem_desc_sw128_template(kAtomBytes, 1024)
                                       : smem_desc_sw128_template(16, 1024);
            const uint64_t dQ = p.q_mn ? smem_desc_sw128_template(kAtomBytes, 1024)
                                       : smem_desc_sw128_template(16, 1024);
            // Start-address step per 16-deep K slice: 32 bytes along a K-major
            // swizzle row, 16 rows of 128 bytes for an MN-major tile.
            const uint32_t stepP = p.p_mn ? kUmmaK * 128 : kUmmaK * 2;
            const uint32_t stepQ = p.q_mn ? kUmmaK * 128 : kUmmaK * 2;
            const uint32_t stage_base = smem_u32(s.stages);
            // Loop invariants in registers: each issue below is an asm with a
            // memory clobber, after which parameters would be read again.
            const uint32_t stage_bytes = p.p_bytes + p.q_bytes + p.sf_bytes;
            const uint32_t pq_bytes = p.p_bytes + p.q_bytes;
            // Scale slots (MX): a no-swizzle K-major source of 16-byte rows, 8-row
            // groups 128 bytes apart (a second 16-byte unit of each row 2 KB on,
            // for the replicated Q image); each stage has its own slot in
            // tensor memory.
            const uint64_t dSF = smem_desc_template(512, 128, kDescLayoutNone);
            const uint64_t dSF2 = smem_desc_template(2048, 128, kDescLayoutNone);
            const bool sf_q_wide = p.sf_q_rows == 8;
            const uint32_t sf_slot0 = tmem + uint32_t(p.sf_col0);
            const uint32_t sf_cols = uint32_t(p.sf_cols);
            const int sf_spr = p.sf_spr > 0 ? p.sf_spr : 1;
            const uint32_t half_cols = uint32_t(p.tmem_cols / 2);
            const uint32_t p_bytes = p.p_bytes;
            const int nstages = p.stages;
            int stage = 0;
            uint32_t phase = 0;
            int it = 0;
            bool ok = true;
            SegIter iter(cid, ncl, p);
            Seg u;
            // The MMA kind is fixed per launch: the issue loop is instantiated
            // once per kind and chosen once, so no test sits between MMAs.
            auto issue_all = [&](auto fp8_tag) {
            constexpr bool FP8 = decltype(fp8_tag)::value;
            for (; ok && iter.next(ncl, p, u); ++it) {
                const uint32_t idesc = u.width == p.bn ? p.idesc : p.idesc_tail;
                const int nk = u.kb1 - u.kb0;
                const int b = it & 1;
                const uint32_t acc_phase = (it >> 1) & 1;
                if (!wait_phase(&s.acc_empty[b], acc_phase ^ 1u, s.abort, tmo)) break;
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem + uint32_t(b * acc_stride);
                if (!in_bounds(b * acc_stride + 32 * ((p.bn + 31) / 32) <= p.tmem_cols,
                               kSiteMmaAccumulator)) {
                    ok = false;
                    break;
                }
                for (int i = 0; i < nk; ++i) {
                    if (!wait_phase(&s.full[stage], phase, s.abort, tmo)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t ap = stage_base + uint32_t(stage) * stage_bytes;
                    const uint32_t aq = ap + p_bytes;
                    if constexpr (MX) {
                        // The stage's scales into its slot: tcgen05.cp and the
                        // MMAs below, issued by this thread, run in issue order
                        // (in a pair, the copy fills both CTAs' slots, each from
                        // its own shared memory). A slot is rewritten one ring
                        // later: that fill has landed only after the producer
                        // saw this stage's MMAs complete.
                        const uint32_t sfs = ap + pq_bytes;
                        const int hs = stage / sf_spr;
                        const uint32_t slot = sf_slot0 + uint32_t(hs) * half_cols +
                                              uint32_t(stage - hs * sf_spr) * sf_cols;
                        if (!in_bounds((slot - tmem) + sf_cols <= uint32_t(p.tmem_cols),
                                       kSiteScaleSlot)) {
                            ok = false;
                            break;
                        }
                        tc_cp<CG>(6, slot, smem_desc_with_addr(dSF, sfs));
                        if (sf_q_wide)  // both Q chunks, replicated: 128x256b
                            tc_cp<CG>(1, slot + 4u, smem_desc_with_addr(dSF2, sfs + 512u));
                        else
                            tc_cp<CG>(6, slot + 4u, smem_desc_with_addr(dSF, sfs + 512u));
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint64_t adesc = smem_desc_with_addr(dP, ap + kk * 32);
                            const uint64_t bdesc = smem_desc_with_addr(dQ, aq + kk * 32);
                            // scale-factor IDs (bits 29-30 for A, 4-5 for B) = kk
                            const uint32_t id = idesc | (uint32_t(kk) << 29) | (uint32_t(kk) << 4);
                            if constexpr (PAIR)
                                tc_mma_mx_pair(d_tmem, adesc, bdesc, id, slot, slot + 4u,
                                               (i | kk) != 0);
                            else
                                tc_mma_mx(d_tmem, adesc, bdesc, id, slot, slot + 4u, (i | kk) != 0);
                        }
                        if (PAIR)
                            tc_commit_pair_multicast(&s.empty[stage], pair_mask);
                        else
                            tc_commit(&s.empty[stage]);
                        if (++stage == nstages) {
                            stage = 0;
                            phase ^= 1u;
                        }
                        continue;
                    }
#pragma unroll
                    for (int kk = 0; kk < kBK / kUmmaK; ++kk) {
                        const uint64_t adesc = smem_desc_with_addr(dP, ap + kk * stepP);
                        const uint64_t bdesc = smem_desc_with_addr(dQ, aq + kk * stepQ);
                        const uint32_t acc = (i | kk) != 0;
                        if constexpr (PAIR) {
                            if constexpr (FP8)
                                tc_mma_f8_pair(d_tmem, adesc, bdesc, idesc, acc);
                            else
                                tc_mma_f16_pair(d_tmem, adesc, bdesc, idesc, acc);
                        } else {
                            if constexpr (FP8)
                                tc_mma_f8(d_tmem, adesc, bdesc, idesc, acc);
                            else
                                tc_mma_f16(d_tmem, adesc, bdesc, idesc, acc);
                        }
                    }
                    // Stage free (in both CTAs of a pair) once these MMAs finish.
                    if (PAIR)
                        tc_commit_pair_multicast(&s.empty[stage], pair_mask);
                    else
                        tc_commit(&s.empty[stage]);
                    if (++stage == nstages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                // Accumulator ready for the epilogue (of both CTAs in pair mode).
                if (PAIR)
                    tc_commit_pair_multicast(&s.acc_full[b], pair_mask);
                else
                    tc_commit(&s.acc_full[b]);
                // The last one also for the helper warps (a barrier of its own,
                // which completes once per launch).
                if (p.epi_help && !iter.more(p)) {
                    if (PAIR)
                        tc_commit_pair_multicast(s.last_full, pair_mask);
                    else
                        tc_commit(s.last_full);
                }
            }
            };
            if (p.fp8)
                issue_all(std::true_type{});
            else
                issue_all(std::false_type{});
            // Drain: every MMA this thread issued has completed before teardown.
            if (PAIR)
                tc_commit_pair(s.drain);
            else
                tc_commit(s.drain);
            wait_phase(s.drain, 0, s.abort, tmo, true);
        }
    } else if (warp >= 2 && (warp < 2 + kEpiQuads * p.epi_groups || p.epi_help)) {
        // (A producing warp of the second group has issued its fills first.)
        // --------------------------------------------------------- epilogue
        if constexpr (EARLY) grid_dependency_wait();
        const int ew = warp - 2;           // 0 .. 4 epi_groups - 1, or 4 .. 7 for a helper
        const int quad = warp & 3;         // tensor-memory lane quadrant of this warp
        // A helper (warps 6..9 of a one-group plan with epi_help) works on the
        // CTA's last segment only, and has no staging tiles of its own: by
        // then the TMA ring is idle and holds its chunks.
        const bool helper = ew >= kEpiQuads * p.epi_groups;
        const EpiShare es = helper ? EpiShare{1, 0, nullptr, nullptr} : epi_share(s, p, ew);
        const int nbw = es.nbw;
        float* bufs = es.bufs;
        uint64_t* cb = es.cb;
        const uint32_t lane_base = uint32_t(quad * 32) << 16;
        // C is read once and D written once: their lines should not push the
        // operand panels that later tiles reuse out of L2. (A stream-K tile's
        // zeros, which its reductions read back, keep the normal policy.)
        const uint64_t pol_cd = l2_policy(p.l2_cd);

        // Output extents in the kernel's (P, Q) frame, for skipping empty chunks.
        const int lim_p = p.Mp;
        const int lim_q = p.Nq;
        if (p.sk && !helper) {
            const int ng = p.epi_groups;
            const int half = es.g;
            // Stream-K: the leftover tile whose first K blocks this cluster
            // holds (at most one) gets this warp's part of its D region zeroed
            // now, under the MMAs of the whole units, and a flag published
            // once the zeros are written; every segment of the tile then adds
            // its accumulator into D with a TMA reduction.
            SegIter pre(cid, ncl, p);
            Seg v;
            while (pre.next(ncl, p, v)) {
                if (!(v.owner && v.has_next)) continue;
                int tps, tq;
                tile_coords(v.T, p, tps, tq);
                const int pw = (tps * MC + rank) * p.bp + quad * 32;
                const int q0 = tq * p.bn + v.q_off;
                const int q_lanes = min(32, p.bp - quad * 32);
                const int live = (pw < lim_p && q_lanes > 0)
                                     ? min((v.width + 31) / 32, (lim_q - q0 + 31) / 32)
                                     : 0;
                const int my_chunks = live > half ? (live - half + ng - 1) / ng : 0;
                if (my_chunks == 0) break;
                const CUtensorMap* dmap = q_lanes == 16 ? &mapDh : &mapD;
                float4* z = reinterpret_cast<float4*>(bufs);
                for (int k = lane; k < kEpiBufFloats / 4; k += 32)
                    z[k] = make_float4(0.f, 0.f, 0.f, 0.f);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    for (int j = 0; j < my_chunks; ++j) {
                        const int c = ng * j + half;
                        const int x = SWAP ? pw : q0 + 32 * c;
                        const int y = SWAP ? q0 + 32 * c : pw;
                        if (in_bounds(x >= 0 && y >= 0 && x % 4 == 0, kSiteStore))
                            tma_store_2d(dmap, bufs, x, y);
                    }
                    bulk_commit_group();
                    bulk_wait_group<0>();  // written, not just read
                    fence_proxy_async_global();
                    if (in_bounds(int(blockIdx.x) * kEpiWarps + ew < kTcMaxFlagSlots * kEpiWarps,
                                  kSiteFlag)) {
                        st_release_gpu(&p.sk_flags[blockIdx.x * kEpiWarps + ew], p.sk_epoch);
                        // This warp zeroed every chunk of its quadrant, so the
                        // quadrant's helper may add into them too.
                        if (p.epi_help)
                            st_release_gpu(&p.sk_flags[blockIdx.x * kEpiWarps + ew + kEpiQuads],
                                           p.sk_epoch);
                    }
                }
                __syncwarp();
                break;
            }
        }
        int it = 0;
        SegIter iter(cid, ncl, p);
        Seg u;
        for (; iter.next(ncl, p, u); ++it) {
            const bool last = !iter.more(p);
            if (helper && !last) continue;
            // The last segment of an epi_help plan: the quadrant's first warp
            // takes the even chunks, its helper the odd ones.
            const bool shared_last = p.epi_help && last;
            const int ng = shared_last ? 2 : p.epi_groups;
            const int half = shared_last ? (helper ? 1 : 0) : es.g;
            int tps, tq;
            tile_coords(u.T, p, tps, tq);
            const int tp = tps * MC + rank;
            const int pw = tp * p.bp + quad * 32;  // first P row of this warp's quadrant
            const int q0 = tq * p.bn + u.q_off;
            const int nchunks = (u.width + 31) / 32;
            // Lanes of this quadrant inside the tile's bp rows: 32, 16 (the
            // half-width boxes) or none.
            const int q_lanes = min(32, p.bp - quad * 32);
            const bool half_q = q_lanes == 16;
            const bool warp_live = pw < lim_p && q_lanes > 0;
            int live_chunks = 0;
            if (warp_live) live_chunks = min(nchunks, (lim_q - q0 + 31) / 32);
            // This warp's chunks: c = ng j + half for j < my_chunks.
            const int my_chunks = live_chunks > half ? (live_chunks - half + ng - 1) / ng : 0;
            // Stream-K: a tile split into K segments gets its D region zeroed
            // by its first segment (the owner, which also adds C), and every
            // segment adds its accumulator into D with a TMA reduction; two
            // or more f32 addends onto zero, so the order of the reductions
            // does not matter when there are two. The owner publishes a flag
            // once its zeros are written; the others wait for it before their
            // first reduction.
            const bool split = !(u.owner && !u.has_next);
            const bool add_src = p.beta && u.owner;
            const int owner_block =
                (u.owner ? cid : sk_owner_cluster(u.T - p.full_units, p)) * MC + rank;
            auto box_x = [&](int c) { return SWAP ? pw : q0 + 32 * c; };
            auto box_y = [&](int c) { return SWAP ? q0 + 32 * c : pw; };
            // D / C boxes: (x = column, y = row) of D.
            const CUtensorMap* src_map = half_q ? &mapCh : &mapC;
            const CUtensorMap* dst_map = half_q ? &mapDh : &mapD;
            const uint32_t src_bytes = half_q ? kEpiBufFloats * 2 : kEpiBufFloats * 4;
            auto src_x = [&](int c) { return box_x(c); };
            auto src_y = [&](int c) { return box_y(c); };
            auto dst_x = [&](int c) { return box_x(c); };
            auto dst_y = [&](int c) { return box_y(c); };

            // All staging buffers free: every earlier store has read its source.
            if (lane == 0) bulk_wait_group_read<0>();
            // Prefetch C for the first chunks (all of them when they fit the
            // staging buffers) while the MMAs run.
            if (add_src) {
                for (int j = 0; j < nbw && j < my_chunks; ++j) {
                    const int c = ng * j + half;
                    if (lane == 0 && in_bounds(src_x(c) % 4 == 0, kSiteLoadC)) {
                        mbar_arrive_expect_tx(&cb[j], src_bytes);
                        tma_load_2d_hint(bufs + j * kEpiBufFloats, src_map, &cb[j], src_x(c),
                                         src_y(c), pol_cd);
                    }
                    cpend |= 1u << j;
                }
            }
            __syncwarp();
            if (helper && my_chunks == 0) break;
            const int b = it & 1;
            const uint32_t acc_phase = (it >> 1) & 1;
            // (A helper may wait from kernel start: its bound covers each of
            // the cluster's segments, as the other waits cover one.)
            bool ok = helper ? wait_phase(s.last_full, 0, s.abort, tmo * uint64_t(it + 1))
                             : wait_phase(&s.acc_full[b], acc_phase, s.abort, tmo);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            // A helper of the tile's owner waits for the zeros as well: the
            // owner's first warps wrote them.
            if (split && (!u.owner || helper) && my_chunks > 0) {
                // The owner's zeros are in D before this segment adds to it.
                bool fok = true;
                if (lane == 0) {
                    fok = in_bounds(owner_block * kEpiWarps + ew < kTcMaxFlagSlots * kEpiWarps,
                                    kSiteFlag) &&
                          wait_flag(&p.sk_flags[owner_block * kEpiWarps + ew], p.sk_epoch, s.abort,
                                    tmo);
                    fence_proxy_async_global();
                }
                ok = __shfl_sync(0xffffffffu, fok ? 1 : 0, 0) != 0;
                if (!ok) break;
            }
            tc_fence_after_sync();
            const uint32_t acc_col = uint32_t(b * acc_stride);
            // This warp's j-th chunk (column chunk c = ng j + half): its
            // accumulator registers `cur` were loaded by the previous step; the
            // next chunk's tcgen05.ld is issued into `nxt` before this one's
            // shared-memory work so the two overlap.
            // This CTA's last unit, with no source to load: once its MMAs are
            // done (acc_full, which in a pair also covers the leader's reads
            // of this CTA's half) no fill or MMA touches the TMA ring again,
            // so D is staged through the ring, one buffer per chunk, and no
            // chunk waits for an earlier store to have read its buffer.
            // A helper always stages this way (the plan checks that its chunks
            // fit), and loads the segment's C, if any, once the ring is idle.
            int snbw = nbw;
            if ((helper || !add_src) && last) {
                const int per_warp =
                    int((uint32_t(p.stages) * (p.p_bytes + p.q_bytes + p.sf_bytes)) /
                        (uint32_t(kEpiQuads * ng) * uint32_t(kEpiBufFloats * sizeof(float))));
                if (per_warp >= my_chunks && (helper || my_chunks > nbw)) {
                    snbw = my_chunks;
                    bufs = reinterpret_cast<float*>(s.stages) + ew * per_warp * kEpiBufFloats;
                }
            }
            if (helper) {
                if (!in_bounds(snbw == my_chunks, kSiteHelperStaging)) break;
                if (add_src) {
                    if (lane == 0) {
                        uint32_t bytes = 0;
                        for (int j = 0; j < my_chunks; ++j)
                            if (in_bounds(src_x(ng * j + half) % 4 == 0, kSiteLoadC))
                                bytes += src_bytes;
                        mbar_arrive_expect_tx(&s.hbar[quad], bytes);
                        for (int j = 0; j < my_chunks; ++j) {
                            const int c = ng * j + half;
                            if (in_bounds(src_x(c) % 4 == 0, kSiteLoadC))
                                tma_load_2d_hint(bufs + j * kEpiBufFloats, src_map, &s.hbar[quad],
                                                 src_x(c), src_y(c), pol_cd);
                        }
                    }
                    hpend = true;
                    bool cok = wait_phase(&s.hbar[quad], 0, s.abort, tmo);
                    ok = __all_sync(0xffffffffu, cok);
                    if (!ok) break;
                    hpend = false;
                }
            }
            auto chunk = [&](int j, uint32_t (&cur)[32], uint32_t (&nxt)[32]) -> bool {
                const int c = ng * j + half;
                const int bi = j % snbw;
                float* buf = bufs + bi * kEpiBufFloats;
                tmem_ld_wait(cur);
                if (j + 1 < my_chunks &&
                    in_bounds(acc_col + uint32_t(32 * (c + ng)) + 32u <=
                                  acc_col + uint32_t(acc_stride),
                              kSiteEpilogueLoad))
                    tmem_ld_32x32b_x32(tmem + lane_base + acc_col + uint32_t(32 * (c + ng)), nxt);
                if (add_src && !helper) {
                    bool cok = wait_phase(&cb[bi], (cphase >> bi) & 1u, s.abort, tmo);
                    cok = __all_sync(0xffffffffu, cok);
                    if (!cok) {
                        tmem_ld_wait_all();
                        return false;
                    }
                    cphase ^= 1u << bi;
                    cpend &= ~(1u << bi);
                } else if (j >= snbw) {
                    // The store that last used buf (this warp's chunk j - nbw) has read it.
                    if (lane == 0) {
                        if (snbw == 1)
                            bulk_wait_group_read<0>();
                        else
                            bulk_wait_group_read<1>();
                    }
                    __syncwarp();
                }
                if (!SWAP) {
                    // Lane = P row = D row; 8 16-byte chunks of its 32 columns,
                    // placed by the 128-byte swizzle (chunk ^ row % 8). All C
                    // reads are issued before any D write.
                    float4* row = reinterpret_cast<float4*>(buf + lane * 32);
                    float4 cv[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        cv[j] = add_src ? row[j ^ (lane & 7)] : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        row[j ^ (lane & 7)] = make_float4(__uint_as_float(cur[4 * j]) + cv[j].x,
                                                          __uint_as_float(cur[4 * j + 1]) + cv[j].y,
                                                          __uint_as_float(cur[4 * j + 2]) + cv[j].z,
                                                          __uint_as_float(cur[4 * j + 3]) + cv[j].w);
                } else {
                    // Lane = P row = D column; register i is D row 32c + i.
                    float cv[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        cv[i] = add_src ? buf[i * 32 + (((lane >> 2) ^ (i & 7)) << 2) + (lane & 3)]
                                        : 0.f;
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        buf[i * 32 + (((lane >> 2) ^ (i & 7)) << 2) + (lane & 3)] =
                            __uint_as_float(cur[i]) + cv[i];
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0 && in_bounds(dst_x(c) >= 0 && dst_y(c) >= 0 && dst_x(c) % 4 == 0,
                                           kSiteStore)) {
                    if (split)
                        tma_reduce_add_2d(dst_map, buf, dst_x(c), dst_y(c));
                    else
                        tma_store_2d_hint(dst_map, buf, dst_x(c), dst_y(c), pol_cd);
                    bulk_commit_group();
                    if (add_src && !helper && j + nbw < my_chunks) {
                        const int cn = c + ng * nbw;  // this warp's chunk j + nbw
                        bulk_wait_group_read<0>();  // the store just issued has read buf
                        mbar_arrive_expect_tx(&cb[bi], src_bytes);
                        tma_load_2d_hint(buf, src_map, &cb[bi], src_x(cn), src_y(cn), pol_cd);
                    }
                }
                if (add_src && !helper && j + nbw < my_chunks) cpend |= 1u << bi;
                __syncwarp();
                return true;
            };
            uint32_t ra[32], rb[32];
            uint32_t first_col = acc_col + uint32_t(32 * half);
#ifdef TPGEMM_DEBUG
            if (p.debug_plant) first_col += uint32_t(p.tmem_cols);  // caught below
#endif
            if (my_chunks > 0 &&
                in_bounds(first_col + 32u <= acc_col + uint32_t(acc_stride), kSiteEpilogueLoad))
                tmem_ld_32x32b_x32(tmem + lane_base + first_col, ra);
            for (int j = 0; j < my_chunks && ok; j += 2) {
                ok = chunk(j, ra, rb);
                if (ok && j + 1 < my_chunks) ok = chunk(j + 1, rb, ra);
            }
            // Accumulator buffer b may be overwritten by the next tile's MMAs
            // (issued by the pair's leader in pair mode).
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0 && !helper) {
                if (PAIR)
                    mbar_arrive_cluster(mapa_shared(smem_u32(&s.acc_empty[b]), 0));
                else
                    mbar_arrive(&s.acc_empty[b]);
            }
            if (!ok) break;
        }
        // Staging tiles must be read by their stores before shared memory is
        // released; the stores' global writes complete with the grid.
        if (lane == 0) bulk_wait_group_read<0>();
    }

    // --------------------------------------------------------------- teardown
    tc_fence_before_sync();
    __syncthreads();
    if (*s.abort) {
        // An aborted CTA lets every TMA fill it issued land before it exits.
        // (In pair mode both CTAs' fills complete on the leader's barriers,
        // so the leader drains for both before the final cluster sync.)
        if (prod_r >= 0 && lane == 0 && (!PAIR || rank == 0))
            for (int i = 0; i < p.stages; ++i)
                if (issued_any & (1u << i))
                    wait_phase(&s.full[i], (issued_parity >> i) & 1u, s.abort, tmo, true);
        if (warp >= 2 && warp < 2 + kEpiQuads * p.epi_groups) {
            const EpiShare es = epi_share(s, p, warp - 2);
            for (int i = 0; i < es.nbw; ++i)
                if (cpend & (1u << i))
                    wait_phase(&es.cb[i], (cphase >> i) & 1u, s.abort, tmo, true);
        }
        if (hpend) wait_phase(&s.hbar[warp & 3], 0, s.abort, tmo, true);
        __syncthreads();
    }
    // No CTA of a pair leaves while its peer may still arrive on its barriers.
    if constexpr (PAIR) cluster_sync();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after_sync();
        tmem_dealloc<CG>(tmem, uint32_t(p.tmem_cols));
    }
}

}  // namespace

using TcKernelFn = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap,
                            CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap,
                            TcParams);

template <bool EARLY>
TcKernelFn pick_kernel_dep(const TcParams& p) {
    if (p.mx) {
        if (p.pair)
            return p.swap ? tc_gemm_kernel<true, true, EARLY, true>
                          : tc_gemm_kernel<false, true, EARLY, true>;
        return p.swap ? tc_gemm_kernel<true, false, EARLY, true>
                      : tc_gemm_kernel<false, false, EARLY, true>;
    }
    if (p.pair)
        return p.swap ? tc_gemm_kernel<true, true, EARLY, false>
                      : tc_gemm_kernel<false, true, EARLY, false>;
    return p.swap ? tc_gemm_kernel<true, false, EARLY, false>
                  : tc_gemm_kernel<false, false, EARLY, false>;
}

// The early-start choice is a template parameter, not a runtime test: a
// runtime test of it cost 8192^3 about 1.4 % (same register use).
TcKernelFn pick_kernel(const TcParams& p) {
    return p.dep_early ? pick_kernel_dep<true>(p) : pick_kernel_dep<false>(p);
}


size_t tc_smem_bytes(int stages, uint32_t stage_bytes, int epi_bufs) {
    return 1024 + size_t(stages) * stage_bytes +
           size_t(kEpiQuads) * epi_bufs * kEpiBufFloats * sizeof(float) +
           sizeof(uint64_t) * (2 * size_t(stages) + 4 + kTcMaxEpiBufs * kEpiQuads + 2 + kEpiQuads) +
           16;
}

bool tc_epi_help_fits(const TcParams& p) {
    const uint32_t ring = uint32_t(p.stages) * (p.p_bytes + p.q_bytes + p.sf_bytes);
    const uint32_t per_warp = ring / (uint32_t(2 * kEpiQuads) * kEpiBufFloats * sizeof(float));
    const int chunks = (p.bn + 31) / 32;
    return per_warp >= uint32_t((chunks + 1) / 2);
}

cudaError_t launch_tc(const TcMaps& maps, const TcParams& p, int grid, cudaStream_t stream) {
    if (p.epi_bufs < 2 || p.epi_bufs > kTcMaxEpiBufs || p.stages < 2 || p.stages > 32 ||
        p.producers < 1 || p.producers > 4 || p.producers > p.stages ||
        !(p.epi_groups == 1 || p.epi_groups == 2) ||
        p.mc != (p.pair ? 2 : 1) || grid % p.mc != 0 ||
        !(p.tmem_cols == 64 || p.tmem_cols == 128 || p.tmem_cols == 256 || p.tmem_cols == 512) ||
        p.tmem_cols / 2 < 32 * ((p.bn + 31) / 32))
        return cudaErrorInvalidValue;
    // MX: one scale slot per stage in the accumulator halves past the tile's
    // columns, 1024-aligned stages (P tiles of bp rows, packed as such).
    if (p.mx && (p.tail_split != 1 || p.sk || p.tmem_cols != 512 ||
                 !(p.sf_q_chunks == 1 || p.sf_q_chunks == 2) ||
                 p.sf_q_rows != (p.sf_q_chunks == 2 ? 8 : 1) ||
                 p.sf_cols != 4 + 4 * p.sf_q_chunks || p.sf_col0 < 32 * ((p.bn + 31) / 32) ||
                 p.sf_spr < 1 || p.sf_col0 + p.sf_spr * p.sf_cols > 256 ||
                 p.stages > 2 * p.sf_spr || p.sf_bytes < 512u * uint32_t(1 + p.sf_q_rows) ||
                 (p.p_bytes + p.q_bytes + p.sf_bytes) % 1024 != 0))
        return cudaErrorInvalidValue;
    if (!p.mx && p.sf_bytes != 0) return cudaErrorInvalidValue;
    // Helper warps: one-group plans whose ring holds a helper's share of a tile.
    if (p.epi_help && (p.epi_groups != 1 || !tc_epi_help_fits(p))) return cudaErrorInvalidValue;
    // Every stream-K K block must belong to a cluster of the grid.
    if (p.sk && (p.sk_ncl < 1 || p.sk_ncl > grid / p.mc)) return cudaErrorInvalidValue;
    const size_t smem = tc_smem_bytes(p.stages, p.p_bytes + p.q_bytes + p.sf_bytes, p.epi_bufs);
    if (smem > size_t(kTcMaxSmem)) return cudaErrorInvalidConfiguration;
    auto kernel = pick_kernel(p);
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(smem));
    if (e != cudaSuccess) return e;
    // Programmatic dependent launch: this grid's set-up may overlap the tail of
    // the previous kernel in the stream; the kernel waits (griddepcontrol.wait)
    // before its first global-memory access.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(grid));
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = unsigned(p.mc);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = p.mc > 1 ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kernel, maps.P, maps.Q, maps.C, maps.D, maps.Qt, maps.Ph,
                              maps.Ch, maps.Dh, maps.SP, maps.SQ, p);
}

cudaError_t tc_max_active_clusters(const TcParams& p, int* clusters) {
    const size_t smem = tc_smem_bytes(p.stages, p.p_bytes + p.q_bytes + p.sf_bytes, p.epi_bufs);
    auto kernel = pick_kernel(p);
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(smem));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(p.mc));
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = unsigned(p.mc);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaOccupancyMaxActiveClusters(clusters, kernel, &cfg);
}

cudaError_t tc_static_scratch(void** ptr) {
    // Host code names g_static_scratch only through its device address, taken
    // once per device with that device current; the flags start at zero.
    static std::mutex m;
    static void* addr[kMaxStaticScratchDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxStaticScratchDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(m);
    if (!addr[dev]) {
        void* a = nullptr;
        e = cudaGetSymbolAddress(&a, g_static_scratch);
        if (e != cudaSuccess) return e;
        e = cudaMemset(a, 0, kStaticScratchBytes);
        if (e != cudaSuccess) return e;
        e = cudaDeviceSynchronize();
        if (e != cudaSuccess) return e;
        addr[dev] = a;
    }
    *ptr = addr[dev];
    return cudaSuccess;
}

cudaError_t tc_read_and_clear_device_status(int* status, int* bounds_site) {
    cudaError_t e = cudaMemcpyFromSymbol(status, g_tc_status, sizeof(int));
    if (e == cudaSuccess) e = cudaMemcpyFromSymbol(bounds_site, g_tc_bounds_site, sizeof(int));
    if (e != cudaSuccess) return e;
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_tc_status, &zero, sizeof(int));
    if (e != cudaSuccess) return e;
    return cudaMemcpyToSymbol(g_tc_bounds_site, &zero, sizeof(int));
}

}  // namespace tpg
