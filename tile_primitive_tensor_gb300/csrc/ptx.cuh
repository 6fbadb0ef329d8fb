// Inline-PTX building blocks for sm_103a: mbarrier, TMA (cp.async.bulk.tensor),
// tcgen05 (alloc / mma / commit / ld / fences), warp-level mma.sync, ldmatrix
// and cp.async. Each wrapper is one instruction (or a bounded loop of one), so
// the kernels read as the sequence of hardware operations they issue.
#pragma once

#include <cstdint>
#include <cuda.h>

namespace tpg {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbarrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

// One probe of the phase with the given parity; true once that phase completed.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// ------------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* map, uint64_t* bar,
                                            int32_t x, int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y)
        : "memory");
}

// L2 eviction-priority policy for the cache-hinted copies below: 0 normal,
// 1 evict_first (data read or written once), 2 evict_last (data reused).
__device__ __forceinline__ uint64_t l2_policy(int kind) {
    uint64_t pol;
    if (kind == 1)
        asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    else if (kind == 2)
        asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    else
        asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// tma_load_2d with an L2 eviction-priority policy.
__device__ __forceinline__ void tma_load_2d_hint(void* smem_dst, const CUtensorMap* map,
                                                 uint64_t* bar, int32_t x, int32_t y,
                                                 uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "l"(policy)
        : "memory");
}

// CTA-pair form: the box lands in this CTA's shared memory and its bytes
// complete on an mbarrier that may live in the peer CTA of the pair (a
// shared::cluster address, e.g. from mapa).
__device__ __forceinline__ void tma_load_2d_pair(void* smem_dst, const CUtensorMap* map,
                                                 uint32_t bar_cluster_addr, int32_t x, int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster_addr), "r"(x), "r"(y)
        : "memory");
}

// 1-D bulk copy global -> this CTA's shared memory; `bytes` a multiple of 16,
// both addresses 16-byte aligned; the bytes complete on `bar`.
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes,
                                          uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(gsrc)), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// tma_load_2d_pair with an L2 eviction-priority policy.
__device__ __forceinline__ void tma_load_2d_pair_hint(void* smem_dst, const CUtensorMap* map,
                                                      uint32_t bar_cluster_addr, int32_t x,
                                                      int32_t y, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster_addr), "r"(x), "r"(y), "l"(policy)
        : "memory");
}

// tma_store_2d with an L2 eviction-priority policy.
__device__ __forceinline__ void tma_store_2d_hint(const CUtensorMap* map, const void* smem_src,
                                                  int32_t x, int32_t y, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group.L2::cache_hint"
        " [%0, {%2, %3}], [%1], %4;" ::"l"(reinterpret_cast<uint64_t>(map)),
        "r"(smem_u32(smem_src)), "r"(x), "r"(y), "l"(policy)
        : "memory");
}

// Prefetch one tensor-map box into L2 (no shared-memory destination, no
// completion to wait for).
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap* map, int32_t x, int32_t y) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y)
                 : "memory");
}

// Shared -> global tile reduction: each element of the box is added (f32, in
// L2) to the global element it maps to, as one bulk-group operation.
__device__ __forceinline__ void tma_reduce_add_2d(const CUtensorMap* map, const void* smem_src,
                                                  int32_t x, int32_t y) {
    asm volatile(
        "cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group"
        " [%0, {%2, %3}], [%1];" ::"l"(reinterpret_cast<uint64_t>(map)),
        "r"(smem_u32(smem_src)), "r"(x), "r"(y)
        : "memory");
}

__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* smem_src,
                                             int32_t x, int32_t y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::
                     "l"(reinterpret_cast<uint64_t>(map)),
                 "r"(smem_u32(smem_src)), "r"(x), "r"(y)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit_group() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

template <int N>
__device__ __forceinline__ void bulk_wait_group_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

template <int N>
__device__ __forceinline__ void bulk_wait_group() {
    asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// Orders this thread's generic-proxy shared-memory writes before later
// async-proxy (TMA) reads of the same bytes.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---------------------------------------------- cross-CTA publication (global)
// Flag store with release semantics at GPU scope (orders this thread's prior
// global writes, including completed bulk-async stores, before the flag).
__device__ __forceinline__ void st_release_gpu(uint32_t* addr, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* addr) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(addr) : "memory");
    return v;
}

// Orders generic-proxy accesses to global memory against async-proxy (TMA)
// accesses of the same memory by this thread.
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// ------------------------------------------------------------- clusters
// shared::cluster address of the same shared variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t smem_addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr), "r"(rank));
    return r;
}

// Arrive (release, cluster scope) on an mbarrier given by shared::cluster address.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(
                     bar_cluster_addr)
                 : "memory");
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Every thread of every CTA in the cluster arrives, then waits for all.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
                 ::: "memory");
}

// ------------------------------------------- programmatic dependent launch
// Block until the grids this one depends on have completed and their memory
// is visible (a no-op when the launch carried no programmatic dependency).
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Allow the next grid in the stream to begin launching (its CTAs still wait
// in grid_dependency_wait for this grid to finish before touching memory).
__device__ __forceinline__ void grid_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" :::);
}

// --------------------------------------------------------------- tcgen05
// CG = 1: this CTA's tensor memory. CG = 2: one warp of each CTA of a pair
// executes it, for a pair that issues cta_group::2 MMAs.
template <int CG>
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
    if constexpr (CG == 2)
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(dst_smem)),
                     "r"(ncols)
                     : "memory");
    else
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(dst_smem)),
                     "r"(ncols)
                     : "memory");
}

template <int CG>
__device__ __forceinline__ void tmem_relinquish_alloc_permit() {
    if constexpr (CG == 2)
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    else
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

template <int CG>
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    if constexpr (CG == 2)
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr),
                     "r"(ncols)
                     : "memory");
    else
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr),
                     "r"(ncols)
                     : "memory");
}

__device__ __forceinline__ void tc_fence_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Arrive once on the mbarrier when every tcgen05 operation this thread issued
// so far has completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// CTA-pair commits: track the pair's cta_group::2 MMAs issued by this thread.
__device__ __forceinline__ void tc_commit_pair(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tc_commit_pair_multicast(uint64_t* bar, uint16_t cta_mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(smem_u32(bar)),
        "h"(cta_mask)
        : "memory");
}

// CTA-pair MMA (M = 256): A rows 0..127 from this CTA's shared memory and rows
// 128..255 from the peer's at the same offset; B split along N between the
// two; each CTA's tensor memory receives its 128 rows of D.
__device__ __forceinline__ void tc_mma_f16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                                uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc], kind::f16 (f16/bf16 in, f32 acc).
__device__ __forceinline__ void tc_mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                           uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// kind::f8f6f4 (e4m3 / e5m2 in, f32 accumulate): the same operand forms and
// instruction descriptor fields as kind::f16, K = 32 per instruction (32 bytes
// of each row, as for kind::f16).
__device__ __forceinline__ void tc_mma_f8_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                               uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tc_mma_f8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Block-scaled MMA (kind::mxf8f6f4, one E8M0 scale per 32 K: scale_vec::1X):
// D[tmem] (+)= (A . SA) * (B . SB) with e4m3 / e5m2 operands from shared-memory
// descriptors, K = 32 per instruction. sfa_tmem / sfb_tmem address the scale
// columns in tensor memory; the instruction descriptor's scale-factor IDs pick
// the byte of each 32-bit scale cell.
__device__ __forceinline__ void tc_mma_mx(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, "
        "[%4], [%5], p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

// CTA-pair form (M = 256 across the pair, issued by the even CTA): each CTA's
// tensor memory holds the scales of its own 128 A rows and of all N B columns.
__device__ __forceinline__ void tc_mma_mx_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                               uint32_t idesc, uint32_t sfa_tmem,
                                               uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, "
        "[%4], [%5], p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread t of the warp receives
// lane (quadrant base + t), columns [col, col + 32).
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_ld_wait_all() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Wait for this thread's tcgen05.ld to land. The registers are passed through
// the asm so no use of them can be scheduled before the wait.
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.wait::ld.sync.aligned;"
        : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
          "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
          "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]),
          "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]),
          "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
        :
        : "memory");
}

// 32 lanes x 8 consecutive 32-bit columns, in both directions: thread t of
// the warp owns lane (quadrant base + t), register j column col + j.
__device__ __forceinline__ void tmem_st_32x32b_x8(uint32_t taddr, const uint32_t (&r)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::
                     "r"(taddr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
                 "r"(r[7])
                 : "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_ld_32x32b_x8(uint32_t taddr, uint32_t (&r)[8]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7])
        : "r"(taddr)
        : "memory");
}

// Shared memory -> tensor memory copy, issued by one thread. The source is the
// matrix named by the shared-memory descriptor; `form` selects the shape and
// multicast qualifier (1 128x256b, 2 4x256b, 3 128x128b, 4 64x128b.warpx2::02_13,
// 5 64x128b.warpx2::01_23, 6 32x128b.warpx4). CG = 2: issued by the even CTA
// of a pair; each CTA copies from its own shared memory into its own tensor
// memory.
template <int CG>
__device__ __forceinline__ void tc_cp(int form, uint32_t taddr, uint64_t sdesc) {
#define TPG_CP(SHAPE)                                                                         \
    do {                                                                                      \
        if constexpr (CG == 2)                                                                \
            asm volatile("tcgen05.cp.cta_group::2." SHAPE " [%0], %1;" ::"r"(taddr), "l"(sdesc) \
                         : "memory");                                                         \
        else                                                                                  \
            asm volatile("tcgen05.cp.cta_group::1." SHAPE " [%0], %1;" ::"r"(taddr), "l"(sdesc) \
                         : "memory");                                                         \
    } while (0)
    switch (form) {
        case 1: TPG_CP("128x256b"); break;
        case 2: TPG_CP("4x256b"); break;
        case 3: TPG_CP("128x128b"); break;
        case 4: TPG_CP("64x128b.warpx2::02_13"); break;
        case 5: TPG_CP("64x128b.warpx2::01_23"); break;
        case 6: TPG_CP("32x128b.warpx4"); break;
        default: break;
    }
#undef TPG_CP
}

// tcgen05.st / tcgen05.ld of any shape with N registers (N = 1, 2, 4, 8, 16):
// SHAPE_NUM is the literal "<shape>.x<num>" (e.g. "16x256b.x1"); R an array of
// uint32 registers. The caller issues tcgen05.wait::st / wait::ld.
#define TPG_TMEM_ARGS_ST1 "{%1}"
#define TPG_TMEM_ARGS_ST2 "{%1, %2}"
#define TPG_TMEM_ARGS_ST4 "{%1, %2, %3, %4}"
#define TPG_TMEM_ARGS_ST8 "{%1, %2, %3, %4, %5, %6, %7, %8}"
#define TPG_TMEM_ARGS_ST16 \
    "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16}"
#define TPG_TMEM_IN1(R) "r"((R)[0])
#define TPG_TMEM_IN2(R) TPG_TMEM_IN1(R), "r"((R)[1])
#define TPG_TMEM_IN4(R) TPG_TMEM_IN2(R), "r"((R)[2]), "r"((R)[3])
#define TPG_TMEM_IN8(R) TPG_TMEM_IN4(R), "r"((R)[4]), "r"((R)[5]), "r"((R)[6]), "r"((R)[7])
#define TPG_TMEM_IN16(R)                                                                   \
    TPG_TMEM_IN8(R), "r"((R)[8]), "r"((R)[9]), "r"((R)[10]), "r"((R)[11]), "r"((R)[12]), \
        "r"((R)[13]), "r"((R)[14]), "r"((R)[15])
#define TPG_TMEM_ST(SHAPE_NUM, N, TADDR, R)                                                   \
    asm volatile("tcgen05.st.sync.aligned." SHAPE_NUM ".b32 [%0], " TPG_TMEM_ARGS_ST##N ";" :: \
                     "r"(TADDR),                                                              \
                 TPG_TMEM_IN##N(R)                                                            \
                 : "memory")
#define TPG_TMEM_ARGS_LD1 "{%0}, [%1]"
#define TPG_TMEM_ARGS_LD2 "{%0, %1}, [%2]"
#define TPG_TMEM_ARGS_LD4 "{%0, %1, %2, %3}, [%4]"
#define TPG_TMEM_ARGS_LD8 "{%0, %1, %2, %3, %4, %5, %6, %7}, [%8]"
#define TPG_TMEM_ARGS_LD16 \
    "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16]"
#define TPG_TMEM_OUT1(R) "=r"((R)[0])
#define TPG_TMEM_OUT2(R) TPG_TMEM_OUT1(R), "=r"((R)[1])
#define TPG_TMEM_OUT4(R) TPG_TMEM_OUT2(R), "=r"((R)[2]), "=r"((R)[3])
#define TPG_TMEM_OUT8(R) \
    TPG_TMEM_OUT4(R), "=r"((R)[4]), "=r"((R)[5]), "=r"((R)[6]), "=r"((R)[7])
#define TPG_TMEM_OUT16(R)                                                                   \
    TPG_TMEM_OUT8(R), "=r"((R)[8]), "=r"((R)[9]), "=r"((R)[10]), "=r"((R)[11]),             \
        "=r"((R)[12]), "=r"((R)[13]), "=r"((R)[14]), "=r"((R)[15])
#define TPG_TMEM_LD(SHAPE_NUM, N, TADDR, R)                                                \
    asm volatile("tcgen05.ld.sync.aligned." SHAPE_NUM ".b32 " TPG_TMEM_ARGS_LD##N ";"      \
                 : TPG_TMEM_OUT##N(R)                                                      \
                 : "r"(TADDR)                                                              \
                 : "memory")

// -------------------------------------------------- descriptors (tcgen05)
// Shared-memory matrix descriptor (the PTX ISA's tcgen05 "shared memory
// descriptor" table). Fields: bits 0-13 start address >> 4, 16-29
// leading-dimension byte offset >> 4, 32-45 stride-dimension byte offset >> 4,
// 46-48 fixed 0b001, 49-51 base offset (0: buffers are aligned to the swizzle
// pattern's repeat), 52 LBO mode (0, relative), 61-63 layout type: 0 no swizzle,
// 2 128-byte, 4 64-byte, 6 32-byte swizzle.
enum : uint32_t {
    kDescLayoutNone = 0,
    kDescLayoutSw128 = 2,
    kDescLayoutSw64 = 4,
    kDescLayoutSw32 = 6,
};

// Encoded once with start address 0; each use ORs in the 14-bit start
// address (a tile stays inside the 256 KB shared window).
__host__ __device__ constexpr uint64_t smem_desc_template(uint32_t lbo_bytes, uint32_t sbo_bytes,
                                                          uint32_t layout) {
    return (uint64_t((lbo_bytes >> 4) & 0x3FFFu) << 16) |
           (uint64_t((sbo_bytes >> 4) & 0x3FFFu) << 32) | (uint64_t(1) << 46) |
           (uint64_t(layout & 7u) << 61);
}

__host__ __device__ constexpr uint64_t smem_desc_sw128_template(uint32_t lbo_bytes,
                                                                uint32_t sbo_bytes) {
    return smem_desc_template(lbo_bytes, sbo_bytes, kDescLayoutSw128);
}

__host__ __device__ constexpr uint64_t smem_desc_with_addr(uint64_t tmpl, uint32_t smem_addr) {
    return (tmpl & ~uint64_t(0x3FFF)) | uint64_t((smem_addr >> 4) & 0x3FFFu);
}

// Instruction descriptor for kind::f16 (and kind::f8f6f4) with an f32
// accumulator (the PTX ISA's instruction-descriptor table for those kinds):
// bits 4-5 D format (1 = f32), 7-9 A format and 10-12 B format (kind::f16:
// 0 = f16, 1 = bf16; kind::f8f6f4: 0 = e4m3, 1 = e5m2), 15 / 16 A / B
// major-ness (0 = K-major, 1 = MN-major), 17-22 N >> 3, 24-28 M >> 4. Dense,
// no negation, no saturation.
__host__ __device__ constexpr uint32_t idesc_f16_f32(uint32_t fmt, bool a_mn_major, bool b_mn_major,
                                                     int m, int n) {
    return (1u << 4) | ((fmt & 7u) << 7) | ((fmt & 7u) << 10) |
           (uint32_t(a_mn_major) << 15) | (uint32_t(b_mn_major) << 16) |
           (uint32_t(n >> 3) << 17) | (uint32_t(m >> 4) << 24);
}

// Instruction descriptor for the block-scaled kind::mxf8f6f4 (the PTX ISA's
// instruction-descriptor table for the block-scaled kinds; the accumulator is
// always f32): bits 4-5 B scale-factor ID, 7-9 A format and 10-12 B format
// (0 = e4m3, 1 = e5m2, 5 = e2m1), 15 / 16 A / B major-ness (0 = K-major), 17-22 N >> 3,
// 23 scale type (1 = E8M0), 24-28 M >> 4, 29-30 A scale-factor ID. Dense, no
// negation. A scale-factor ID selects the byte of each 32-bit scale cell.
__host__ __device__ constexpr uint32_t idesc_mx_f32(uint32_t fmt, int m, int n, uint32_t a_sf_id,
                                                    uint32_t b_sf_id) {
    return ((b_sf_id & 3u) << 4) | ((fmt & 7u) << 7) | ((fmt & 7u) << 10) |
           (uint32_t(n >> 3) << 17) | (1u << 23) | (uint32_t(m >> 4) << 24) |
           ((a_sf_id & 3u) << 29);
}

// ------------------------------------------------------- warp-level mma.sync
template <bool BF16>
__device__ __forceinline__ void mma_m16n8k16(float (&d)[4], const uint32_t (&a)[4],
                                             uint32_t b0, uint32_t b1) {
    if constexpr (BF16) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
            "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    } else {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
            "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
}

template <bool BF16>
__device__ __forceinline__ void mma_m16n8k8(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t b0) {
    if constexpr (BF16) {
        asm volatile(
            "mma.sync.aligned.m16n8k8.row.col.f32.bf16.bf16.f32 "
            "{%0, %1, %2, %3}, {%4, %5}, {%6}, {%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(a1), "r"(b0));
    } else {
        asm volatile(
            "mma.sync.aligned.m16n8k8.row.col.f32.f16.f16.f32 "
            "{%0, %1, %2, %3}, {%4, %5}, {%6}, {%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(a1), "r"(b0));
    }
}

template <bool TRANS>
__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], uint32_t saddr) {
    if constexpr (TRANS) {
        asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                     : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                     : "r"(saddr));
    } else {
        asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                     : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                     : "r"(saddr));
    }
}

// 16-byte global -> shared copy; src_bytes = 0 writes zeros (out-of-range chunk).
__device__ __forceinline__ void cp_async_16(uint32_t saddr, const void* gptr, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(saddr), "l"(gptr),
                 "r"(src_bytes)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

}  // namespace tpg
