// Shared memory -> tensor memory copies (tcgen05.cp): the host planner, a
// round-trip kernel, and their C-ABI entry points.
//
// Follows the smem-tmem variant of copy_async on the page "TVM Blackwell
// tcgen05.cp 全解析":
//   - the six shape / multicast forms and the multicast each form requires
//     (section 形状选择), parsed with the same rejections;
//   - each form's row -> lane and replica pattern (形状 → 行/复制模式映射表);
//   - widest-first inference over the page's candidate order;
//   - one shared-memory matrix descriptor encoded per copy with only its 14-bit
//     start address patched for each instruction, and the issue loop over the
//     region's row tiles and column steps (调度算法四步, steps 3 and 4);
//   - single-thread issue, completion by a caller-side tcgen05.commit to an
//     mbarrier, read-back with tcgen05.ld (演示程序);
//   - the page's negative checks as readable errors (负向校验).
// The round trip follows the page's GPU test method (测试矩阵): a known image in
// shared memory, the planned copy, and every warp reading its 32-lane slab.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "ptx.cuh"
#include "tpgemm.h"
#include "tpgemm_internal.h"

namespace tpg {

__device__ int g_cp_status;  // 0 = ok, kStatusTimeout after an expired wait

namespace {

constexpr int kMaxCpInstr = 256;
constexpr uint32_t kMaxImageBytes = 196608;
constexpr int kCpThreads = 256;  // 8 warps: up to 8 issuers; warps 0..3 hold the lane quadrants

struct Form {
    const char* name;
    int rows;  // rows one instruction copies
    int bits;  // bits of each of those rows
    tpgemm_cp_lanes lanes;
};

// Indexed by tpgemm_cp_shape; entries 1..6 are also the inference order.
const Form kForms[7] = {
    {"auto", 0, 0, TPGEMM_CP_LANES_ROWS},
    {"128x256b", 128, 256, TPGEMM_CP_LANES_ROWS},
    {"4x256b", 4, 256, TPGEMM_CP_LANES_QUADRANTS},
    {"128x128b", 128, 128, TPGEMM_CP_LANES_ROWS},
    {"64x128b.warpx2::02_13", 64, 128, TPGEMM_CP_LANES_PAIRS_02_13},
    {"64x128b.warpx2::01_23", 64, 128, TPGEMM_CP_LANES_PAIRS_01_23},
    {"32x128b.warpx4", 32, 128, TPGEMM_CP_LANES_ALL_QUADS},
};

const char* lanes_text(tpgemm_cp_lanes l) {
    switch (l) {
        case TPGEMM_CP_LANES_ROWS: return "row r -> lane r";
        case TPGEMM_CP_LANES_QUADRANTS: return "row 4i+q -> lane 32q+i";
        case TPGEMM_CP_LANES_PAIRS_02_13: return "row r -> lanes r, r+64";
        case TPGEMM_CP_LANES_PAIRS_01_23: return "row r -> lanes (r%32)+64(r/32) + {0,32}";
        case TPGEMM_CP_LANES_ALL_QUADS: return "row r -> lanes r + {0,32,64,96}";
    }
    return "?";
}

tpgemm_status cp_fail(tpgemm_status s, std::string* why, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    set_error_detail(buf);
    if (why) *why = buf;
    return s;
}

struct CpPlan {
    int form = 0;
    int n = 0;
    uint64_t desc = 0;      // descriptor template (start address 0)
    uint32_t max_byte = 0;  // one past the last shared-memory byte the copy reads
    int last_col = 0;       // one past the last tensor-memory column written
    uint32_t smem_off[kMaxCpInstr];
    uint32_t taddr[kMaxCpInstr];  // lane << 16 | column, relative to the allocation
};

// Bytes per row of the swizzle pattern (16 for the unswizzled core matrix).
uint32_t row_stride(tpgemm_cp_swizzle s) {
    switch (s) {
        case TPGEMM_CP_SWIZZLE_32B: return 32;
        case TPGEMM_CP_SWIZZLE_64B: return 64;
        case TPGEMM_CP_SWIZZLE_128B: return 128;
        default: return 16;
    }
}

// Layout-type field (bits 61-63) of the shared-memory matrix descriptor.
uint32_t layout_code(tpgemm_cp_swizzle s) {
    switch (s) {
        case TPGEMM_CP_SWIZZLE_32B: return kDescLayoutSw32;
        case TPGEMM_CP_SWIZZLE_64B: return kDescLayoutSw64;
        case TPGEMM_CP_SWIZZLE_128B: return kDescLayoutSw128;
        default: return kDescLayoutNone;
    }
}

// Byte offset, before swizzling, of 16-byte unit u of row r of the region:
// 8-row groups SBO apart; unswizzled, a row's units LBO apart; swizzled, a row
// holds S / 16 consecutive units and the next S / 16 continue in the next
// swizzle atom, LBO further on.
uint64_t unit_offset(const tpgemm_cp_desc& d, int r, int u) {
    const uint64_t group = uint64_t(r / 8) * d.sbo_bytes;
    if (d.swizzle == TPGEMM_CP_SWIZZLE_NONE)
        return d.smem_offset + group + uint64_t(r % 8) * 16 + uint64_t(u) * d.lbo_bytes;
    const uint32_t S = row_stride(d.swizzle);
    const int per_row = int(S / 16);
    return d.smem_offset + uint64_t(u / per_row) * d.lbo_bytes + group + uint64_t(r % 8) * S +
           16ull * uint64_t(u % per_row);
}

// Where a byte offset lands once the swizzle is applied (offsets from a
// 1024-byte aligned buffer): bits [4, 4 + b) XOR bits [7, 7 + b).
uint64_t swizzle_offset(uint64_t a, tpgemm_cp_swizzle s) {
    if (s == TPGEMM_CP_SWIZZLE_NONE) return a;
    const uint64_t mask = row_stride(s) / 16 - 1;
    return a ^ (((a >> 7) & mask) << 4);
}

bool form_fits(int f, const tpgemm_cp_desc& d, std::string* why) {
    const Form& F = kForms[f];
    if (F.lanes != d.lanes) {
        if (why)
            *why = std::string("replica mismatch: ") + F.name + " places " + lanes_text(F.lanes) +
                   ", the destination asks for " + lanes_text(d.lanes);
        return false;
    }
    char buf[256];
    if (d.row_bits % F.bits) {
        snprintf(buf, sizeof(buf), "a %d-bit row is not a whole number of %s's %d-bit rows",
                 d.row_bits, F.name, F.bits);
        if (why) *why = buf;
        return false;
    }
    if (F.lanes == TPGEMM_CP_LANES_QUADRANTS) {
        if (d.rows % 4) {
            snprintf(buf, sizeof(buf), "%s tiles rows by 4; the region has %d rows", F.name,
                     d.rows);
            if (why) *why = buf;
            return false;
        }
        if (d.lane_offset + d.rows / 4 > 32) {
            snprintf(buf, sizeof(buf),
                     "%d rows from lane offset %d overflow the 128-lane space (%s fills lanes "
                     "32q + offset .. 32q + offset + rows/4 - 1)",
                     d.rows, d.lane_offset, F.name);
            if (why) *why = buf;
            return false;
        }
        return true;
    }
    if (d.rows != F.rows) {
        snprintf(buf, sizeof(buf), "%s copies exactly %d rows; the region has %d", F.name, F.rows,
                 d.rows);
        if (why) *why = buf;
        return false;
    }
    if (d.lane_offset != 0) {
        snprintf(buf, sizeof(buf), "lane offset %d overflows the 128-lane space for %s",
                 d.lane_offset, F.name);
        if (why) *why = buf;
        return false;
    }
    return true;
}

tpgemm_status build_plan(const tpgemm_cp_desc* dp, CpPlan* plan, std::string* why) {
    if (!dp) return cp_fail(TPGEMM_ERR_NULL, why, "null copy description");
    const tpgemm_cp_desc& d = *dp;
    if (d.rows <= 0 || d.rows > 128)
        return cp_fail(TPGEMM_ERR_SHAPE, why, "rows=%d must be in 1..128", d.rows);
    if (d.row_bits <= 0 || d.row_bits % 128)
        return cp_fail(TPGEMM_ERR_SHAPE, why, "row_bits=%d is not a positive multiple of 128",
                       d.row_bits);
    if (int(d.swizzle) < 0 || int(d.swizzle) > 3)
        return cp_fail(TPGEMM_ERR_SHAPE, why, "unknown swizzle mode %d", int(d.swizzle));
    if (int(d.lanes) < 0 || int(d.lanes) > 4)
        return cp_fail(TPGEMM_ERR_SHAPE, why, "unknown lane pattern %d", int(d.lanes));
    if (int(d.shape) < 0 || int(d.shape) > 6)
        return cp_fail(TPGEMM_ERR_SHAPE, why, "unknown tcgen05.cp shape %d", int(d.shape));
    if (d.cta_group != 1 && d.cta_group != 2)
        return cp_fail(TPGEMM_ERR_SHAPE, why, "cta_group=%d must be 1 or 2", d.cta_group);
    if (d.tmem_col < 0 || d.tmem_col % 4)
        return cp_fail(TPGEMM_ERR_SHAPE, why,
                       "tensor-memory column offset %d is not 128b-aligned (a multiple of 4)",
                       d.tmem_col);
    if (d.lane_offset < 0 || d.lane_offset >= 128)
        return cp_fail(TPGEMM_ERR_SHAPE, why, "lane offset %d overflows the 128-lane space",
                       d.lane_offset);
    if (d.sbo_bytes % 16 || d.sbo_bytes >= (1u << 18))
        return cp_fail(TPGEMM_ERR_SHAPE, why,
                       "row-group stride (SBO) of %u bytes is not 16B-aligned or exceeds the "
                       "descriptor's 14-bit field",
                       d.sbo_bytes);
    const uint32_t S = row_stride(d.swizzle);
    if (d.lbo_bytes % 16 || d.lbo_bytes >= (1u << 18))
        return cp_fail(TPGEMM_ERR_SHAPE, why,
                       "unit / atom stride (LBO) of %u bytes is not 16B-aligned or exceeds the "
                       "descriptor's 14-bit field",
                       d.lbo_bytes);
    if (d.swizzle == TPGEMM_CP_SWIZZLE_NONE) {
        if (d.smem_offset % 16)
            return cp_fail(TPGEMM_ERR_SHAPE, why, "region start %u is not 16B-aligned",
                           d.smem_offset);
    } else {
        if (d.smem_offset % (8 * S))
            return cp_fail(TPGEMM_ERR_SHAPE, why,
                           "region start %u is not aligned to the %u-byte swizzle atom",
                           d.smem_offset, 8 * S);
        if (uint32_t(d.row_bits) > 8 * S && d.lbo_bytes % (8 * S))
            return cp_fail(TPGEMM_ERR_SHAPE, why,
                           "a %d-bit row spans several %u-byte swizzle rows; the atom stride "
                           "(LBO) %u must be a positive multiple of the %u-byte swizzle atom",
                           d.row_bits, S, d.lbo_bytes, 8 * S);
    }
    // The form: explicit, or the first candidate (widest first) that fits.
    int f = int(d.shape);
    std::string reason;
    if (f == TPGEMM_CP_AUTO) {
        std::string first_reason;
        for (int c = 1; c <= 6 && f == 0; ++c) {
            std::string r;
            if (form_fits(c, d, &r))
                f = c;
            else if (kForms[c].lanes == d.lanes && first_reason.empty())
                first_reason = r;
        }
        if (f == 0)
            return cp_fail(TPGEMM_ERR_SHAPE, why, "no tcgen05.cp form fits the region: %s",
                           first_reason.empty() ? "no form has this lane pattern"
                                                : first_reason.c_str());
    } else if (!form_fits(f, d, &reason)) {
        return cp_fail(TPGEMM_ERR_SHAPE, why, "%s", reason.c_str());
    }
    const Form& F = kForms[f];
    const int tiles = F.lanes == TPGEMM_CP_LANES_QUADRANTS ? d.rows / 4 : 1;
    const int steps = d.row_bits / F.bits;
    if (tiles * steps > kMaxCpInstr)
        return cp_fail(TPGEMM_ERR_SHAPE, why, "the copy needs %d instructions; at most %d",
                       tiles * steps, kMaxCpInstr);
    plan->form = f;
    plan->n = 0;
    // Swizzled K-major rows: the descriptor's LBO field is not used within one
    // swizzle row (every instruction stays inside one); it is set to 16 bytes.
    const uint32_t lbo = d.swizzle == TPGEMM_CP_SWIZZLE_NONE ? d.lbo_bytes : 16;
    plan->desc = smem_desc_template(lbo, d.sbo_bytes, layout_code(d.swizzle));
    for (int i = 0; i < tiles; ++i) {
        for (int s = 0; s < steps; ++s) {
            const int r0 = tiles > 1 ? 4 * i : 0;
            const int u0 = s * (F.bits / 128);
            const int lane = d.lane_offset + (F.lanes == TPGEMM_CP_LANES_QUADRANTS ? i : 0);
            const int col = d.tmem_col + s * (F.bits / 32);
            plan->smem_off[plan->n] = uint32_t(unit_offset(d, r0, u0));
            plan->taddr[plan->n] = (uint32_t(lane) << 16) | uint32_t(col);
            ++plan->n;
        }
    }
    // Where every unit of the region lives; two units on the same bytes mean
    // the strides overlap (a layout the copy cannot read as described).
    uint64_t hi = 0;
    std::vector<uint64_t> at;
    at.reserve(size_t(d.rows) * size_t(d.row_bits / 128));
    for (int r = 0; r < d.rows; ++r)
        for (int u = 0; u < d.row_bits / 128; ++u) {
            at.push_back(swizzle_offset(unit_offset(d, r, u), d.swizzle));
            hi = std::max(hi, at.back() + 16);
        }
    std::sort(at.begin(), at.end());
    for (size_t i = 1; i < at.size(); ++i)
        if (at[i] == at[i - 1])
            return cp_fail(TPGEMM_ERR_SHAPE, why,
                           "the layout maps two 16-byte units to shared-memory offset %llu "
                           "(LBO %u, SBO %u overlap)",
                           (unsigned long long)at[i], d.lbo_bytes, d.sbo_bytes);
    if (hi > kMaxImageBytes)
        return cp_fail(TPGEMM_ERR_SHAPE, why,
                       "the region reaches byte %llu, beyond the %u-byte staging buffer",
                       (unsigned long long)hi, kMaxImageBytes);
    plan->max_byte = uint32_t(hi);
    plan->last_col = d.tmem_col + d.row_bits / 32;
    return TPGEMM_OK;
}

// ------------------------------------------------------------------ kernel
struct CpKernelParams {
    uint64_t desc;
    uint64_t timeout_ns;
    uint32_t image_words;  // 16-byte words of one CTA's image
    uint32_t fill_base;
    int n, form, ncols, alloc_cols;
    int repeat;   // times the whole instruction list is issued before the commit
    int issuers;  // threads (lane 0 of warps 0..issuers-1) sharing the list, each committing
    uint32_t smem_off[kMaxCpInstr];
    uint32_t taddr[kMaxCpInstr];
};

__device__ __forceinline__ bool cp_wait(uint64_t* bar, uint64_t timeout_ns) {
    if (mbar_try_wait(bar, 0)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, 0))
        if (globaltimer_ns() - t0 > timeout_ns) return false;
    return true;
}

template <int CG>
__global__ void __launch_bounds__(kCpThreads, 1)
    cp_roundtrip_kernel(uint32_t* __restrict__ out, const uint4* __restrict__ image,
                        const __grid_constant__ CpKernelParams p) {
    extern __shared__ uint8_t raw[];
    __shared__ uint64_t bar;
    __shared__ uint32_t tmem_base;
    uint8_t* buf = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) &
                                              ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int rank = CG == 2 ? int(cluster_ctarank()) : 0;
    // CTA pairs: each CTA of a pair has its own image; all pairs (or all single
    // CTAs) share the images and write their own rows of out.

    if (warp == 0) {
        tmem_alloc<CG>(&tmem_base, uint32_t(p.alloc_cols));
        tmem_relinquish_alloc_permit<CG>();
    }
    if (threadIdx.x == 0) {
        mbar_init(&bar, uint32_t(p.issuers));
        fence_mbarrier_init();
    }
    // The image, with 16-byte loads and stores; then made visible to the async
    // proxy that tcgen05.cp reads through.
    const uint4* src = image + size_t(CG == 2 ? rank : 0) * p.image_words;
    uint4* dst = reinterpret_cast<uint4*>(buf);
    for (uint32_t i = threadIdx.x; i < p.image_words; i += kCpThreads) dst[i] = src[i];
    fence_proxy_async_smem();
    tc_fence_before_sync();
    if (CG == 2)
        cluster_sync();
    else
        __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = tmem_base;
    // Warps 0..3 reach tensor-memory lane quadrants 0..3; warps 4..7 only
    // stage the image and issue.
    const bool quad_warp = warp < 4;
    const uint32_t lane_base = uint32_t(warp * 32) << 16;
    const uint32_t row = uint32_t(warp * 32 + lane);

    // Every column that is read back starts from a known value.
    if (quad_warp) {
        for (int c = 0; c < p.ncols; c += 8) {
            uint32_t v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] = p.fill_base + row * 65536u + uint32_t(c + j);
            tmem_st_32x32b_x8(tmem + lane_base + uint32_t(c), v);
        }
        tmem_st_wait();
    }
    tc_fence_before_sync();
    if (CG == 2)
        cluster_sync();
    else
        __syncthreads();
    tc_fence_after_sync();

    // One thread issues the planned instructions and commits them (the page's
    // protocol); with issuers > 1, lane 0 of each of the first `issuers` warps
    // takes every issuers-th instruction and commits its own.
    if (lane == 0 && warp < p.issuers && rank == 0) {
        const uint32_t base = smem_u32(buf);
        for (int k = 0; k < p.repeat; ++k)
            for (int i = warp; i < p.n; i += p.issuers)
                tc_cp<CG>(p.form, tmem + p.taddr[i],
                          smem_desc_with_addr(p.desc, base + p.smem_off[i]));
        if (CG == 2)
            tc_commit_pair_multicast(&bar, 0x3);
        else
            tc_commit(&bar);
    }
    bool ok = cp_wait(&bar, p.timeout_ns);
    if (!ok) {
        atomicExch(&g_cp_status, kStatusTimeout);
        ok = cp_wait(&bar, p.timeout_ns);  // let the copies finish before dealloc
    }
    tc_fence_after_sync();
    if (ok && quad_warp) {
        uint32_t* o = out + (size_t(blockIdx.x) * 128 + row) * size_t(p.ncols);
        for (int c = 0; c < p.ncols; c += 8) {
            uint32_t v[8];
            tmem_ld_32x32b_x8(tmem + lane_base + uint32_t(c), v);
            reinterpret_cast<uint4*>(o + c)[0] = make_uint4(v[0], v[1], v[2], v[3]);
            reinterpret_cast<uint4*>(o + c)[1] = make_uint4(v[4], v[5], v[6], v[7]);
        }
    }
    tc_fence_before_sync();
    if (CG == 2)
        cluster_sync();
    else
        __syncthreads();
    if (warp == 0) {
        tc_fence_after_sync();
        tmem_dealloc<CG>(tmem, uint32_t(p.alloc_cols));
    }
}

// ---------------------------------------------- tensor memory <-> registers
// The tmem<->local copy of the page "TVM TIRx copy_async -> tcgen05_ldst": a
// warpgroup moves a 128-lane x C-column tile between tensor memory and its
// registers (C per thread). .32x32b covers a warp's 32 lanes in one issue;
// the .16x{64,128,256}b shapes cover 16 lanes, so each warp issues them twice
// (lanes +0 and +16, section Algorithm step 3), registers [0, C/2) for the
// first slab and [C/2, C) for the second.
template <int C>
__device__ __forceinline__ void ldst_store(int shape, uint32_t taddr, const uint32_t (&v)[C]) {
    const uint32_t s16 = 16u << 16;
    if constexpr (C == 2) {
        if (shape == TPGEMM_TMEM_32x32b) TPG_TMEM_ST("32x32b.x2", 2, taddr, v);
        if (shape == TPGEMM_TMEM_16x64b) {
            TPG_TMEM_ST("16x64b.x1", 1, taddr, v);
            TPG_TMEM_ST("16x64b.x1", 1, taddr + s16, v + 1);
        }
    } else if constexpr (C == 4) {
        if (shape == TPGEMM_TMEM_32x32b) TPG_TMEM_ST("32x32b.x4", 4, taddr, v);
        if (shape == TPGEMM_TMEM_16x64b) {
            TPG_TMEM_ST("16x64b.x2", 2, taddr, v);
            TPG_TMEM_ST("16x64b.x2", 2, taddr + s16, v + 2);
        }
        if (shape == TPGEMM_TMEM_16x128b) {
            TPG_TMEM_ST("16x128b.x1", 2, taddr, v);
            TPG_TMEM_ST("16x128b.x1", 2, taddr + s16, v + 2);
        }
    } else if constexpr (C == 8) {
        if (shape == TPGEMM_TMEM_32x32b) TPG_TMEM_ST("32x32b.x8", 8, taddr, v);
        if (shape == TPGEMM_TMEM_16x64b) {
            TPG_TMEM_ST("16x64b.x4", 4, taddr, v);
            TPG_TMEM_ST("16x64b.x4", 4, taddr + s16, v + 4);
        }
        if (shape == TPGEMM_TMEM_16x128b) {
            TPG_TMEM_ST("16x128b.x2", 4, taddr, v);
            TPG_TMEM_ST("16x128b.x2", 4, taddr + s16, v + 4);
        }
        if (shape == TPGEMM_TMEM_16x256b) {
            TPG_TMEM_ST("16x256b.x1", 4, taddr, v);
            TPG_TMEM_ST("16x256b.x1", 4, taddr + s16, v + 4);
        }
    } else {
        static_assert(C == 16, "C is 2, 4, 8 or 16");
        if (shape == TPGEMM_TMEM_32x32b) TPG_TMEM_ST("32x32b.x16", 16, taddr, v);
        if (shape == TPGEMM_TMEM_16x64b) {
            TPG_TMEM_ST("16x64b.x8", 8, taddr, v);
            TPG_TMEM_ST("16x64b.x8", 8, taddr + s16, v + 8);
        }
        if (shape == TPGEMM_TMEM_16x128b) {
            TPG_TMEM_ST("16x128b.x4", 8, taddr, v);
            TPG_TMEM_ST("16x128b.x4", 8, taddr + s16, v + 8);
        }
        if (shape == TPGEMM_TMEM_16x256b) {
            TPG_TMEM_ST("16x256b.x2", 8, taddr, v);
            TPG_TMEM_ST("16x256b.x2", 8, taddr + s16, v + 8);
        }
    }
}

template <int C>
__device__ __forceinline__ void ldst_load(int shape, uint32_t taddr, uint32_t (&v)[C]) {
    const uint32_t s16 = 16u << 16;
    if constexpr (C == 2) {
        if (shape == TPGEMM_TMEM_32x32b) TPG_TMEM_LD("32x32b.x2", 2, taddr, v);
        if (shape == TPGEMM_TMEM_16x64b) {
            TPG_TMEM_LD("16x64b.x1", 1, taddr, v);
            TPG_TMEM_LD("16x64b.x1", 1, taddr + s16, v + 1);
        }
    } else if constexpr (C == 4) {
        if (shape == TPGEMM_TMEM_32x32b) TPG_TMEM_LD("32x32b.x4", 4, taddr, v);
        if (shape == TPGEMM_TMEM_16x64b) {
            TPG_TMEM_LD("16x64b.x2", 2, taddr, v);
            TPG_TMEM_LD("16x64b.x2", 2, taddr + s16, v + 2);
        }
        if (shape == TPGEMM_TMEM_16x128b) {
            TPG_TMEM_LD("16x128b.x1", 2, taddr, v);
            TPG_TMEM_LD("16x128b.x1", 2, taddr + s16, v + 2);
        }
    } else if constexpr (C == 8) {
        if (shape == TPGEMM_TMEM_32x32b) TPG_TMEM_LD("32x32b.x8", 8, taddr, v);
        if (shape == TPGEMM_TMEM_16x64b) {
            TPG_TMEM_LD("16x64b.x4", 4, taddr, v);
            TPG_TMEM_LD("16x64b.x4", 4, taddr + s16, v + 4);
        }
        if (shape == TPGEMM_TMEM_16x128b) {
            TPG_TMEM_LD("16x128b.x2", 4, taddr, v);
            TPG_TMEM_LD("16x128b.x2", 4, taddr + s16, v + 4);
        }
        if (shape == TPGEMM_TMEM_16x256b) {
            TPG_TMEM_LD("16x256b.x1", 4, taddr, v);
            TPG_TMEM_LD("16x256b.x1", 4, taddr + s16, v + 4);
        }
    } else {
        if (shape == TPGEMM_TMEM_32x32b) TPG_TMEM_LD("32x32b.x16", 16, taddr, v);
        if (shape == TPGEMM_TMEM_16x64b) {
            TPG_TMEM_LD("16x64b.x8", 8, taddr, v);
            TPG_TMEM_LD("16x64b.x8", 8, taddr + s16, v + 8);
        }
        if (shape == TPGEMM_TMEM_16x128b) {
            TPG_TMEM_LD("16x128b.x4", 8, taddr, v);
            TPG_TMEM_LD("16x128b.x4", 8, taddr + s16, v + 8);
        }
        if (shape == TPGEMM_TMEM_16x256b) {
            TPG_TMEM_LD("16x256b.x2", 8, taddr, v);
            TPG_TMEM_LD("16x256b.x2", 8, taddr + s16, v + 8);
        }
    }
    tmem_ld_wait_all();
}

constexpr int kLdstCols = 32;  // tensor-memory columns allocated and read back

// One warpgroup: fill columns [0, 32) of all 128 lanes with a known pattern,
// store the C registers of every thread with st_shape at column tmem_col, read
// all 32 columns back with .32x32b into tmem_out, then load with ld_shape into
// regs_out.
template <int C>
__global__ void __launch_bounds__(128, 1)
    ldst_roundtrip_kernel(uint32_t* __restrict__ regs_out, uint32_t* __restrict__ tmem_out,
                          const uint32_t* __restrict__ regs_in, int st_shape, int ld_shape,
                          int tmem_col, uint32_t fill_base) {
    __shared__ uint32_t tmem_base;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t row = uint32_t(threadIdx.x);
    if (warp == 0) {
        tmem_alloc<1>(&tmem_base, uint32_t(kLdstCols));
        tmem_relinquish_alloc_permit<1>();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t warp_base = tmem_base + (uint32_t(warp * 32) << 16);
    for (int c = 0; c < kLdstCols; c += 8) {
        uint32_t f[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) f[j] = fill_base + row * 65536u + uint32_t(c + j);
        tmem_st_32x32b_x8(warp_base + uint32_t(c), f);
    }
    tmem_st_wait();
    uint32_t v[C];
#pragma unroll
    for (int j = 0; j < C; ++j) v[j] = regs_in[size_t(row) * C + j];
    ldst_store<C>(st_shape, warp_base + uint32_t(tmem_col), v);
    tmem_st_wait();
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    for (int c = 0; c < kLdstCols; c += 8) {
        uint32_t r[8];
        tmem_ld_32x32b_x8(warp_base + uint32_t(c), r);
#pragma unroll
        for (int j = 0; j < 8; ++j) tmem_out[size_t(row) * kLdstCols + c + j] = r[j];
    }
    uint32_t w[C];
    ldst_load<C>(ld_shape, warp_base + uint32_t(tmem_col), w);
#pragma unroll
    for (int j = 0; j < C; ++j) regs_out[size_t(row) * C + j] = w[j];
    (void)lane;
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after_sync();
        tmem_dealloc<1>(tmem_base, uint32_t(kLdstCols));
    }
}

int describe(const tpgemm_cp_desc& d, const CpPlan& pl, char* buf, int buflen) {
    if (!buf || buflen <= 0) return 0;
    std::string t;
    char line[256];
    snprintf(line, sizeof(line),
             "form=%s instructions=%d lbo=%u sbo=%u swizzle=%s desc=0x%016llx last_col=%d "
             "max_byte=%u cta_group=%d",
             kForms[pl.form].name, pl.n, d.lbo_bytes,
             d.sbo_bytes,
             d.swizzle == TPGEMM_CP_SWIZZLE_NONE  ? "none"
             : d.swizzle == TPGEMM_CP_SWIZZLE_32B ? "32B"
             : d.swizzle == TPGEMM_CP_SWIZZLE_64B ? "64B"
                                                  : "128B",
             (unsigned long long)pl.desc, pl.last_col, pl.max_byte, d.cta_group);
    t = line;
    for (int i = 0; i < pl.n; ++i) {
        snprintf(line, sizeof(line), "; [%d] smem=%u lane=%u col=%u", i, pl.smem_off[i],
                 pl.taddr[i] >> 16, pl.taddr[i] & 0xFFFFu);
        t += line;
    }
    strncpy(buf, t.c_str(), size_t(buflen) - 1);
    buf[buflen - 1] = '\0';
    return int(t.size());
}

}  // namespace

cudaError_t cp_read_and_clear_device_status(int* status) {
    cudaError_t e = cudaMemcpyFromSymbol(status, g_cp_status, sizeof(int));
    if (e != cudaSuccess) return e;
    const int zero = 0;
    return cudaMemcpyToSymbol(g_cp_status, &zero, sizeof(int));
}

}  // namespace tpg

extern "C" {

tpgemm_status tpgemm_cp_parse_shape(const char* name, tpgemm_cp_shape* out) {
    using namespace tpg;
    set_error_detail("");
    if (!name || !out) return cp_fail(TPGEMM_ERR_NULL, nullptr, "null argument");
    std::string s(name);
    const size_t dot = s.find('.');
    const std::string shape = s.substr(0, dot);
    const std::string mc = dot == std::string::npos ? "" : s.substr(dot + 1);
    const char* legal = "128x256b, 4x256b, 128x128b, 64x128b, 32x128b";
    if (shape == "128x256b" || shape == "4x256b" || shape == "128x128b") {
        if (!mc.empty())
            return cp_fail(TPGEMM_ERR_SHAPE, nullptr,
                           "illegal multicast '%s' for %s (it takes none)", mc.c_str(),
                           shape.c_str());
        *out = shape == "128x256b" ? TPGEMM_CP_128x256b
               : shape == "4x256b" ? TPGEMM_CP_4x256b
                                   : TPGEMM_CP_128x128b;
        return TPGEMM_OK;
    }
    if (shape == "64x128b") {
        if (mc.empty())
            return cp_fail(TPGEMM_ERR_SHAPE, nullptr,
                           "64x128b requires an explicit multicast config: warpx2::02_13 or "
                           "warpx2::01_23");
        if (mc == "warpx2::02_13") {
            *out = TPGEMM_CP_64x128b_WARPX2_02_13;
            return TPGEMM_OK;
        }
        if (mc == "warpx2::01_23") {
            *out = TPGEMM_CP_64x128b_WARPX2_01_23;
            return TPGEMM_OK;
        }
        return cp_fail(TPGEMM_ERR_SHAPE, nullptr,
                       "illegal multicast '%s' for 64x128b (warpx2::02_13 or warpx2::01_23)",
                       mc.c_str());
    }
    if (shape == "32x128b") {
        if (!mc.empty() && mc != "warpx4")
            return cp_fail(TPGEMM_ERR_SHAPE, nullptr,
                           "illegal multicast '%s' for 32x128b (it requires warpx4)", mc.c_str());
        *out = TPGEMM_CP_32x128b_WARPX4;
        return TPGEMM_OK;
    }
    return cp_fail(TPGEMM_ERR_SHAPE, nullptr, "unknown tcgen05.cp shape '%s' (legal: %s)",
                   shape.c_str(), legal);
}

tpgemm_status tpgemm_cp_plan(const tpgemm_cp_desc* d, char* buf, int buflen) {
    using namespace tpg;
    set_error_detail("");
    static thread_local CpPlan plan;
    std::string why;
    tpgemm_status s = build_plan(d, &plan, &why);
    if (s != TPGEMM_OK) {
        if (buf && buflen > 0) {
            strncpy(buf, why.c_str(), size_t(buflen) - 1);
            buf[buflen - 1] = '\0';
        }
        return s;
    }
    describe(*d, plan, buf, buflen);
    return TPGEMM_OK;
}

tpgemm_status tpgemm_cp_roundtrip(uint32_t* tmem_out, const void* smem_image, size_t image_bytes,
                                  const tpgemm_cp_desc* d, uint32_t fill_base, int ncols,
                                  void* stream) {
    return tpgemm_cp_roundtrip_repeat(tmem_out, smem_image, image_bytes, d, fill_base, ncols, 1,
                                      d ? d->cta_group : 1, 1, stream);
}

tpgemm_status tpgemm_cp_roundtrip_repeat(uint32_t* tmem_out, const void* smem_image,
                                         size_t image_bytes, const tpgemm_cp_desc* d,
                                         uint32_t fill_base, int ncols, int repeat, int ctas,
                                         int issuers, void* stream) {
    using namespace tpg;
    set_error_detail("");
    if (!tmem_out || !smem_image) return cp_fail(TPGEMM_ERR_NULL, nullptr, "null device pointer");
    if ((reinterpret_cast<uintptr_t>(tmem_out) | reinterpret_cast<uintptr_t>(smem_image)) & 15)
        return cp_fail(TPGEMM_ERR_ALIGN, nullptr, "device pointers must be 16-byte aligned");
    if (image_bytes == 0 || image_bytes % 16 || image_bytes > kMaxImageBytes)
        return cp_fail(TPGEMM_ERR_SHAPE, nullptr,
                       "image_bytes=%zu must be a positive multiple of 16, at most %u",
                       image_bytes, kMaxImageBytes);
    if (ncols < 32 || ncols > 512 || ncols % 32)
        return cp_fail(TPGEMM_ERR_SHAPE, nullptr, "ncols=%d must be a multiple of 32 in 32..512",
                       ncols);
    static thread_local CpPlan plan;
    tpgemm_status s = build_plan(d, &plan, nullptr);
    if (s != TPGEMM_OK) return s;
    if (issuers < 1 || issuers > kCpThreads / 32)
        return cp_fail(TPGEMM_ERR_SHAPE, nullptr, "issuers=%d must be 1..%d (one per warp)",
                       issuers, kCpThreads / 32);
    if (repeat < 1 || repeat > (1 << 20))
        return cp_fail(TPGEMM_ERR_SHAPE, nullptr, "repeat=%d must be in 1..2^20", repeat);
    if (ctas < 1 || ctas > 65536 || ctas % d->cta_group)
        return cp_fail(TPGEMM_ERR_SHAPE, nullptr,
                       "ctas=%d must be in 1..65536 and a multiple of cta_group %d", ctas,
                       d->cta_group);
    if (plan.max_byte > image_bytes)
        return cp_fail(TPGEMM_ERR_SHAPE, nullptr,
                       "the copy reads up to byte %u of a %zu-byte image", plan.max_byte,
                       image_bytes);
    if (plan.last_col > ncols)
        return cp_fail(TPGEMM_ERR_SHAPE, nullptr,
                       "the copy writes up to column %d; only %d columns are read back",
                       plan.last_col, ncols);
    int dev = 0, major = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess)
        return cp_fail(TPGEMM_ERR_ARCH, nullptr, "no CUDA device available");
    if (major != 10)
        return cp_fail(TPGEMM_ERR_ARCH, nullptr, "tcgen05 needs compute capability 10.x");

    CpKernelParams kp;
    std::memset(&kp, 0, sizeof(kp));
    kp.desc = plan.desc;
    kp.timeout_ns = wait_timeout_ns();
    kp.image_words = uint32_t(image_bytes / 16);
    kp.fill_base = fill_base;
    kp.n = plan.n;
    kp.repeat = repeat;
    kp.issuers = issuers;
    kp.form = plan.form;
    kp.ncols = ncols;
    kp.alloc_cols = 32;
    while (kp.alloc_cols < ncols) kp.alloc_cols *= 2;
    std::memcpy(kp.smem_off, plan.smem_off, sizeof(uint32_t) * size_t(plan.n));
    std::memcpy(kp.taddr, plan.taddr, sizeof(uint32_t) * size_t(plan.n));

    // A fixed staging buffer, whatever the image: every shared-memory address
    // the planned copy can form stays inside this CTA's allocation.
    const size_t smem = size_t(kMaxImageBytes) + 1024;
    auto kernel = d->cta_group == 2 ? cp_roundtrip_kernel<2> : cp_roundtrip_kernel<1>;
    cudaError_t e =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess)
        return cp_fail(TPGEMM_ERR_LAUNCH, nullptr, "copy kernel attribute: %s",
                       cudaGetErrorString(e));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(ctas));
    cfg.blockDim = dim3(kCpThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = unsigned(d->cta_group);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = d->cta_group == 2 ? 1 : 0;
    e = cudaLaunchKernelEx(&cfg, kernel, tmem_out, static_cast<const uint4*>(smem_image), kp);
    if (e != cudaSuccess)
        return cp_fail(TPGEMM_ERR_LAUNCH, nullptr, "copy kernel launch: %s",
                       cudaGetErrorString(e));
    return TPGEMM_OK;
}

tpgemm_status tpgemm_tmem_ldst_roundtrip(uint32_t* regs_out, uint32_t* tmem_out,
                                        const uint32_t* regs_in, tpgemm_tmem_shape st_shape,
                                        tpgemm_tmem_shape ld_shape, int cols, int tmem_col,
                                        uint32_t fill_base, void* stream) {
    using namespace tpg;
    set_error_detail("");
    if (!regs_out || !tmem_out || !regs_in)
        return cp_fail(TPGEMM_ERR_NULL, nullptr, "null device pointer");
    if ((reinterpret_cast<uintptr_t>(regs_out) | reinterpret_cast<uintptr_t>(tmem_out) |
         reinterpret_cast<uintptr_t>(regs_in)) & 15)
        return cp_fail(TPGEMM_ERR_ALIGN, nullptr, "device pointers must be 16-byte aligned");
    auto min_cols = [](int shape) {
        switch (shape) {
            case TPGEMM_TMEM_32x32b: return 1;
            case TPGEMM_TMEM_16x64b: return 2;
            case TPGEMM_TMEM_16x128b: return 4;
            case TPGEMM_TMEM_16x256b: return 8;
        }
        return 0;
    };
    const char* names[4] = {"32x32b", "16x64b", "16x128b", "16x256b"};
    for (int sh : {int(st_shape), int(ld_shape)}) {
        if (sh < 0 || sh > 3)
            return cp_fail(TPGEMM_ERR_SHAPE, nullptr, "unknown tensor-memory shape %d", sh);
        if (cols < min_cols(sh))
            return cp_fail(TPGEMM_ERR_SHAPE, nullptr,
                           "%s moves at least %d columns per warp; cols=%d", names[sh],
                           min_cols(sh), cols);
    }
    if (cols != 2 && cols != 4 && cols != 8 && cols != 16)
        return cp_fail(TPGEMM_ERR_SHAPE, nullptr, "cols=%d must be 2, 4, 8 or 16", cols);
    if (tmem_col < 0 || tmem_col % 8 || tmem_col + cols > kLdstCols)
        return cp_fail(TPGEMM_ERR_SHAPE, nullptr,
                       "tmem_col=%d must be a multiple of 8 with tmem_col + cols <= %d",
                       tmem_col, kLdstCols);
    int dev = 0, major = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess)
        return cp_fail(TPGEMM_ERR_ARCH, nullptr, "no CUDA device available");
    if (major != 10)
        return cp_fail(TPGEMM_ERR_ARCH, nullptr, "tcgen05 needs compute capability 10.x");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int a = int(st_shape), b = int(ld_shape);
    switch (cols) {
        case 2: ldst_roundtrip_kernel<2><<<1, 128, 0, st>>>(regs_out, tmem_out, regs_in, a, b,
                                                             tmem_col, fill_base); break;
        case 4: ldst_roundtrip_kernel<4><<<1, 128, 0, st>>>(regs_out, tmem_out, regs_in, a, b,
                                                             tmem_col, fill_base); break;
        case 8: ldst_roundtrip_kernel<8><<<1, 128, 0, st>>>(regs_out, tmem_out, regs_in, a, b,
                                                             tmem_col, fill_base); break;
        default: ldst_roundtrip_kernel<16><<<1, 128, 0, st>>>(regs_out, tmem_out, regs_in, a,
                                                               b, tmem_col, fill_base); break;
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return cp_fail(TPGEMM_ERR_LAUNCH, nullptr, "ld/st kernel launch: %s",
                       cudaGetErrorString(e));
    return TPGEMM_OK;
}

}  // extern "C"
