// Vectorised global <-> shared copy: planner, round-trip kernel, C-ABI entry
// points.
//
// Follows the gmem_smem path of the vec_auto copy on the page "TVM TIRx CUDA
// 向量化内存拷贝实战：vec_auto 变体的 global↔shared 实现路径（gmem_smem）":
//   - the gate (接受什么输入): a thread count of 1, 32, 128 or a whole CTA, and
//     an element count the threads divide evenly, else a readable rejection
//     rather than a slow scalar copy;
//   - the [outer, threads, vec] partition (算法核心 step 1): the region's
//     elements in the global side's order, thread tid of round f owning the
//     vec consecutive elements starting at (f * threads + tid) * vec;
//   - the widest-first vector width (step 2): 128, 64, 32, 16, 8 bits, the
//     first whose element count divides the contiguous tail and every
//     non-vector stride and both base offsets;
//   - a serial loop of one vector load and one vector store per round (step 3);
//   - a swizzled shared side: the vector stays inside one 16-byte chunk and
//     its address goes through the XOR (swizzle 小节);
//   - unaligned strides or offsets narrow the vector, down to one element
//     (对齐约束的兜底).
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <type_traits>
#include <string>

#include "tpgemm.h"
#include "tpgemm_internal.h"

namespace tpg {
namespace {

constexpr int kMaxSmemBytes = 200 * 1024;

tpgemm_status vc_fail(tpgemm_status s, std::string* why, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    set_error_detail(buf);
    if (why) *why = buf;
    return s;
}

struct VcPlan {
    int vec_bytes = 0;  // bytes per vector (1..16)
    int vec = 0;        // elements per vector
    int64_t outer = 0;  // rounds per thread
    int tail = 0;       // elements of the contiguous tail on both sides
    int smem_bytes = 0; // shared buffer the kernel allocates
};

int swizzle_bytes(tpgemm_cp_swizzle s) {
    switch (s) {
        case TPGEMM_CP_SWIZZLE_32B: return 32;
        case TPGEMM_CP_SWIZZLE_64B: return 64;
        case TPGEMM_CP_SWIZZLE_128B: return 128;
        default: return 0;
    }
}

tpgemm_status vc_plan(const tpgemm_vcopy_desc* dp, VcPlan* p, std::string* why) {
    if (!dp) return vc_fail(TPGEMM_ERR_NULL, why, "null copy description");
    const tpgemm_vcopy_desc& d = *dp;
    if (d.rows <= 0 || d.cols <= 0)
        return vc_fail(TPGEMM_ERR_SHAPE, why, "region %d x %d must be positive", d.rows, d.cols);
    if (d.elem_bytes != 1 && d.elem_bytes != 2 && d.elem_bytes != 4 && d.elem_bytes != 8)
        return vc_fail(TPGEMM_ERR_DTYPE, why, "elem_bytes=%d must be 1, 2, 4 or 8", d.elem_bytes);
    if (!(d.threads == 1 || d.threads == 32 || d.threads == 128 ||
          (d.threads >= 64 && d.threads <= 1024 && d.threads % 32 == 0)))
        return vc_fail(TPGEMM_ERR_SHAPE, why,
                       "threads=%d is not a scope (1 thread, a warp of 32, a warpgroup of 128, "
                       "or a CTA of 64..1024 in whole warps)",
                       d.threads);
    if (d.g_row_stride < d.cols || d.s_row_stride < d.cols)
        return vc_fail(TPGEMM_ERR_SHAPE, why,
                       "row strides (global %lld, shared %d) must be at least the %d columns",
                       (long long)d.g_row_stride, d.s_row_stride, d.cols);
    if (d.g_offset < 0 || d.s_offset < 0)
        return vc_fail(TPGEMM_ERR_SHAPE, why, "offsets must not be negative");
    if (int(d.s_swizzle) < 0 || int(d.s_swizzle) > 3)
        return vc_fail(TPGEMM_ERR_SHAPE, why, "unknown shared swizzle %d", int(d.s_swizzle));
    const int64_t n = int64_t(d.rows) * d.cols;
    if (n % d.threads)
        return vc_fail(TPGEMM_ERR_SHAPE, why,
                       "%lld elements do not divide among %d threads (a poorly shaped copy is "
                       "rejected, not emitted as scalar code)",
                       (long long)n, d.threads);
    const int64_t s_end =
        (int64_t(d.s_offset) + int64_t(d.rows - 1) * d.s_row_stride + d.cols) * d.elem_bytes;
    const int sw = swizzle_bytes(d.s_swizzle);
    const int64_t s_alloc = sw ? (s_end + 8 * sw - 1) / (8 * sw) * (8 * sw)
                               : (s_end + 15) / 16 * 16;
    if (s_alloc > kMaxSmemBytes)
        return vc_fail(TPGEMM_ERR_SHAPE, why, "the shared region needs %lld bytes; at most %d",
                       (long long)s_alloc, kMaxSmemBytes);
    // The contiguous tail: whole rows fuse into one run when both sides are
    // dense along rows, else a tail is one row.
    const bool fused = d.g_row_stride == d.cols && d.s_row_stride == d.cols;
    const int64_t tail = fused ? n : d.cols;
    const int64_t per_thread = n / d.threads;
    p->vec = 0;
    for (int vb = 16; vb >= 1; vb /= 2) {
        if (vb < d.elem_bytes) break;
        const int v = vb / d.elem_bytes;
        if (tail % v || per_thread % v) continue;
        if (!fused && (d.g_row_stride % v || d.s_row_stride % v)) continue;
        if (d.g_offset % v || d.s_offset % v) continue;
        p->vec_bytes = vb;
        p->vec = v;
        break;
    }
    if (p->vec == 0) {
        // elem_bytes = 8 and nothing narrower than the element: one element.
        p->vec = 1;
        p->vec_bytes = d.elem_bytes;
    }
    p->outer = n / (int64_t(d.threads) * p->vec);
    p->tail = int(std::min<int64_t>(tail, 1 << 30));
    p->smem_bytes = int(s_alloc);
    return TPGEMM_OK;
}

struct VcKernelParams {
    int rows, cols, elem_bytes, threads, vec;
    int outer;           // rounds per thread
    int step_r, step_c;  // divmod(threads * vec, cols)
    int64_t g_row_stride, g_offset, cta_stride;
    int s_row_stride, s_offset, swizzle_mask;  // mask of the 16-byte chunk XOR (0: none)
    int smem_bytes;
};

template <int VB>
struct VecT;
template <>
struct VecT<16> {
    using T = uint4;
};
template <>
struct VecT<8> {
    using T = uint2;
};
template <>
struct VecT<4> {
    using T = uint32_t;
};
template <>
struct VecT<2> {
    using T = uint16_t;
};
template <>
struct VecT<1> {
    using T = uint8_t;
};

// Thread tid's vectors start at fused elements e = (f T + tid) v, f = 0, 1, ...
// The region fits in shared memory, so e, its row r = e / cols and its column
// c = e % cols are 32-bit; one division places the first vector and each later
// one moves (r, c) on by (step_r, step_c) = divmod(T v, cols) with one carry.
struct VcCursor {
    int r, c;
    __device__ __forceinline__ void advance(const VcKernelParams& p) {
        r += p.step_r;
        c += p.step_c;
        if (c >= p.cols) {
            c -= p.cols;
            ++r;
        }
    }
    // Byte offset in global memory (from this CTA's region base).
    __device__ __forceinline__ int64_t global(const VcKernelParams& p) const {
        return (p.g_offset + int64_t(r) * p.g_row_stride + c) * p.elem_bytes;
    }
    // Byte offset in shared memory, after the 16-byte chunk XOR.
    __device__ __forceinline__ uint32_t shared(const VcKernelParams& p) const {
        const uint32_t a = uint32_t((p.s_offset + r * p.s_row_stride + c) * p.elem_bytes);
        return a ^ (((a >> 7) & uint32_t(p.swizzle_mask)) << 4);
    }
};

// global -> shared -> global for this CTA's region; with smem_out, the shared
// buffer (zeroed first, so bytes outside the region are defined) is written out
// between the two copies. Rounds go in batches of kBatch: all of a batch's loads
// are issued before its stores, so each thread keeps kBatch vectors in flight.
template <int VB, int kBatch, int kMaxThreads>
__global__ void __launch_bounds__(kMaxThreads)
    vcopy_kernel(uint8_t* __restrict__ dst, const uint8_t* __restrict__ src,
                 uint8_t* __restrict__ smem_out, const VcKernelParams p) {
    using T = typename VecT<VB>::T;
    extern __shared__ __align__(1024) uint8_t smem[];
    const int tid = threadIdx.x;
    const int64_t base = int64_t(blockIdx.x) * p.cta_stride * p.elem_bytes;
    if (smem_out) {
        for (int i = tid; i < p.smem_bytes / 16; i += p.threads)
            reinterpret_cast<uint4*>(smem)[i] = make_uint4(0, 0, 0, 0);
        __syncthreads();
    }
    VcCursor first;
    first.r = tid * p.vec / p.cols;
    first.c = tid * p.vec - first.r * p.cols;
    VcCursor at = first;
    for (int f0 = 0; f0 < p.outer; f0 += kBatch) {
        T v[kBatch];
        uint32_t so[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            if (f0 + u < p.outer) {
                so[u] = at.shared(p);
                v[u] = *reinterpret_cast<const T*>(src + base + at.global(p));
                at.advance(p);
            }
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u)
            if (f0 + u < p.outer) *reinterpret_cast<T*>(smem + so[u]) = v[u];
    }
    __syncthreads();
    if (smem_out) {
        uint4* o = reinterpret_cast<uint4*>(smem_out + size_t(blockIdx.x) * p.smem_bytes);
        for (int i = tid; i < p.smem_bytes / 16; i += p.threads)
            o[i] = reinterpret_cast<const uint4*>(smem)[i];
    }
    at = first;
    for (int f0 = 0; f0 < p.outer; f0 += kBatch) {
        T v[kBatch];
        int64_t go[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            if (f0 + u < p.outer) {
                go[u] = at.global(p);
                v[u] = *reinterpret_cast<const T*>(smem + at.shared(p));
                at.advance(p);
            }
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u)
            if (f0 + u < p.outer) *reinterpret_cast<T*>(dst + base + go[u]) = v[u];
    }
}

}  // namespace
}  // namespace tpg

extern "C" {

tpgemm_status tpgemm_vcopy_plan(const tpgemm_vcopy_desc* d, char* buf, int buflen) {
    using namespace tpg;
    set_error_detail("");
    VcPlan p;
    std::string why;
    tpgemm_status s = vc_plan(d, &p, &why);
    char text[256];
    if (s == TPGEMM_OK)
        snprintf(text, sizeof(text), "vec_bytes=%d vec=%d outer=%lld threads=%d tail=%d smem=%d",
                 p.vec_bytes, p.vec, (long long)p.outer, d->threads, p.tail, p.smem_bytes);
    if (buf && buflen > 0) {
        strncpy(buf, s == TPGEMM_OK ? text : why.c_str(), size_t(buflen) - 1);
        buf[buflen - 1] = '\0';
    }
    return s;
}

tpgemm_status tpgemm_vcopy_roundtrip(void* dst, const void* src, size_t buffer_bytes,
                                     const tpgemm_vcopy_desc* d, int ctas, int64_t cta_stride,
                                     void* smem_out, void* stream) {
    using namespace tpg;
    set_error_detail("");
    if (!dst || !src) return vc_fail(TPGEMM_ERR_NULL, nullptr, "null device pointer");
    if ((reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(src) |
         reinterpret_cast<uintptr_t>(smem_out)) & 15)
        return vc_fail(TPGEMM_ERR_ALIGN, nullptr, "device pointers must be 16-byte aligned");
    if (dst == src) return vc_fail(TPGEMM_ERR_ALIAS, nullptr, "dst and src must differ");
    VcPlan p;
    tpgemm_status s = vc_plan(d, &p, nullptr);
    if (s != TPGEMM_OK) return s;
    if (ctas < 1 || ctas > (1 << 24))
        return vc_fail(TPGEMM_ERR_SHAPE, nullptr, "ctas=%d must be in 1..2^24", ctas);
    if (cta_stride < 0 || (ctas > 1 && cta_stride % p.vec))
        return vc_fail(TPGEMM_ERR_SHAPE, nullptr,
                       "cta_stride=%lld must be a non-negative multiple of the %d-element vector",
                       (long long)cta_stride, p.vec);
    const int64_t last = (int64_t(ctas - 1) * cta_stride + d->g_offset +
                          int64_t(d->rows - 1) * d->g_row_stride + d->cols) *
                         d->elem_bytes;
    if (uint64_t(last) > buffer_bytes)
        return vc_fail(TPGEMM_ERR_SHAPE, nullptr,
                       "the regions reach byte %lld of %zu-byte buffers", (long long)last,
                       buffer_bytes);
    VcKernelParams kp;
    std::memset(&kp, 0, sizeof(kp));
    kp.rows = d->rows;
    kp.cols = d->cols;
    kp.elem_bytes = d->elem_bytes;
    kp.threads = d->threads;
    kp.vec = p.vec;
    kp.outer = int(p.outer);
    kp.step_r = d->threads * p.vec / d->cols;
    kp.step_c = d->threads * p.vec % d->cols;
    kp.g_row_stride = d->g_row_stride;
    kp.g_offset = d->g_offset;
    kp.cta_stride = cta_stride;
    kp.s_row_stride = d->s_row_stride;
    kp.s_offset = d->s_offset;
    const int sw = swizzle_bytes(d->s_swizzle);
    kp.swizzle_mask = sw ? sw / 16 - 1 : 0;
    kp.smem_bytes = p.smem_bytes;
    auto* so = static_cast<uint8_t*>(smem_out);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    auto* o = static_cast<uint8_t*>(dst);
    auto* i = static_cast<const uint8_t*>(src);
    cudaError_t e = cudaSuccess;
    auto launch = [&](auto kernel) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 p.smem_bytes);
        if (e == cudaSuccess) {
            kernel<<<ctas, d->threads, p.smem_bytes, st>>>(o, i, so, kp);
            e = cudaGetLastError();
        }
    };
    auto dispatch = [&](auto small) {
        constexpr bool S = decltype(small)::value;
        constexpr int B = S ? 8 : 4, T = S ? 256 : 1024;
        switch (p.vec_bytes) {
            case 16: launch(vcopy_kernel<16, B, T>); break;
            case 8: launch(vcopy_kernel<8, B, T>); break;
            case 4: launch(vcopy_kernel<4, B, T>); break;
            case 2: launch(vcopy_kernel<2, B, T>); break;
            default: launch(vcopy_kernel<1, B, T>); break;
        }
    };
    if (d->threads <= 256)
        dispatch(std::true_type{});
    else
        dispatch(std::false_type{});
    if (e != cudaSuccess)
        return vc_fail(TPGEMM_ERR_LAUNCH, nullptr, "copy kernel launch: %s", cudaGetErrorString(e));
    return TPGEMM_OK;
}

}  // extern "C"
