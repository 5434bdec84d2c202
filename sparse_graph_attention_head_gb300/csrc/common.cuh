// common.cuh - internal helpers shared by the libgat translation units.
#pragma once

#include <type_traits>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "gat.h"

namespace gat {

constexpr unsigned kFull = 0xffffffffu;

// ---------------------------------------------------------------------------
// host-side error reporting (thread-local detail string, see gat_last_error)
// ---------------------------------------------------------------------------
gat_status_t fail(gat_status_t st, const char *fmt, ...);
gat_status_t cuda_fail(cudaError_t err, const char *what);
gat_status_t check_launch(const char *what);

// ---------------------------------------------------------------------------
// plan (host object)
// ---------------------------------------------------------------------------
}  // namespace gat

struct gat_plan_s {
    int64_t n_rows = 0, n_edges = 0;
    int32_t heavy_threshold = 0, chunk_edges = 0;
    int64_t n_heavy = 0, n_chunks = 0;
    int64_t heavy_edges = 0;         // edges owned by heavy rows
    int32_t *heavy_rows = nullptr;   // [n_heavy]
    int32_t *chunk_start = nullptr;  // [n_heavy + 1]
    int32_t *chunk_row = nullptr;    // [n_chunks]
    int32_t *counters = nullptr;     // [n_heavy], arrival counters, zero between calls
    int4 *chunk_desc = nullptr;      // [n_chunks] {row, e0, e1, heavy index} of each chunk
    int32_t *sched = nullptr;        // [4] work counters and finished-block count, zero between calls
    int device = 0;
};

// Transposed (source-major) view of a CSR graph, built by gat_transpose_create.
struct gat_transpose_s {
    int64_t n_rows = 0, n_src = 0, n_edges = 0;
    int32_t max_src_degree = 0;
    int32_t *src_ptr = nullptr;  // [n_src + 1] offsets of each source's edge group
    int32_t *perm = nullptr;     // [n_edges] edge ids, grouped by source, edge order within
    int32_t *dst = nullptr;      // [n_edges] destination row of perm[k]
    gat_plan_t src_plan = nullptr;  // degree plan over src_ptr (heavy sources)
    int device = 0;
};

namespace gat {

// ---------------------------------------------------------------------------
// device helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(kFull, x, o);
    return x;
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(kFull, x, o));
    return x;
}

// 16-byte global load that bypasses L1 allocation (read-once gathers).
__device__ __forceinline__ uint4 ld_stream16(const void *p) {
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// 16-byte global load through L2 only (data written earlier in the same
// kernel by another SM: must not be served from a stale L1 line).
__device__ __forceinline__ float4 ld_cg_f4(const float *p) {
    return __ldcg(reinterpret_cast<const float4 *>(p));
}

// 16-byte streaming store (evict-first; the output is not re-read).
__device__ __forceinline__ void st_stream16(void *p, uint4 v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

// Elements of a 16-byte vector as fp32.
template <typename T>
struct Vec;

template <>
struct Vec<float> {
    static constexpr int N = 4;
    __device__ __forceinline__ static void unpack(const uint4 &u, float *f) {
        f[0] = __uint_as_float(u.x);
        f[1] = __uint_as_float(u.y);
        f[2] = __uint_as_float(u.z);
        f[3] = __uint_as_float(u.w);
    }
    __device__ __forceinline__ static uint4 pack(const float *f) {
        return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                          __float_as_uint(f[3]));
    }
};

// bf16 -> fp32 is exact: the bf16 bits are the high half of the fp32 bits.
template <>
struct Vec<__nv_bfloat16> {
    static constexpr int N = 8;
    __device__ __forceinline__ static void unpack(const uint4 &u, float *f) {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
    __device__ __forceinline__ static uint4 pack(const float *f) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
            w[i] = *reinterpret_cast<uint32_t *>(&h);
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
};

// <a, b> over 8 bf16 pairs (16-byte vectors) with mixed-precision FMAs: each
// bf16 x bf16 product is exact in fp32 and each sum rounded once, as fmaf on
// the converted values; two partial sums (elements 0, 2, .. and 1, 3, ..)
__device__ __forceinline__ float dot_bf16x8(const uint4 &a, const uint4 &b) {
    float s0 = 0.f, s1 = 0.f;
    asm("{\n\t.reg .b16 a0, a1, b0, b1;\n\t"
        "mov.b32 {a0, a1}, %2;\n\tmov.b32 {b0, b1}, %6;\n\t"
        "fma.rn.f32.bf16 %0, a0, b0, %0;\n\tfma.rn.f32.bf16 %1, a1, b1, %1;\n\t"
        "mov.b32 {a0, a1}, %3;\n\tmov.b32 {b0, b1}, %7;\n\t"
        "fma.rn.f32.bf16 %0, a0, b0, %0;\n\tfma.rn.f32.bf16 %1, a1, b1, %1;\n\t"
        "mov.b32 {a0, a1}, %4;\n\tmov.b32 {b0, b1}, %8;\n\t"
        "fma.rn.f32.bf16 %0, a0, b0, %0;\n\tfma.rn.f32.bf16 %1, a1, b1, %1;\n\t"
        "mov.b32 {a0, a1}, %5;\n\tmov.b32 {b0, b1}, %9;\n\t"
        "fma.rn.f32.bf16 %0, a0, b0, %0;\n\tfma.rn.f32.bf16 %1, a1, b1, %1;\n\t}"
        : "+f"(s0), "+f"(s1)
        : "r"(a.x), "r"(a.y), "r"(a.z), "r"(a.w), "r"(b.x), "r"(b.y), "r"(b.z), "r"(b.w));
    return s0 + s1;
}

// Scalar element access for the non-vector kernels.
__device__ __forceinline__ float load_elem(const float *p, int64_t i) { return __ldg(p + i); }
__device__ __forceinline__ float load_elem(const __nv_bfloat16 *p, int64_t i) {
    return __bfloat162float(p[i]);
}
__device__ __forceinline__ void store_elem(float *p, int64_t i, float x) { p[i] = x; }
__device__ __forceinline__ void store_elem(__nv_bfloat16 *p, int64_t i, float x) {
    p[i] = __float2bfloat16_rn(x);
}

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Launch quantities are cached per device ordinal (attributes and occupancy
// belong to a device context), in atomics so host threads making their first
// calls at the same time are safe: a race only computes the same value twice.
constexpr int kMaxDevices = 64;

inline int current_device() {
    int dev = 0;
    cudaGetDevice(&dev);
    return (dev < 0 || dev >= kMaxDevices) ? 0 : dev;
}

// Multiprocessor count of the current device.
inline int sm_count() {
    static std::atomic<int> cache[kMaxDevices];
    const int dev = current_device();
    int n = cache[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (n < 1) n = 1;
        cache[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

// Resident blocks of `kernel` on the whole current device (blocks per SM at
// this block size and dynamic shared memory, times the SM count), computed
// once per device into `cache` (a static array of kMaxDevices atomics owned
// by the call site, one per kernel instance and launch shape).
template <typename Kernel>
inline int64_t device_blocks(std::atomic<int64_t> *cache, Kernel kernel, int threads,
                             size_t smem) {
    const int dev = current_device();
    int64_t cap = cache[dev].load(std::memory_order_relaxed);
    if (cap == 0) {
        int per_sm = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem) !=
                cudaSuccess ||
            per_sm < 1)
            per_sm = 1;
        cap = (int64_t)sm_count() * per_sm;
        cache[dev].store(cap, std::memory_order_relaxed);
    }
    return cap;
}

// Allow `kernel` up to `bytes` of dynamic shared memory on the current device
// (the attribute is per device context), once per device into `done` (a
// static array of kMaxDevices atomic flags owned by the call site). Pass the
// largest amount the kernel is ever launched with, so concurrent first calls
// all set the same value.
template <typename Kernel>
inline cudaError_t allow_dynamic_smem(std::atomic<int> *done, Kernel kernel, int bytes) {
    const int dev = current_device();
    if (done[dev].load(std::memory_order_acquire)) return cudaSuccess;
    const cudaError_t e =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done[dev].store(1, std::memory_order_release);
    return e;
}

}  // namespace gat
