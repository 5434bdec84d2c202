// edge_softmax.cu - segmented, numerically stable softmax over each CSR
// row's edge range, independently per head (FW-GLM-5-1 l1_p6, reference
// model: softmax of every node's edge scores, max-subtracted).
//
// scores/out are [E, H] with heads contiguous, so a row's scores form one
// contiguous run of deg*H floats, and consecutive rows' runs are adjacent.
// For H <= 32 runs are staged through shared memory (cp.async, every copy of
// a run in flight at once), reduced there and written back with one bulk
// copy (TMA engine) per run. Threads work on W consecutive heads at once:
// W = 4 (16-byte shared-memory accesses) when H % 4 == 0 and the pointers are
// 16-byte aligned, else W = 1 with 4-byte copies and plain stores.
//   light rows: a warp stages a run of consecutive light rows (up to 2048
//     scores) and computes its short rows with one thread per (row, group of
//     W heads) and its longer rows (more than kWarpRowDeg edges) with the
//     whole warp, one row at a time;
//   heavy rows (with a plan): a block stages one row in chunks of up to
//     12288 scores and reduces each head group over its threads.
// Rows of a plan's heavy class that still fit a warp's buffer (up to 2048
// scores) are done by the light-row kernel; a light row longer than the
// buffer (possible without a plan, or with a large threshold) is read
// straight from global memory by the whole warp. H > 32 takes the
// head-at-a-time kernels further down.
// out may alias scores: every score of a row is read before its first write.
#include <climits>

#include "common.cuh"

namespace gat {

constexpr int kSoftmaxThreads = 256;     // light-row kernels
constexpr int kSpanFloats = 2048;        // light-row staging buffer per warp (8 KB)
constexpr int kSpanSmemBytes = kSoftmaxThreads / 32 * kSpanFloats * 4;
constexpr int kHeavyThreads = 256;       // heavy-row kernel
constexpr int kHeavySpanFloats = 12288;  // heavy-row staging buffer (48 KB)
constexpr int kSoftmaxCache = 8;         // direct path: loads per thread per tile
constexpr int kWarpRowDeg = 8;           // light rows longer than this: whole-warp softmax
constexpr float kLog2e = 1.4426950408889634f;

// exp(x) as exp2f(x * log2 e) (rarely taken paths)
__device__ __forceinline__ float exp_e(float x) { return exp2f(x * kLog2e); }

// 2^x by the hardware approximation (relative error about 2^-22; results
// below 2^-126 flush to zero, far under the absolute parity bound)
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// W consecutive floats in shared memory
template <int W>
struct SVec;
template <>
struct SVec<1> {
    __device__ static void ld(const float *p, float (&v)[1]) { v[0] = *p; }
    __device__ static void st(float *p, const float (&v)[1]) { *p = v[0]; }
};
template <>
struct SVec<4> {
    __device__ static void ld(const float *p, float (&v)[4]) {
        const float4 t = *reinterpret_cast<const float4 *>(p);
        v[0] = t.x;
        v[1] = t.y;
        v[2] = t.z;
        v[3] = t.w;
    }
    __device__ static void st(float *p, const float (&v)[4]) {
        *reinterpret_cast<float4 *>(p) = make_float4(v[0], v[1], v[2], v[3]);
    }
};

// In-place softmax over d edges of W heads: p[e*H + w], e < d, w < W (one row,
// in shared memory). The maximum is exact, so no -inf guard is needed: a head
// whose scores are all -inf gets (-inf) - (-inf) = NaN terms and NaN outputs,
// as the two-pass definition does.
template <int W>
__device__ __forceinline__ void segment_softmax(float *p, int d, int H) {
    float m[W], z[W], v[W];
#pragma unroll
    for (int w = 0; w < W; ++w) m[w] = -INFINITY, z[w] = 0.f;
#pragma unroll 4
    for (int e = 0; e < d; ++e) {
        SVec<W>::ld(p + e * H, v);
#pragma unroll
        for (int w = 0; w < W; ++w) m[w] = fmaxf(m[w], v[w]);
    }
#pragma unroll 2
    for (int e = 0; e < d; ++e) {
        SVec<W>::ld(p + e * H, v);
#pragma unroll
        for (int w = 0; w < W; ++w) {
            v[w] = ex2_approx((v[w] - m[w]) * kLog2e);
            z[w] += v[w];
        }
        SVec<W>::st(p + e * H, v);
    }
#pragma unroll
    for (int w = 0; w < W; ++w) z[w] = 1.f / z[w];
#pragma unroll 4
    for (int e = 0; e < d; ++e) {
        SVec<W>::ld(p + e * H, v);
#pragma unroll
        for (int w = 0; w < W; ++w) v[w] *= z[w];
        SVec<W>::st(p + e * H, v);
    }
}

// In-place softmax of one row of d edges (H heads, H % 4 == 0, Q = H/4 a power
// of two) by the whole warp: lane l takes float4s l, l+32, ... of the row, all
// of head group l % Q, and the lanes of a head group merge their maxima and
// sums with xor-shuffles over offsets 16 .. Q. Exact maximum, so no -inf guard
// (an all -inf head gives NaN, as the two-pass definition).
__device__ __forceinline__ void warp_row_softmax4(float *p, int d, int H, int lane) {
    const int Q = H >> 2, n4 = d * Q;
    float4 *p4 = reinterpret_cast<float4 *>(p);
    float4 m = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    for (int j = lane; j < n4; j += 32) {
        const float4 v = p4[j];
        m = make_float4(fmaxf(m.x, v.x), fmaxf(m.y, v.y), fmaxf(m.z, v.z), fmaxf(m.w, v.w));
    }
    for (int o = 16; o >= Q; o >>= 1) {
        m.x = fmaxf(m.x, __shfl_xor_sync(kFull, m.x, o));
        m.y = fmaxf(m.y, __shfl_xor_sync(kFull, m.y, o));
        m.z = fmaxf(m.z, __shfl_xor_sync(kFull, m.z, o));
        m.w = fmaxf(m.w, __shfl_xor_sync(kFull, m.w, o));
    }
    float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = lane; j < n4; j += 32) {
        float4 v = p4[j];
        v = make_float4(ex2_approx((v.x - m.x) * kLog2e), ex2_approx((v.y - m.y) * kLog2e),
                        ex2_approx((v.z - m.z) * kLog2e), ex2_approx((v.w - m.w) * kLog2e));
        p4[j] = v;
        z = make_float4(z.x + v.x, z.y + v.y, z.z + v.z, z.w + v.w);
    }
    for (int o = 16; o >= Q; o >>= 1) {
        z.x += __shfl_xor_sync(kFull, z.x, o);
        z.y += __shfl_xor_sync(kFull, z.y, o);
        z.z += __shfl_xor_sync(kFull, z.z, o);
        z.w += __shfl_xor_sync(kFull, z.w, o);
    }
    const float4 inv = make_float4(1.f / z.x, 1.f / z.y, 1.f / z.z, 1.f / z.w);
    for (int j = lane; j < n4; j += 32) {
        const float4 v = p4[j];
        p4[j] = make_float4(v.x * inv.x, v.y * inv.y, v.z * inv.z, v.w * inv.w);
    }
}

// Threads laid over Q head groups: thread t works on group t % Q, slice
// t / Q; the first A = G*Q of `threads` are active.
struct HeadLanes {
    int H, G, A, grp, head;
    bool active;
    __device__ HeadLanes(int q, int threads, int t) {
        H = q;
        G = threads / q;
        A = G * q;
        grp = t / q;
        head = t - grp * q;
        active = t < A;
    }
};

template <bool IS_MAX>
__device__ __forceinline__ float head_op(float a, float b) {
    return IS_MAX ? fmaxf(a, b) : a + b;
}

// ---- direct path: one light row read straight from global memory by a warp
// (lane l strides through the run by A = floor(32/H)*H and sees head l % H)

template <int K>
__device__ __forceinline__ void load_tile(const float *scores, int64_t t0, int64_t x1, int t,
                                          const HeadLanes &hl, float (&v)[K]) {
#pragma unroll
    for (int k = 0; k < K; ++k) {
        const int64_t x = t0 + t + (int64_t)hl.A * k;
        v[k] = (hl.active && x < x1) ? scores[x] : -INFINITY;
    }
}

// reduction over the lanes of a warp that share a head (lanes h, h+H, ...);
// every lane returns its head's result
template <bool IS_MAX>
__device__ __forceinline__ float head_reduce_warp(float v, const HeadLanes &hl) {
    if ((hl.H & (hl.H - 1)) == 0) {
        for (int o = 16; o >= hl.H; o >>= 1) v = head_op<IS_MAX>(v, __shfl_xor_sync(kFull, v, o));
        return v;
    }
    for (int off = 1; off < hl.G; off <<= 1) {
        const float ov = __shfl_down_sync(kFull, v, off * hl.H);
        if (hl.grp + off < hl.G) v = head_op<IS_MAX>(v, ov);
    }
    return __shfl_sync(kFull, v, hl.head);
}

// Tile 0 (registers) is kept; tiles 1.. are folded into a running (max, sum)
// at tile granularity and read again to write. A -inf score adds nothing to
// the running sum, so a head whose scores are all -inf ends with maximum -inf
// and sum 0 and gets 0 * (1/0) = NaN outputs, as the two-pass definition.
__device__ __noinline__ void softmax_row_direct(const float *scores, float *out, int64_t x0,
                                                int64_t x1, int32_t H, int lane) {
    constexpr int K = kSoftmaxCache;
    const HeadLanes hl(H, 32, lane);
    const int64_t step = (int64_t)hl.A * K;
    float c[K];
    load_tile(scores, x0, x1, lane, hl, c);
    float m = -INFINITY, z = 0.f;
#pragma unroll
    for (int k = 0; k < K; ++k) m = fmaxf(m, c[k]);
    for (int64_t t0 = x0 + step; t0 < x1; t0 += step) {
        float v[K];
        load_tile(scores, t0, x1, lane, hl, v);
        float tm = -INFINITY;
#pragma unroll
        for (int k = 0; k < K; ++k) tm = fmaxf(tm, v[k]);
        if (tm > m) {
            z *= exp_e(m - tm);
            m = tm;
        }
#pragma unroll
        for (int k = 0; k < K; ++k) z += v[k] == -INFINITY ? 0.f : exp_e(v[k] - m);
    }
    const float mg = head_reduce_warp<true>(m, hl);
    z = z == 0.f ? 0.f : z * (m == mg ? 1.f : exp_e(m - mg));
#pragma unroll
    for (int k = 0; k < K; ++k) {
        c[k] = c[k] == -INFINITY ? 0.f : exp_e(c[k] - mg);
        z += c[k];
    }
    const float inv = 1.f / head_reduce_warp<false>(z, hl);
#pragma unroll
    for (int k = 0; k < K; ++k) {
        const int64_t x = x0 + lane + (int64_t)hl.A * k;
        if (hl.active && x < x1) out[x] = c[k] * inv;
    }
    for (int64_t t0 = x0 + step; t0 < x1; t0 += step) {
        float v[K];
        load_tile(scores, t0, x1, lane, hl, v);
#pragma unroll
        for (int k = 0; k < K; ++k) {
            const int64_t x = t0 + lane + (int64_t)hl.A * k;
            if (hl.active && x < x1) out[x] = exp_e(v[k] - mg) * inv;
        }
    }
}

// ---- asynchronous copies

__device__ __forceinline__ void cp_async_16(float *dst, const float *src) {
    const unsigned d = (unsigned)__cvta_generic_to_shared(dst);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_4(float *dst, const float *src) {
    const unsigned d = (unsigned)__cvta_generic_to_shared(dst);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(d), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_all;" ::: "memory");
}
// shared -> global bulk copy (TMA engine); 16-byte aligned, size % 16 == 0
__device__ __forceinline__ void bulk_store(float *dst, const float *src, unsigned bytes) {
    const unsigned s = (unsigned)__cvta_generic_to_shared(src);
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
                 ::"l"(dst), "r"(s), "r"(bytes) : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// copy n floats global -> shared with the calling threads (t of nt)
template <int W>
__device__ __forceinline__ void stage_in(float *dst, const float *src, int n, int t, int nt) {
    if (W == 4) {
        for (int j = t; j < (n >> 2); j += nt) cp_async_16(dst + 4 * j, src + 4 * j);
    } else {
        for (int j = t; j < n; j += nt) cp_async_4(dst + j, src + j);
    }
    cp_async_wait_all();
}

// ---- light rows, H <= 32

// A warp takes batches of 32 consecutive rows (one coalesced row_ptr load
// per batch). Consecutive light rows of a batch own one contiguous run of
// scores; the warp stages such a run (at most kSpanFloats scores) into its
// buffer, computes it with one thread per (row, group of W heads) (Q = H/W
// groups, R = 32/Q rows at a time, lane = r*Q + q) and writes it back. Heavy
// rows are left to the heavy-row kernel.
template <int W>
__global__ void __launch_bounds__(kSoftmaxThreads)
softmax_rows_kernel(const int32_t *__restrict__ row_ptr, int64_t n_rows, int32_t H,
                    const float *scores, float *out, int32_t heavy_threshold) {
    extern __shared__ __align__(16) float span_smem[];
    __shared__ int order_smem[kSoftmaxThreads / 32][32];
    const int lane = threadIdx.x & 31;
    float *sb = span_smem + (threadIdx.x >> 5) * kSpanFloats;
    int *order = order_smem[threadIdx.x >> 5];
    const int Q = H / W, R = 32 / Q;
    const int r = lane / Q, q = lane - r * Q;
    const int32_t cap_e = kSpanFloats / H;  // edges per buffer
    const int64_t wpb = blockDim.x >> 5;
    const int64_t n_warps = (int64_t)gridDim.x * wpb;
    const int64_t n_batches = (n_rows + 31) / 32;
    for (int64_t b = (int64_t)blockIdx.x * wpb + (threadIdx.x >> 5); b < n_batches; b += n_warps) {
        const int64_t r0 = b * 32;
        const int nb = n_rows - r0 < 32 ? (int)(n_rows - r0) : 32;
        const int32_t e0_lane = row_ptr[r0 + (lane < nb ? lane : nb - 1)];
        const int32_t rp_end = row_ptr[r0 + nb];
        const int32_t nxt = __shfl_down_sync(kFull, e0_lane, 1);
        const int32_t e1_lane = lane + 1 < nb ? nxt : rp_end;
        const int32_t deg_lane = e1_lane - e0_lane;
        // a row the staging buffer holds is done here even when the plan
        // counts it heavy (the heavy-row kernel skips such rows)
        const bool fits = lane < nb && deg_lane <= cap_e;
        int i0 = 0;
        while (i0 < nb) {
            // the run: rows i0 .. i1-1, all light and within one buffer
            const int32_t base = __shfl_sync(kFull, e0_lane, i0);
            const bool ok = lane >= i0 && fits && e1_lane - base <= cap_e;
            const unsigned bad = ~__ballot_sync(kFull, ok) & (0xffffffffu << i0);
            int i1 = bad ? __ffs(bad) - 1 : 32;
            if (i1 > nb) i1 = nb;
            if (i1 == i0) {  // a heavy row, or a light row longer than the buffer
                const int32_t d = __shfl_sync(kFull, deg_lane, i0);
                if (d <= heavy_threshold)  // light but too long: straight from global
                    softmax_row_direct(scores, out, (int64_t)base * H, (int64_t)(base + d) * H, H,
                                       lane);
                ++i0;
                continue;
            }
            const int32_t end = __shfl_sync(kFull, e1_lane, i1 - 1);
            const int64_t x0 = (int64_t)base * H;
            const int n = (end - base) * H;
            if (n > 0) {
                if (W == 4 && lane == 0) bulk_wait_read();  // the buffer's last bulk store
                __syncwarp();
                stage_in<W>(sb, scores + x0, n, lane, 32);
                __syncwarp();
                // rows of more than kWarpRowDeg edges (W = 4, Q a power of two):
                // the whole warp, one row at a time; the rest one thread per
                // (row, head group), R rows at a time, so a warp instruction
                // never waits on one long row
                const unsigned run_mask = (i1 - i0 == 32 ? 0xffffffffu : ((1u << (i1 - i0)) - 1u)) << i0;
                const bool warp_ok = W == 4 && (Q & (Q - 1)) == 0;
                const unsigned long_mask =
                    __ballot_sync(kFull, warp_ok && deg_lane > kWarpRowDeg) & run_mask;
                const unsigned short_mask = run_mask & ~long_mask;
                if ((short_mask >> lane) & 1u) order[__popc(short_mask & ((1u << lane) - 1u))] = lane;
                __syncwarp();
                const int ns = __popc(short_mask);
                for (int g0 = 0; g0 < ns; g0 += R) {
                    const int slot = g0 + r;
                    const bool has = r < R && slot < ns;
                    const int i = has ? order[slot] : 0;
                    const int32_t ri0 = __shfl_sync(kFull, e0_lane, i);
                    const int32_t ri1 = __shfl_sync(kFull, e1_lane, i);
                    if (has) segment_softmax<W>(sb + (ri0 - base) * H + q * W, ri1 - ri0, H);
                }
                for (unsigned lm = long_mask; lm; lm &= lm - 1u) {
                    const int i = __ffs(lm) - 1;
                    const int32_t ri0 = __shfl_sync(kFull, e0_lane, i);
                    const int32_t ri1 = __shfl_sync(kFull, e1_lane, i);
                    __syncwarp();
                    warp_row_softmax4(sb + (ri0 - base) * H, ri1 - ri0, H, lane);
                }
                if (W == 4) {
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    __syncwarp();
                    if (lane == 0) bulk_store(out + x0, sb, (unsigned)n * 4u);
                } else {
                    __syncwarp();
                    for (int j = lane; j < n; j += 32) out[x0 + j] = sb[j];
                    __syncwarp();
                }
            }
            i0 = i1;
        }
    }
    if (W == 4 && lane == 0) bulk_wait_all();
}

// ---- heavy rows, H <= 32

// reduction over the threads of a block that share a head group (W values
// each); red holds kHeavyThreads * 4 floats; every thread gets its group's
// result
template <bool IS_MAX, int W>
__device__ __forceinline__ void head_reduce_block(float (&v)[W], const HeadLanes &hl, float *red) {
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5, nw = blockDim.x >> 5;
    const int Q = hl.H;
    if ((Q & (Q - 1)) == 0) {
        // Q divides 32: lane % Q == t % Q, so reduce in the warp first
        for (int o = 16; o >= Q; o >>= 1)
#pragma unroll
            for (int w = 0; w < W; ++w) v[w] = head_op<IS_MAX>(v[w], __shfl_xor_sync(kFull, v[w], o));
        if (lane < Q)
#pragma unroll
            for (int w = 0; w < W; ++w) red[(warp * Q + lane) * W + w] = v[w];
        __syncthreads();
#pragma unroll
        for (int w = 0; w < W; ++w) {
            float x = red[hl.head * W + w];
            for (int k = 1; k < nw; ++k) x = head_op<IS_MAX>(x, red[(k * Q + hl.head) * W + w]);
            v[w] = x;
        }
        __syncthreads();
        return;
    }
#pragma unroll
    for (int w = 0; w < W; ++w) red[t * W + w] = v[w];
    __syncthreads();
    for (int off = 1; off < hl.G; off <<= 1) {
        if (hl.grp % (2 * off) == 0 && hl.grp + off < hl.G)
#pragma unroll
            for (int w = 0; w < W; ++w)
                red[t * W + w] = head_op<IS_MAX>(red[t * W + w], red[(t + off * Q) * W + w]);
        __syncthreads();
    }
#pragma unroll
    for (int w = 0; w < W; ++w) v[w] = red[hl.head * W + w];
    __syncthreads();
}

// One block per heavy row. The row's run is staged through shared memory in
// chunks of whole edges; thread t works on head group t % Q (W heads) and
// edges t / Q, t / Q + S, ... of a chunk (S = floor(256 / Q)), so a warp
// reads consecutive words. A run that fits one chunk is read once (maximum,
// exp terms and scaling in shared memory, one bulk store); a longer run is
// read twice: the first pass folds each chunk into a per-thread (max, sum of
// exp), the second recomputes and writes.
template <int W>
__global__ void __launch_bounds__(kHeavyThreads)
softmax_heavy_rows_kernel(const int32_t *__restrict__ row_ptr,
                          const int32_t *__restrict__ heavy_rows, int64_t n_heavy, int32_t H,
                          const float *scores, float *out, int32_t light_cap) {
    extern __shared__ __align__(16) float hs[];
    __shared__ float red[kHeavyThreads * 4];
    const int t = threadIdx.x;
    const HeadLanes hl(H / W, kHeavyThreads, t);
    const int S = hl.G;
    const int col = hl.head * W;
    const int32_t ce = kHeavySpanFloats / H;  // edges per chunk
    auto stage = [&](int64_t f0, int32_t d) {
        if (W == 4 && t == 0) bulk_wait_read();
        __syncthreads();
        stage_in<W>(hs, scores + f0 * H, d * H, t, kHeavyThreads);
        __syncthreads();
    };
    auto flush = [&](int64_t f0, int32_t d) {
        const int n = d * H;
        if (W == 4) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncthreads();
            if (t == 0) bulk_store(out + f0 * H, hs, (unsigned)n * 4u);
        } else {
            __syncthreads();
            for (int j = t; j < n; j += kHeavyThreads) out[f0 * H + j] = hs[j];
            __syncthreads();
        }
    };
    for (int64_t b = blockIdx.x; b < n_heavy; b += gridDim.x) {
        const int64_t row = heavy_rows[b];
        const int64_t e0 = row_ptr[row];
        const int32_t deg = row_ptr[row + 1] - row_ptr[row];
        if (deg <= light_cap) continue;  // the light-row kernel's
        float m[W], z[W], v[W];
#pragma unroll
        for (int w = 0; w < W; ++w) m[w] = -INFINITY, z[w] = 0.f;
        if (deg <= ce) {
            stage(e0, deg);
            if (hl.active)
#pragma unroll 4
                for (int e = hl.grp; e < deg; e += S) {
                    SVec<W>::ld(hs + e * H + col, v);
#pragma unroll
                    for (int w = 0; w < W; ++w) m[w] = fmaxf(m[w], v[w]);
                }
            head_reduce_block<true, W>(m, hl, red);
            // m is the group's exact maximum: a head whose scores are all
            // -inf gets NaN terms and NaN outputs, as the two-pass definition
            if (hl.active)
#pragma unroll 2
                for (int e = hl.grp; e < deg; e += S) {
                    SVec<W>::ld(hs + e * H + col, v);
#pragma unroll
                    for (int w = 0; w < W; ++w) {
                        v[w] = ex2_approx((v[w] - m[w]) * kLog2e);
                        z[w] += v[w];
                    }
                    SVec<W>::st(hs + e * H + col, v);
                }
            head_reduce_block<false, W>(z, hl, red);
#pragma unroll
            for (int w = 0; w < W; ++w) z[w] = 1.f / z[w];
            if (hl.active)
#pragma unroll 4
                for (int e = hl.grp; e < deg; e += S) {
                    SVec<W>::ld(hs + e * H + col, v);
#pragma unroll
                    for (int w = 0; w < W; ++w) v[w] *= z[w];
                    SVec<W>::st(hs + e * H + col, v);
                }
            flush(e0, deg);
            continue;
        }
        // first pass: per-thread (max, sum) folded chunk by chunk; a -inf
        // score adds nothing, so an all -inf head ends with (-inf, 0) and
        // gets 0 * (1/0) = NaN outputs
        for (int32_t c0 = 0; c0 < deg; c0 += ce) {
            const int32_t d = deg - c0 < ce ? deg - c0 : ce;
            stage(e0 + c0, d);
            float cm[W];
#pragma unroll
            for (int w = 0; w < W; ++w) cm[w] = -INFINITY;
            if (hl.active)
                for (int e = hl.grp; e < d; e += S) {
                    SVec<W>::ld(hs + e * H + col, v);
#pragma unroll
                    for (int w = 0; w < W; ++w) cm[w] = fmaxf(cm[w], v[w]);
                }
#pragma unroll
            for (int w = 0; w < W; ++w)
                if (cm[w] > m[w]) {
                    z[w] *= exp_e(m[w] - cm[w]);
                    m[w] = cm[w];
                }
            if (hl.active)
                for (int e = hl.grp; e < d; e += S) {
                    SVec<W>::ld(hs + e * H + col, v);
#pragma unroll
                    for (int w = 0; w < W; ++w) z[w] += v[w] == -INFINITY ? 0.f : exp_e(v[w] - m[w]);
                }
        }
        float mg[W];
#pragma unroll
        for (int w = 0; w < W; ++w) mg[w] = m[w];
        head_reduce_block<true, W>(mg, hl, red);
#pragma unroll
        for (int w = 0; w < W; ++w)
            z[w] = z[w] == 0.f ? 0.f : z[w] * (m[w] == mg[w] ? 1.f : exp_e(m[w] - mg[w]));
        head_reduce_block<false, W>(z, hl, red);
#pragma unroll
        for (int w = 0; w < W; ++w) z[w] = 1.f / z[w];
        // second pass: recompute and write
        for (int32_t c0 = 0; c0 < deg; c0 += ce) {
            const int32_t d = deg - c0 < ce ? deg - c0 : ce;
            stage(e0 + c0, d);
            if (hl.active)
                for (int e = hl.grp; e < d; e += S) {
                    SVec<W>::ld(hs + e * H + col, v);
#pragma unroll
                    for (int w = 0; w < W; ++w) v[w] = exp_e(v[w] - mg[w]) * z[w];
                    SVec<W>::st(hs + e * H + col, v);
                }
            flush(e0 + c0, d);
        }
    }
    if (W == 4 && t == 0) bulk_wait_all();
}

// H > 32: lanes over edges, one head at a time
__global__ void __launch_bounds__(kSoftmaxThreads)
softmax_rows_generic_kernel(const int32_t *__restrict__ row_ptr, int64_t n_rows, int32_t H,
                            const float *scores, float *out, int32_t heavy_threshold) {
    const int lane = threadIdx.x & 31;
    const int64_t wpb = blockDim.x >> 5;
    const int64_t n_warps = (int64_t)gridDim.x * wpb;
    for (int64_t row = (int64_t)blockIdx.x * wpb + (threadIdx.x >> 5); row < n_rows;
         row += n_warps) {
        const int64_t e0 = row_ptr[row], e1 = row_ptr[row + 1];
        if (e1 - e0 > heavy_threshold || e1 == e0) continue;
        for (int h = 0; h < H; ++h) {
            float m = -INFINITY;
            for (int64_t e = e0 + lane; e < e1; e += 32) m = fmaxf(m, scores[e * H + h]);
            m = warp_max(m);
            float z = 0.f;
            for (int64_t e = e0 + lane; e < e1; e += 32) z += expf(scores[e * H + h] - m);
            z = warp_sum(z);
            for (int64_t e = e0 + lane; e < e1; e += 32)
                out[e * H + h] = expf(scores[e * H + h] - m) / z;
        }
    }
}

// heavy rows, H > 32: one block per row, heads one at a time, block reductions
__global__ void __launch_bounds__(kSoftmaxThreads)
softmax_heavy_kernel(const int32_t *__restrict__ row_ptr, const int32_t *__restrict__ heavy_rows,
                     int64_t n_heavy, int32_t H, const float *scores, float *out) {
    __shared__ float red[kSoftmaxThreads / 32];
    __shared__ float bcast;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nw = blockDim.x >> 5;
    for (int64_t b = blockIdx.x; b < n_heavy; b += gridDim.x) {
        const int64_t row = heavy_rows[b];
        const int64_t e0 = row_ptr[row], e1 = row_ptr[row + 1];
        for (int h = 0; h < H; ++h) {
            float m = -INFINITY;
            for (int64_t e = e0 + threadIdx.x; e < e1; e += blockDim.x)
                m = fmaxf(m, scores[e * H + h]);
            m = warp_max(m);
            if (lane == 0) red[warp] = m;
            __syncthreads();
            if (threadIdx.x == 0) {
                float t = red[0];
                for (int w = 1; w < nw; ++w) t = fmaxf(t, red[w]);
                bcast = t;
            }
            __syncthreads();
            m = bcast;
            __syncthreads();
            float z = 0.f;
            for (int64_t e = e0 + threadIdx.x; e < e1; e += blockDim.x)
                z += expf(scores[e * H + h] - m);
            z = warp_sum(z);
            if (lane == 0) red[warp] = z;
            __syncthreads();
            if (threadIdx.x == 0) {
                float t = red[0];
                for (int w = 1; w < nw; ++w) t += red[w];
                bcast = t;
            }
            __syncthreads();
            z = bcast;
            __syncthreads();
            for (int64_t e = e0 + threadIdx.x; e < e1; e += blockDim.x)
                out[e * H + h] = expf(scores[e * H + h] - m) / z;
            __syncthreads();
        }
    }
}

}  // namespace gat

using namespace gat;

extern "C" gat_status_t gat_edge_softmax(const int32_t *row_ptr, int64_t n_rows, int64_t n_edges,
                                         int32_t H, const float *scores, float *out,
                                         gat_plan_t plan, void *stream) {
    if (n_rows < 0 || n_edges < 0 || H < 1)
        return fail(GAT_ERR_INVALID_ARG, "gat_edge_softmax: bad sizes n_rows=%lld n_edges=%lld H=%d",
                    (long long)n_rows, (long long)n_edges, (int)H);
    if (n_rows == 0 || n_edges == 0) return GAT_OK;
    if (!row_ptr || !scores || !out)
        return fail(GAT_ERR_INVALID_ARG, "gat_edge_softmax: NULL pointer");
    if (plan && (plan->n_rows != n_rows || plan->n_edges != n_edges))
        return fail(GAT_ERR_PLAN_MISMATCH, "gat_edge_softmax: plan is for n_rows=%lld n_edges=%lld",
                    (long long)plan->n_rows, (long long)plan->n_edges);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int32_t T = plan ? plan->heavy_threshold : INT_MAX;
    const int64_t wpb = kSoftmaxThreads / 32;
    // a warp per batch of 32 rows (H <= 32) or per row (H > 32)
    const int64_t warps = H <= 32 ? (n_rows + 31) / 32 : n_rows;
    int64_t blocks = (warps + wpb - 1) / wpb;
    // W = 4 heads per thread (16-byte accesses) when the layout allows it
    const bool vec4 = H % 4 == 0 && aligned16(scores) && aligned16(out);
    if (H <= 32) {
        auto kern = vec4 ? softmax_rows_kernel<4> : softmax_rows_kernel<1>;
        cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               kSpanSmemBytes);
        if (err != cudaSuccess) return cuda_fail(err, "gat_edge_softmax: shared memory attribute");
        int per_sm = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kSoftmaxThreads,
                                                          kSpanSmemBytes) != cudaSuccess ||
            per_sm < 1)
            per_sm = 1;
        const int64_t cap = (int64_t)sm_count() * per_sm;
        if (blocks > cap) blocks = cap;
        kern<<<(unsigned)blocks, kSoftmaxThreads, kSpanSmemBytes, s>>>(row_ptr, n_rows, H, scores,
                                                                       out, T);
    } else {
        const int64_t cap = (int64_t)sm_count() * 8;
        if (blocks > cap) blocks = cap;
        softmax_rows_generic_kernel<<<(unsigned)blocks, kSoftmaxThreads, 0, s>>>(
            row_ptr, n_rows, H, scores, out, T);
    }
    gat_status_t st = check_launch("gat_edge_softmax: rows");
    if (st != GAT_OK) return st;
    if (plan && plan->n_heavy > 0) {
        int64_t hb = plan->n_heavy;
        if (H <= 32) {
            auto hk = vec4 ? softmax_heavy_rows_kernel<4> : softmax_heavy_rows_kernel<1>;
            const int smem = kHeavySpanFloats * 4;
            cudaError_t err =
                cudaFuncSetAttribute(hk, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
            if (err != cudaSuccess)
                return cuda_fail(err, "gat_edge_softmax: shared memory attribute");
            int per_sm = 0;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, hk, kHeavyThreads, smem) !=
                    cudaSuccess ||
                per_sm < 1)
                per_sm = 1;
            const int64_t hcap = (int64_t)sm_count() * per_sm;
            if (hb > hcap) hb = hcap;
            hk<<<(unsigned)hb, kHeavyThreads, smem, s>>>(row_ptr, plan->heavy_rows, plan->n_heavy,
                                                         H, scores, out, kSpanFloats / H);
        } else {
            const int64_t hcap = (int64_t)sm_count() * 8;
            if (hb > hcap) hb = hcap;
            softmax_heavy_kernel<<<(unsigned)hb, kSoftmaxThreads, 0, s>>>(
                row_ptr, plan->heavy_rows, plan->n_heavy, H, scores, out);
        }
        st = check_launch("gat_edge_softmax: heavy rows");
    }
    return st;
}
