// edge_softmax.cu - segmented, numerically stable softmax over each CSR
// row's edge range, independently per head (FW-GLM-5-1 l1_p6, reference
// model: softmax of every node's edge scores, max-subtracted).
//
// scores/out are [E, H] with heads contiguous, so a row's scores form one
// contiguous run of deg*H floats, and consecutive rows' runs are adjacent.
// H <= 32 is one launch of softmax_rows_kernel, a grid of the resident
// blocks (8 warps, 64 KB of staging buffer each):
//   phase 1 (with a plan): the plan's heavy rows longer than a warp buffer,
//     one block per row. With W = 4 and H <= 32 the block takes list entries
//     blockIdx.x, blockIdx.x + gridDim.x, ... and streams their chunks
//     through a ring of eight 8 KB slots (softmax_heavy_ring: up to seven
//     chunks in flight, no barrier per chunk, two per row); otherwise it
//     fetches 8 list entries at a time from a counter in the plan and
//     streams each row through two 32 KB halves of the block buffer (the
//     next chunk's copies in flight while this one is computed); rows longer
//     than the resident limit are read twice (fold, then normalise);
//   phase 2: batches of 32 consecutive rows, fetched from a second counter
//     (static stride without a plan). A warp stages runs of consecutive rows
//     (up to 2048 scores: one bulk copy in, on the warp's mbarrier, with
//     W = 4; cp.async with every copy in flight otherwise), computes them in
//     shared memory / registers and writes each run back with one bulk copy
//     (TMA engine).
// Threads work on W consecutive heads at once: W = 4 (16-byte accesses) when
// H % 4 == 0 and the pointers are 16-byte aligned, else W = 1 with 4-byte
// copies and plain stores. With W = 4 and Q = H/4 a power of two, a light
// row goes to a sub-warp of S lanes (S = Q .. 32, a power of two) holding up
// to 4 float4s per lane in registers, or 8 per lane with the whole warp, or
// past that to the whole warp through shared memory; a row beyond the buffer
// that the plan does not call heavy (any such row without a plan) streams
// through the warp's buffer twice (fold, then normalise). Other layouts use
// one thread per (row, group of W heads), and read a light row longer than
// the buffer straight from global memory with the whole warp. The launch
// serves H <= 32, and H = 64 or 128 with W = 4 (Q = 16 or 32 head groups,
// still at most one per lane); other head counts take the head-at-a-time
// kernels further down. The last block to finish resets the plan's
// counters, so a plan serves one launch at a time.
// out may alias scores: every score of a row (or chunk) is read before its
// first write.
#include <climits>

#include "common.cuh"

namespace gat {

constexpr int kSoftmaxThreads = 256;     // light-row kernels
constexpr int kSpanFloats = 2048;        // light-row staging buffer per warp (8 KB)
constexpr int kSpanBlockFloats = kSoftmaxThreads / 32 * kSpanFloats;  // heavy rows: 2 chunks
constexpr int kHeavyUnit = 8;            // heavy-list entries per fetch
constexpr int kHeavyRegs = 8;            // heavy rows: float4s per thread and chunk
constexpr int kSpanSmemBytes = kSpanBlockFloats * 4;
constexpr int kSoftmaxCache = 8;         // direct path: loads per thread per tile
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

// 1/x by the hardware approximation (about 1 ulp). The softmax sums it
// inverts are at least 1 (the maximum's own term) or NaN (a head of -inf
// scores), so no denormal or zero input reaches it from a finite row.
__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
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
    const float4 inv = make_float4(rcp_approx(z.x), rcp_approx(z.y), rcp_approx(z.z), rcp_approx(z.w));
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

// one bulk copy (TMA engine) of `bytes` (a multiple of 16, both addresses
// 16-byte aligned) global -> shared, completing on the mbarrier `bar`, which
// the calling thread arms with the byte count
__device__ __forceinline__ void bulk_load(float *dst, const float *src, unsigned bytes, uint64_t *bar) {
    const unsigned d = (unsigned)__cvta_generic_to_shared(dst);
    const unsigned b = (unsigned)__cvta_generic_to_shared(bar);
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(b), "r"(bytes)
                 : "memory");
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(d),
        "l"(src), "r"(bytes), "r"(b)
        : "memory");
}
// wait for the phase of parity `ph` of `bar` (bounded: 2^30 polls, far beyond
// any copy; the data is then used as it stands)
__device__ __forceinline__ void mbar_wait_bounded(uint64_t *bar, unsigned ph) {
    const unsigned b = (unsigned)__cvta_generic_to_shared(bar);
    for (unsigned it = 0; it < (1u << 30); ++it) {
        unsigned done;
        asm volatile(
            "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(b), "r"(ph)
            : "memory");
        if (done) return;
    }
}

// start copying n floats global -> shared with the calling threads (t of nt)
template <int W>
__device__ __forceinline__ void stage_issue(float *dst, const float *src, int n, int t, int nt) {
    if (W == 4) {
        for (int j = t; j < (n >> 2); j += nt) cp_async_16(dst + 4 * j, src + 4 * j);
    } else {
        for (int j = t; j < n; j += nt) cp_async_4(dst + j, src + j);
    }
}
// copy n floats global -> shared with the calling threads and wait for them
template <int W>
__device__ __forceinline__ void stage_in(float *dst, const float *src, int n, int t, int nt) {
    stage_issue<W>(dst, src, n, t, nt);
    cp_async_wait_all();
}

// ---- light rows in registers (W = 4, Q = H/4 a power of two)

__device__ __forceinline__ float4 max4(float4 a, float4 b) {
    return make_float4(fmaxf(a.x, b.x), fmaxf(a.y, b.y), fmaxf(a.z, b.z), fmaxf(a.w, b.w));
}
__device__ __forceinline__ float4 shfl_xor4(float4 a, int o) {
    return make_float4(__shfl_xor_sync(kFull, a.x, o), __shfl_xor_sync(kFull, a.y, o),
                       __shfl_xor_sync(kFull, a.z, o), __shfl_xor_sync(kFull, a.w, o));
}

// Softmax of the rows in `tm` (lanes of the batch whose rows lie in the
// staged run at sb, first edge `base`; results written back in place), each
// row on a sub-warp of S lanes
// (Q <= S <= 32, powers of two), 32/S rows at a time. A row's run is d*Q
// float4s; lane s of the sub-warp holds float4s s, s+S, ..., at most KV of
// them, all of head group s % Q, in registers from one shared-memory read to
// the one write of the result. Maximum and sum are merged over the lanes of
// a head group with xor-shuffles over offsets S/2 .. Q. The sub-warps visit
// their KV slots in rotated order, so that rows starting at equal bank
// offsets do not meet in one wavefront. Exact maximum: a head whose scores
// are all -inf gets NaN outputs, as the two-pass definition.
template <int KV>
__device__ __forceinline__ void softmax_tier4(float *sb, int32_t base, int H, int Q, int S,
                                              unsigned tm, int32_t e0_lane, int32_t e1_lane,
                                              int *order, int lane) {
    if ((tm >> lane) & 1u) order[__popc(tm & ((1u << lane) - 1u))] = lane;
    __syncwarp();
    const int cnt = __popc(tm);
    const int lg = __ffs(S) - 1;
    const int slot = lane >> lg, s = lane & (S - 1), P = 32 >> lg;
    const int rot = slot & (KV - 1);
    const float4 ninf = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    for (int p0 = 0; p0 < cnt; p0 += P) {
        const int k = p0 + slot;
        const bool has = k < cnt;
        const int i = has ? order[k] : 0;
        const int32_t ri0 = __shfl_sync(kFull, e0_lane, i);
        const int32_t ri1 = __shfl_sync(kFull, e1_lane, i);
        const int n4 = has ? (ri1 - ri0) * Q : 0;
        float4 *p = reinterpret_cast<float4 *>(sb + (ri0 - base) * H);
        float4 v[KV];
        float4 m = ninf;
#pragma unroll
        for (int t = 0; t < KV; ++t) {
            const int j = s + ((t + rot) & (KV - 1)) * S;
            v[t] = j < n4 ? p[j] : ninf;
            m = max4(m, v[t]);
        }
        for (int o = S >> 1; o >= Q; o >>= 1) m = max4(m, shfl_xor4(m, o));
        float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int t = 0; t < KV; ++t) {
            v[t] = make_float4(ex2_approx((v[t].x - m.x) * kLog2e), ex2_approx((v[t].y - m.y) * kLog2e),
                               ex2_approx((v[t].z - m.z) * kLog2e), ex2_approx((v[t].w - m.w) * kLog2e));
            z = make_float4(z.x + v[t].x, z.y + v[t].y, z.z + v[t].z, z.w + v[t].w);
        }
        for (int o = S >> 1; o >= Q; o >>= 1) {
            const float4 y = shfl_xor4(z, o);
            z = make_float4(z.x + y.x, z.y + y.y, z.z + y.z, z.w + y.w);
        }
        const float4 inv = make_float4(rcp_approx(z.x), rcp_approx(z.y), rcp_approx(z.z), rcp_approx(z.w));
#pragma unroll
        for (int t = 0; t < KV; ++t) {
            const int j = s + ((t + rot) & (KV - 1)) * S;
            if (j < n4)
                p[j] = make_float4(v[t].x * inv.x, v[t].y * inv.y, v[t].z * inv.z, v[t].w * inv.w);
        }
    }
    __syncwarp();
}

// A row of d edges (first edge e0) longer than the warp buffer by the warp
// alone (W = 4, Q a power of two): its run streams through the buffer sb in
// chunks of cap_e edges twice. Fold pass: lane l holds float4s l, l+32, ...
// of a chunk (head group l % Q); per chunk the lane's maximum, then its exp
// terms against the running maximum (the running sum rescaled when the
// maximum grows); the lanes of a head group then merge their (max, sum)
// pairs with xor-shuffles. Normalise pass: the chunk again (the second read
// of a run the warp has just read), exp terms scaled by 1/sum, written back
// with one bulk copy per chunk. A head whose scores are all -inf keeps sum 0
// and gets NaN outputs, as the two-pass definition.
__device__ __noinline__ void softmax_row_medium4(const float *scores, float *out, float *sb,
                                                 int64_t e0, int32_t d, int32_t H, int32_t cap_e,
                                                 int lane) {
    const int Q = H >> 2;
    float4 m = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    const float4 *p4 = reinterpret_cast<const float4 *>(sb);
    auto stage = [&](int32_t c0, int32_t dc) {
        if (lane == 0) bulk_wait_read();  // the buffer's last bulk store has read it
        __syncwarp();
        stage_in<4>(sb, scores + (e0 + c0) * H, dc * H, lane, 32);
        __syncwarp();
    };
    auto fold1 = [](float &mw, float &zw, float cm) {
        if (cm > mw) {
            zw = zw == 0.f ? 0.f : zw * ex2_approx((mw - cm) * kLog2e);
            mw = cm;
        }
    };
    for (int32_t c0 = 0; c0 < d; c0 += cap_e) {
        const int32_t dc = d - c0 < cap_e ? d - c0 : cap_e;
        const int n4 = dc * Q;
        stage(c0, dc);
        float4 cm = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        for (int j = lane; j < n4; j += 32) cm = max4(cm, p4[j]);
        fold1(m.x, z.x, cm.x);
        fold1(m.y, z.y, cm.y);
        fold1(m.z, z.z, cm.z);
        fold1(m.w, z.w, cm.w);
        // with m = -inf every score so far is -inf: the terms stay 0
        const float4 mm = make_float4(m.x == -INFINITY ? 0.f : m.x, m.y == -INFINITY ? 0.f : m.y,
                                      m.z == -INFINITY ? 0.f : m.z, m.w == -INFINITY ? 0.f : m.w);
        for (int j = lane; j < n4; j += 32) {
            const float4 v = p4[j];
            z.x += ex2_approx((v.x - mm.x) * kLog2e);
            z.y += ex2_approx((v.y - mm.y) * kLog2e);
            z.z += ex2_approx((v.z - mm.z) * kLog2e);
            z.w += ex2_approx((v.w - mm.w) * kLog2e);
        }
    }
    // merge the head group's lanes (offsets 16 .. Q keep l % Q)
    auto merge1 = [](float &mw, float &zw, float mo, float zo) {
        const float mx = fmaxf(mw, mo);
        const float a = zw == 0.f ? 0.f : zw * ex2_approx((mw - mx) * kLog2e);
        const float b = zo == 0.f ? 0.f : zo * ex2_approx((mo - mx) * kLog2e);
        mw = mx;
        zw = a + b;
    };
    for (int o = 16; o >= Q; o >>= 1) {
        const float4 mo = shfl_xor4(m, o), zo = shfl_xor4(z, o);
        merge1(m.x, z.x, mo.x, zo.x);
        merge1(m.y, z.y, mo.y, zo.y);
        merge1(m.z, z.z, mo.z, zo.z);
        merge1(m.w, z.w, mo.w, zo.w);
    }
    const float4 inv = make_float4(rcp_approx(z.x), rcp_approx(z.y), rcp_approx(z.z), rcp_approx(z.w));
    float4 *q4 = reinterpret_cast<float4 *>(sb);
    for (int32_t c0 = 0; c0 < d; c0 += cap_e) {
        const int32_t dc = d - c0 < cap_e ? d - c0 : cap_e;
        const int n4 = dc * Q;
        stage(c0, dc);
        for (int j = lane; j < n4; j += 32) {
            const float4 v = q4[j];
            q4[j] = make_float4(ex2_approx((v.x - m.x) * kLog2e) * inv.x,
                                ex2_approx((v.y - m.y) * kLog2e) * inv.y,
                                ex2_approx((v.z - m.z) * kLog2e) * inv.z,
                                ex2_approx((v.w - m.w) * kLog2e) * inv.w);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) bulk_store(out + (e0 + c0) * H, sb, (unsigned)(dc * H) * 4u);
    }
}

// ---- heavy rows, H <= 32

// reduction over the threads of a block that share a head group (W values
// each); red holds kSoftmaxThreads * 4 floats; every thread gets its group's
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

// One chunk task of a heavy row with the thread's (up to 8) float4s of the
// chunk in registers (W = 4, Q a power of two). kind 0: the whole row in one
// chunk (block maximum, exp terms, block sum, scaled write-back); kind 1: a
// fold of the chunk into the running (m, z) = (maximum, sum of exp), merged
// over the block after the row's last chunk into (m, z) = (row maximum,
// 1 / row sum); kind 2: the chunk's outputs from that (m, z). Kinds 0 and 2
// store the outputs from registers to gout, the chunk's place in the output.
// Padding slots hold -inf, whose exp term is 0; a -inf score adds nothing to
// a fold, so a head whose scores are all -inf ends with sum 0 and NaN
// outputs, as the two-pass definition.
__device__ __forceinline__ void heavy_task_regs(const float *cb, float *gout, int32_t d, int kind,
                                                bool first, bool last, const HeadLanes &hl,
                                                int32_t H, float *red, float (&m)[4],
                                                float (&z)[4]) {
    constexpr int KH = kHeavyRegs;
    const int S = hl.G, col = hl.head * 4;
    const float4 ninf = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    float4 x[KH];
#pragma unroll
    for (int t = 0; t < KH; ++t) {
        const int e = hl.grp + t * S;
        x[t] = hl.active && e < d ? *reinterpret_cast<const float4 *>(cb + e * H + col) : ninf;
    }
    auto store = [&]() {
#pragma unroll
        for (int t = 0; t < KH; ++t) {
            const int e = hl.grp + t * S;
            if (hl.active && e < d) *reinterpret_cast<float4 *>(gout + (int64_t)e * H + col) = x[t];
        }
    };
    if (kind == 0) {
        float4 mx = ninf;
#pragma unroll
        for (int t = 0; t < KH; ++t) mx = max4(mx, x[t]);
        float mv[4] = {mx.x, mx.y, mx.z, mx.w};
        head_reduce_block<true, 4>(mv, hl, red);
        float zv[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int t = 0; t < KH; ++t) {
            x[t] = make_float4(ex2_approx((x[t].x - mv[0]) * kLog2e), ex2_approx((x[t].y - mv[1]) * kLog2e),
                               ex2_approx((x[t].z - mv[2]) * kLog2e), ex2_approx((x[t].w - mv[3]) * kLog2e));
            zv[0] += x[t].x;
            zv[1] += x[t].y;
            zv[2] += x[t].z;
            zv[3] += x[t].w;
        }
        head_reduce_block<false, 4>(zv, hl, red);
        const float4 inv = make_float4(rcp_approx(zv[0]), rcp_approx(zv[1]), rcp_approx(zv[2]), rcp_approx(zv[3]));
#pragma unroll
        for (int t = 0; t < KH; ++t)
            x[t] = make_float4(x[t].x * inv.x, x[t].y * inv.y, x[t].z * inv.z, x[t].w * inv.w);
        store();
        return;
    }
    if (kind == 1) {
        if (first)
#pragma unroll
            for (int w = 0; w < 4; ++w) m[w] = -INFINITY, z[w] = 0.f;
        float4 cm = ninf;
#pragma unroll
        for (int t = 0; t < KH; ++t) cm = max4(cm, x[t]);
        const float cmv[4] = {cm.x, cm.y, cm.z, cm.w};
#pragma unroll
        for (int w = 0; w < 4; ++w)
            if (cmv[w] > m[w]) {
                z[w] = z[w] == 0.f ? 0.f : z[w] * ex2_approx((m[w] - cmv[w]) * kLog2e);
                m[w] = cmv[w];
            }
        // with m = -inf every score so far is -inf: the terms stay 0
        const float mm[4] = {m[0] == -INFINITY ? 0.f : m[0], m[1] == -INFINITY ? 0.f : m[1],
                             m[2] == -INFINITY ? 0.f : m[2], m[3] == -INFINITY ? 0.f : m[3]};
#pragma unroll
        for (int t = 0; t < KH; ++t) {
            z[0] += ex2_approx((x[t].x - mm[0]) * kLog2e);
            z[1] += ex2_approx((x[t].y - mm[1]) * kLog2e);
            z[2] += ex2_approx((x[t].z - mm[2]) * kLog2e);
            z[3] += ex2_approx((x[t].w - mm[3]) * kLog2e);
        }
        if (last) {
            float mg[4] = {m[0], m[1], m[2], m[3]};
            head_reduce_block<true, 4>(mg, hl, red);
#pragma unroll
            for (int w = 0; w < 4; ++w)
                z[w] = z[w] == 0.f ? 0.f : z[w] * ex2_approx((m[w] - mg[w]) * kLog2e);
            head_reduce_block<false, 4>(z, hl, red);
#pragma unroll
            for (int w = 0; w < 4; ++w) m[w] = mg[w], z[w] = 1.f / z[w];
        }
        return;
    }
#pragma unroll
    for (int t = 0; t < KH; ++t)
        x[t] = make_float4(ex2_approx((x[t].x - m[0]) * kLog2e) * z[0], ex2_approx((x[t].y - m[1]) * kLog2e) * z[1],
                           ex2_approx((x[t].z - m[2]) * kLog2e) * z[2], ex2_approx((x[t].w - m[3]) * kLog2e) * z[3]);
    store();
}

// The block's heavy rows (first edges e0s[i], degrees degs[i], i < nh, in
// shared memory) as one stream of chunk tasks through two buffers: the
// copies of task k+1 are in flight while task k is computed. Thread t works
// on head group t % Q (W heads) and edges t / Q, t / Q + S, ... of a chunk
// (S = floor(blockDim / Q)), so a warp reads consecutive words. A row of at
// most ce edges is one task, read once (maximum, exp terms and scaling in
// shared memory, one bulk store). A longer row is read twice in chunks of
// ce edges: fold tasks accumulate a per-thread (max, sum of exp), the block
// merges them after the last one, and normalise tasks recompute and write.
// Entered and left by all threads of the block; on return thread 0's last
// bulk store may still be reading its buffer.
template <int W>
__device__ __forceinline__ void softmax_heavy_rows(const int32_t *e0s, const int32_t *degs, int nh,
                                                   int32_t H, const float *scores, float *out,
                                                   float *buf0, float *buf1, int32_t ce,
                                                   float *red) {
    const int t = threadIdx.x;
    const HeadLanes hl(H / W, kSoftmaxThreads, t);
    const int S = hl.G;
    const int col = hl.head * W;
    auto chunk_len = [&](int ii, int32_t cc) {
        const int32_t dd = degs[ii] - cc;
        return dd < ce ? dd : ce;
    };
    auto issue = [&](int ii, int32_t cc, float *dst) {
        stage_issue<W>(dst, scores + ((int64_t)e0s[ii] + cc) * H, chunk_len(ii, cc) * H, t,
                       kSoftmaxThreads);
        asm volatile("cp.async.commit_group;" ::: "memory");
    };
    auto flush = [&](const float *src, int64_t f0, int32_t d) {
        const int n = d * H;
        if (W == 4) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncthreads();
            if (t == 0) bulk_store(out + f0 * H, src, (unsigned)n * 4u);
        } else {
            __syncthreads();
            for (int j = t; j < n; j += kSoftmaxThreads) out[f0 * H + j] = src[j];
            __syncthreads();
        }
    };
    if (nh == 0) return;
    // W = 4 with Q a power of two and at most 8 edges per thread in a chunk:
    // a thread's float4s stay in registers from their one shared-memory read
    // to their one write
    const bool regs = W == 4 && (hl.H & (hl.H - 1)) == 0;
    if (regs && ce > kHeavyRegs * S) ce = kHeavyRegs * S;
    issue(0, 0, buf0);
    float m[W], z[W], v[W];
#pragma unroll
    for (int w = 0; w < W; ++w) m[w] = -INFINITY, z[w] = 0.f;
    int i = 0, pass = 0;
    int32_t c0 = 0;
    for (int k = 0; i < nh; ++k) {
        const int32_t deg = degs[i];
        // the task after this one
        int ni = i, np = pass;
        int32_t nc = c0;
        if (deg <= ce) {
            ni = i + 1;
        } else if (c0 + ce < deg) {
            nc = c0 + ce;
        } else if (pass == 0) {
            np = 1;
            nc = 0;
        } else {
            ni = i + 1;
            np = 0;
            nc = 0;
        }
        float *cb = (k & 1) ? buf1 : buf0;
        float *nb = (k & 1) ? buf0 : buf1;
        cp_async_wait_all();                           // this task's copies
        if (W == 4 && !regs && t == 0) bulk_wait_read();  // the previous task's store has left nb
        __syncthreads();
        if (ni < nh) issue(ni, nc, nb);
        const int32_t d = chunk_len(i, c0);
        const int64_t f0 = (int64_t)e0s[i] + c0;
        if constexpr (W == 4) {
            if (regs) {
                heavy_task_regs(cb, out + f0 * H, d, deg <= ce ? 0 : (pass == 0 ? 1 : 2), c0 == 0,
                                np == 1, hl, H, red, m, z);
                i = ni;
                pass = np;
                c0 = nc;
                continue;
            }
        }
        if (deg <= ce) {
#pragma unroll
            for (int w = 0; w < W; ++w) m[w] = -INFINITY, z[w] = 0.f;
            if (hl.active)
#pragma unroll 4
                for (int e = hl.grp; e < d; e += S) {
                    SVec<W>::ld(cb + e * H + col, v);
#pragma unroll
                    for (int w = 0; w < W; ++w) m[w] = fmaxf(m[w], v[w]);
                }
            head_reduce_block<true, W>(m, hl, red);
            // m is the group's exact maximum: a head whose scores are all
            // -inf gets NaN terms and NaN outputs, as the two-pass definition
            if (hl.active)
#pragma unroll 2
                for (int e = hl.grp; e < d; e += S) {
                    SVec<W>::ld(cb + e * H + col, v);
#pragma unroll
                    for (int w = 0; w < W; ++w) {
                        v[w] = ex2_approx((v[w] - m[w]) * kLog2e);
                        z[w] += v[w];
                    }
                    SVec<W>::st(cb + e * H + col, v);
                }
            head_reduce_block<false, W>(z, hl, red);
#pragma unroll
            for (int w = 0; w < W; ++w) z[w] = 1.f / z[w];
            if (hl.active)
#pragma unroll 4
                for (int e = hl.grp; e < d; e += S) {
                    SVec<W>::ld(cb + e * H + col, v);
#pragma unroll
                    for (int w = 0; w < W; ++w) v[w] *= z[w];
                    SVec<W>::st(cb + e * H + col, v);
                }
            flush(cb, f0, d);
        } else if (pass == 0) {
            // fold: a -inf score adds nothing, so an all -inf head ends with
            // (-inf, 0) and gets 0 * (1/0) = NaN outputs
            if (c0 == 0)
#pragma unroll
                for (int w = 0; w < W; ++w) m[w] = -INFINITY, z[w] = 0.f;
            float cm[W];
#pragma unroll
            for (int w = 0; w < W; ++w) cm[w] = -INFINITY;
            if (hl.active)
                for (int e = hl.grp; e < d; e += S) {
                    SVec<W>::ld(cb + e * H + col, v);
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
                    SVec<W>::ld(cb + e * H + col, v);
#pragma unroll
                    for (int w = 0; w < W; ++w) z[w] += v[w] == -INFINITY ? 0.f : exp_e(v[w] - m[w]);
                }
            if (np == 1) {  // the row's last chunk: merge over the block
                float mg[W];
#pragma unroll
                for (int w = 0; w < W; ++w) mg[w] = m[w];
                head_reduce_block<true, W>(mg, hl, red);
#pragma unroll
                for (int w = 0; w < W; ++w)
                    z[w] = z[w] == 0.f ? 0.f : z[w] * (m[w] == mg[w] ? 1.f : exp_e(m[w] - mg[w]));
                head_reduce_block<false, W>(z, hl, red);
#pragma unroll
                for (int w = 0; w < W; ++w) m[w] = mg[w], z[w] = 1.f / z[w];
            }
        } else {
            // normalise with the row's (maximum, 1 / sum) in (m, z)
            if (hl.active)
                for (int e = hl.grp; e < d; e += S) {
                    SVec<W>::ld(cb + e * H + col, v);
#pragma unroll
                    for (int w = 0; w < W; ++w) v[w] = exp_e(v[w] - m[w]) * z[w];
                    SVec<W>::st(cb + e * H + col, v);
                }
            flush(cb, f0, d);
        }
        i = ni;
        pass = np;
        c0 = nc;
    }
}

// ---- heavy rows, W = 4 and Q = H/4 a power of two: a ring of chunk loads
//
// The block buffer is kRing slots of kSpanFloats scores, one chunk of cap_e
// = kSpanFloats / H edges each. The block's heavy rows form one stream of
// chunk loads: a row of at most kResident chunks is loaded once and stays in
// its slots until it is written; a longer row is loaded twice (fold pass,
// then normalise pass; the second read of a row the block has just read is
// served by L2). Thread t copies (cp.async) and later reads float4 positions
// t + 256 i of every slot and no others, so a chunk needs no block barrier:
// the thread's own cp.async.wait_group covers it. Up to kRing - 1 chunks are
// in flight while one is computed; the block synchronises only in each row's
// merge of its per-thread (maximum, sum) pairs. Serves Q = H/4 <= 8 head
// groups (H = 4, 8, 16, 32).
constexpr int kRing = kSpanBlockFloats / kSpanFloats;       // 8 slots
constexpr int kResident = 4;                                // rows read once: <= 4 chunks
constexpr int kRingPer = kSpanFloats / 4 / kSoftmaxThreads;  // float4s per thread and slot

// wait until at most `pending` (0 .. kRing - 1) of the thread's most recent
// cp.async groups are still in flight
__device__ __forceinline__ void cp_async_wait_upto(int pending) {
    switch (pending) {
        case 0: asm volatile("cp.async.wait_group 0;" ::: "memory"); break;
        case 1: asm volatile("cp.async.wait_group 1;" ::: "memory"); break;
        case 2: asm volatile("cp.async.wait_group 2;" ::: "memory"); break;
        case 3: asm volatile("cp.async.wait_group 3;" ::: "memory"); break;
        case 4: asm volatile("cp.async.wait_group 4;" ::: "memory"); break;
        case 5: asm volatile("cp.async.wait_group 5;" ::: "memory"); break;
        case 6: asm volatile("cp.async.wait_group 6;" ::: "memory"); break;
        default: asm volatile("cp.async.wait_group 7;" ::: "memory"); break;
    }
}

// The issuing side of the stream: rows are the set bits of `left` (lanes of
// every warp hold the same rows' first edge and degree), each row's loads
// in order (resident: one pass; otherwise two).
struct ChunkIssuer {
    unsigned left;
    int32_t e0, deg, nc, c;
    int pass;
    bool have;
    int issued;

    // issue loads while fewer than kRing are unconsumed (loads before `freed`
    // are consumed); block-uniform control flow
    __device__ __forceinline__ void pump(const float *scores, float *buf, int32_t H, int32_t cap_e,
                                         int32_t e0_lane, int32_t deg_lane, int freed, int t) {
        while (issued - freed < kRing) {
            if (!have) {
                if (!left) return;
                const int l = __ffs(left) - 1;
                left &= left - 1u;
                e0 = __shfl_sync(kFull, e0_lane, l);
                deg = __shfl_sync(kFull, deg_lane, l);
                nc = (deg + cap_e - 1) / cap_e;
                c = 0;
                pass = 0;
                have = true;
            }
            const int32_t c0 = c * cap_e;
            const int32_t dc = deg - c0 < cap_e ? deg - c0 : cap_e;
            const int n4 = dc * (H >> 2);
            float *slot = buf + (issued % kRing) * kSpanFloats;
            const float *src = scores + ((int64_t)e0 + c0) * H;
#pragma unroll
            for (int i = 0; i < kRingPer; ++i) {
                const int j = t + i * kSoftmaxThreads;
                if (j < n4) cp_async_16(slot + 4 * j, src + 4 * j);
            }
            asm volatile("cp.async.commit_group;" ::: "memory");  // one group per load, maybe empty
            ++issued;
            if (++c == nc) {
                c = 0;
                if (nc > kResident && pass == 0)
                    pass = 1;
                else
                    have = false;
            }
        }
    }
};

// fold the thread's float4s of one chunk into its running (m, z) of 4 heads
__device__ __forceinline__ void ring_fold(const float *slot, int n4, int t, float4 &m, float4 &z) {
    const float4 ninf = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    float4 v[kRingPer];
    float4 cm = ninf;
#pragma unroll
    for (int i = 0; i < kRingPer; ++i) {
        const int j = t + i * kSoftmaxThreads;
        v[i] = j < n4 ? reinterpret_cast<const float4 *>(slot)[j] : ninf;
        cm = max4(cm, v[i]);
    }
    auto rescale = [](float &mw, float &zw, float cw) {
        if (cw > mw) {
            zw = zw == 0.f ? 0.f : zw * ex2_approx((mw - cw) * kLog2e);
            mw = cw;
        }
    };
    rescale(m.x, z.x, cm.x);
    rescale(m.y, z.y, cm.y);
    rescale(m.z, z.z, cm.z);
    rescale(m.w, z.w, cm.w);
    // a -inf score adds nothing (also while the running maximum is -inf)
    auto term = [](float x, float mw) { return x == -INFINITY ? 0.f : ex2_approx((x - mw) * kLog2e); };
#pragma unroll
    for (int i = 0; i < kRingPer; ++i) {
        z.x += term(v[i].x, m.x);
        z.y += term(v[i].y, m.y);
        z.z += term(v[i].z, m.z);
        z.w += term(v[i].w, m.w);
    }
}

// write the thread's float4s of one chunk as 2^((x - m) log2 e) * inv
__device__ __forceinline__ void ring_write(const float *slot, int n4, int t, float4 m, float4 inv,
                                           float *gout) {
#pragma unroll
    for (int i = 0; i < kRingPer; ++i) {
        const int j = t + i * kSoftmaxThreads;
        if (j < n4) {
            const float4 v = reinterpret_cast<const float4 *>(slot)[j];
            reinterpret_cast<float4 *>(gout)[j] =
                make_float4(ex2_approx((v.x - m.x) * kLog2e) * inv.x,
                            ex2_approx((v.y - m.y) * kLog2e) * inv.y,
                            ex2_approx((v.z - m.z) * kLog2e) * inv.z,
                            ex2_approx((v.w - m.w) * kLog2e) * inv.w);
        }
    }
}

// The row's (maximum, sum) of each of the thread's 4 heads from every
// thread's running (m, z), Q = H/4 <= 8 head groups: xor-shuffles inside the
// warps, then two barriers (maxima; sums rescaled to the row maximum)
// through the two regions of red. A warp writes a region again only after
// the next barrier, which every warp reaches after its reads, so no barrier
// follows the reads.
__device__ __forceinline__ void ring_merge(float4 &m, float4 &z, int Q, float *red) {
    constexpr int NW = kSoftmaxThreads / 32;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int q = lane & (Q - 1);  // = t % Q, the thread's head group
    float4 *rm = reinterpret_cast<float4 *>(red);   // [NW][Q] warp maxima
    float4 *rz = rm + NW * 8;                       // [NW][Q] warp sums
    float4 mw = m;
    for (int o = 16; o >= Q; o >>= 1) mw = max4(mw, shfl_xor4(mw, o));
    if (lane < Q) rm[warp * Q + lane] = mw;
    __syncthreads();
    float4 M = rm[q];
#pragma unroll
    for (int w = 1; w < NW; ++w) M = max4(M, rm[w * Q + q]);
    // a zero sum stays zero (its maximum may be -inf)
    auto sc = [](float zz, float mm, float MM) {
        return zz == 0.f ? 0.f : zz * ex2_approx((mm - MM) * kLog2e);
    };
    float4 zs = make_float4(sc(z.x, m.x, M.x), sc(z.y, m.y, M.y), sc(z.z, m.z, M.z),
                            sc(z.w, m.w, M.w));
    for (int o = 16; o >= Q; o >>= 1) {
        const float4 y = shfl_xor4(zs, o);
        zs = make_float4(zs.x + y.x, zs.y + y.y, zs.z + y.z, zs.w + y.w);
    }
    if (lane < Q) rz[warp * Q + lane] = zs;
    __syncthreads();
    float4 Z = rz[q];
#pragma unroll
    for (int w = 1; w < NW; ++w) {
        const float4 y = rz[w * Q + q];
        Z = make_float4(Z.x + y.x, Z.y + y.y, Z.z + y.z, Z.w + y.w);
    }
    m = M;
    z = Z;
}

// The plan's heavy rows longer than cap_e edges, entries blockIdx.x,
// blockIdx.x + gridDim.x, ... of its list (interleaved, so every warp of the
// block knows the block's upcoming rows without a hand-off; the light
// batches that follow are fetched dynamically and even out the load).
// Entered and left by all threads of the block, every copy waited for.
__device__ __forceinline__ void softmax_heavy_ring(const int32_t *__restrict__ row_ptr,
                                                   const int32_t *__restrict__ heavy_rows,
                                                   int64_t n_heavy, int32_t H, int32_t cap_e,
                                                   const float *scores, float *out, float *buf,
                                                   float *red) {
    const int t = threadIdx.x, lane = t & 31;
    const int Q = H >> 2;
    const int64_t G = gridDim.x;
    for (int64_t g0 = 0; (int64_t)blockIdx.x + g0 * G < n_heavy; g0 += 32) {
        // 32 list entries at a time, one per lane (every warp the same)
        const int64_t k = (int64_t)blockIdx.x + (g0 + lane) * G;
        int32_t e0_lane = 0, deg_lane = 0;
        if (k < n_heavy) {
            const int32_t row = __ldg(heavy_rows + k);
            e0_lane = __ldg(row_ptr + row);
            deg_lane = __ldg(row_ptr + row + 1) - e0_lane;
        }
        const unsigned rows = __ballot_sync(kFull, deg_lane > cap_e);
        ChunkIssuer is{rows, 0, 0, 0, 0, 0, false, 0};
        int freed = 0, kc = 0;  // loads consumed and freed; next load to consume
        is.pump(scores, buf, H, cap_e, e0_lane, deg_lane, freed, t);
        for (unsigned left = rows; left; left &= left - 1u) {
            const int l = __ffs(left) - 1;
            const int32_t e0 = __shfl_sync(kFull, e0_lane, l);
            const int32_t deg = __shfl_sync(kFull, deg_lane, l);
            const int32_t nc = (deg + cap_e - 1) / cap_e;
            const bool resident = nc <= kResident;
            float4 m = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
            float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
            const int k_row = kc;
            for (int32_t c = 0; c < nc; ++c) {
                const int32_t dc = deg - c * cap_e < cap_e ? deg - c * cap_e : cap_e;
                cp_async_wait_upto(is.issued - 1 - kc);
                ring_fold(buf + (kc % kRing) * kSpanFloats, dc * Q, t, m, z);
                ++kc;
                if (!resident) {
                    ++freed;
                    is.pump(scores, buf, H, cap_e, e0_lane, deg_lane, freed, t);
                }
            }
            // merge over the block; an all -inf head: maximum -inf, sum 0,
            // NaN outputs (two-pass definition)
            ring_merge(m, z, Q, red);
            const float4 mg = m;
            const float4 inv = make_float4(rcp_approx(z.x), rcp_approx(z.y), rcp_approx(z.z),
                                           rcp_approx(z.w));
            for (int32_t c = 0; c < nc; ++c) {
                const int32_t dc = deg - c * cap_e < cap_e ? deg - c * cap_e : cap_e;
                int kk;
                if (resident) {
                    kk = k_row + c;  // still in its slot
                } else {
                    kk = kc++;
                    cp_async_wait_upto(is.issued - 1 - kk);
                }
                ring_write(buf + (kk % kRing) * kSpanFloats, dc * Q, t, mg, inv,
                           out + ((int64_t)e0 + c * cap_e) * H);
                ++freed;
                is.pump(scores, buf, H, cap_e, e0_lane, deg_lane, freed, t);
            }
        }
    }
}

// ---- all rows, H <= 32, one launch
//
// Phase 1 (with a plan): the plan's heavy rows longer than a warp's buffer,
// one block per row. A block takes kHeavyUnit list entries at a time from
// the plan's heavy counter (the next unit's index requested while this one
// runs); its first warp reads the unit's entries at once and keeps the rows
// above the buffer, so rows the light phase owns cost no serial round trips.
// The kept rows stream through the two halves of the block's buffer
// (softmax_heavy_rows).
// Phase 2: light rows. A warp takes batches of 32 consecutive rows (one
// coalesced row_ptr load per batch), fetched from the plan's batch counter
// when there is a plan (so blocks that had more heavy work take fewer
// batches), else by a static stride. Consecutive light rows of a batch own
// one contiguous run of scores; the warp stages such a run (at most
// kSpanFloats scores) into its buffer (one bulk copy with W = 4), computes
// it and writes it back with one bulk copy. W = 4 with Q = H/4 a power of two: rows go to register
// tiers (up to 4 or 8 float4s per lane) or, past 8 per lane, to the
// whole-warp shared-memory routine, and a row beyond the buffer that the
// plan does not call heavy streams through the warp's buffer twice;
// otherwise one thread per (row, group of W heads)
// (Q = H/W groups, R = 32/Q rows at a time, lane = r*Q + q). The last block
// to finish resets the counters for the next launch on the stream.
template <int W>
__global__ void __launch_bounds__(kSoftmaxThreads, 3)
softmax_rows_kernel(const int32_t *__restrict__ row_ptr, int64_t n_rows, int32_t H,
                    const float *scores, float *out, int32_t heavy_threshold,
                    const int32_t *__restrict__ heavy_rows, int64_t n_heavy, int32_t *sched) {
    extern __shared__ __align__(16) float span_smem[];
    __shared__ int order_smem[kSoftmaxThreads / 32][32];
    __shared__ float red[kSoftmaxThreads * 4];
    __shared__ int32_t h_e0[kHeavyUnit], h_deg[kHeavyUnit];
    __shared__ int hcount;
    __shared__ int32_t s_unit;
    __shared__ __align__(8) uint64_t wbar[kSoftmaxThreads / 32];  // light runs' bulk loads
    const int t = threadIdx.x, lane = t & 31;
    if (W == 4 && lane == 0) {
        const unsigned b = (unsigned)__cvta_generic_to_shared(&wbar[t >> 5]);
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(b) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();
    unsigned wph = 0;
    const int32_t cap_e = kSpanFloats / H;  // edges per warp buffer
    // light rows the buffer does not hold are the warps' (two passes through
    // the buffer with W = 4 and Q a power of two, else straight from global);
    // the plan's heavy rows beyond the buffer are phase 1's
    const bool tiers = W == 4 && ((H / W) & (H / W - 1)) == 0;
    if (n_heavy > 0 && tiers && H <= 32) {
        softmax_heavy_ring(row_ptr, heavy_rows, n_heavy, H, cap_e, scores, out, span_smem, red);
        cp_async_wait_all();
        // this thread's generic accesses to the buffer come before the bulk
        // loads that overwrite it
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncthreads();  // the buffer is the warps' again
    } else if (n_heavy > 0) {
        // units of kHeavyUnit list entries from the plan's second counter;
        // the next unit's index is fetched while this one is computed
        const int32_t ce = kSpanBlockFloats / 2 / H;  // edges per half buffer
        const int64_t n_units = (n_heavy + kHeavyUnit - 1) / kHeavyUnit;
        if (t == 0) s_unit = atomicAdd(sched + 1, 1);
        __syncthreads();
        int64_t unit = s_unit;
        __syncthreads();  // every thread has read s_unit before thread 0 rewrites it
        while (unit < n_units) {
            if (t < 32) {
                const int64_t k = unit * kHeavyUnit + t;
                int32_t e0 = 0, deg = 0;
                if (t < kHeavyUnit && k < n_heavy) {
                    const int32_t row = heavy_rows[k];
                    e0 = row_ptr[row];
                    deg = row_ptr[row + 1] - e0;
                }
                const unsigned hb = __ballot_sync(kFull, deg > cap_e);
                if (deg > cap_e) {
                    const int slot = __popc(hb & ((1u << t) - 1u));
                    h_e0[slot] = e0;
                    h_deg[slot] = deg;
                }
                if (t == 0) {
                    hcount = __popc(hb);
                    s_unit = atomicAdd(sched + 1, 1);
                }
            }
            __syncthreads();
            unit = s_unit;
            softmax_heavy_rows<W>(h_e0, h_deg, hcount, H, scores, out, span_smem,
                                  span_smem + kSpanBlockFloats / 2, ce, red);
            __syncthreads();
        }
        if (W == 4 && t == 0) bulk_wait_read();  // the shared buffer is the warps' again
        // this thread's generic accesses to the buffer come before the bulk
        // loads that overwrite it
        if (W == 4) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncthreads();
    }
    float *sb = span_smem + (t >> 5) * kSpanFloats;
    int *order = order_smem[t >> 5];
    const int Q = H / W, R = 32 / Q;
    const int r = lane / Q, q = lane - r * Q;
    const int64_t n_batches = (n_rows + 31) / 32;
    const int64_t n_warps = (int64_t)gridDim.x * (kSoftmaxThreads / 32);
    const bool dyn = sched != nullptr;
    auto fetch = [&]() -> int64_t {
        int32_t b = 0;
        if (lane == 0) b = atomicAdd(sched, 1);
        return __shfl_sync(kFull, b, 0);
    };
    int64_t b = dyn ? fetch() : (int64_t)blockIdx.x * (kSoftmaxThreads / 32) + (t >> 5);
    while (b < n_batches) {
        // the next batch's index is fetched now and used after this one
        const int64_t b_next = dyn ? fetch() : b + n_warps;
        if (b_next < n_batches) {  // the next batch's 33 row offsets into L2
            const int64_t rn = b_next * 32 + lane;
            if (rn <= n_rows) asm volatile("prefetch.global.L2 [%0];" ::"l"(row_ptr + rn));
        }
        const int64_t r0 = b * 32;
        const int nb = n_rows - r0 < 32 ? (int)(n_rows - r0) : 32;
        const int32_t e0_lane = row_ptr[r0 + (lane < nb ? lane : nb - 1)];
        const int32_t rp_end = row_ptr[r0 + nb];
        const int32_t nxt = __shfl_down_sync(kFull, e0_lane, 1);
        const int32_t e1_lane = lane + 1 < nb ? nxt : rp_end;
        const int32_t deg_lane = e1_lane - e0_lane;
        // a row the staging buffer holds is done here even when the plan
        // counts it heavy (phase 1 skips such rows)
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
                if (tiers && d <= heavy_threshold)  // light but too long: the warp, two passes
                    softmax_row_medium4(scores, out, sb, base, d, H, cap_e, lane);
                else if (d <= heavy_threshold)  // the same, straight from global
                    softmax_row_direct(scores, out, (int64_t)base * H, (int64_t)(base + d) * H, H,
                                       lane);
                ++i0;
                continue;
            }
            const int32_t end = __shfl_sync(kFull, e1_lane, i1 - 1);
            const int64_t x0 = (int64_t)base * H;
            const int n = (end - base) * H;
            if (n > 0) {
                // the buffer's last bulk store has read it
                if (W == 4 && lane == 0) bulk_wait_read();
                if (W == 4) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (W == 4) {
                    // the run is contiguous and 16-byte aligned (H a multiple of
                    // 4): one bulk copy, on the warp's mbarrier
                    if (lane == 0) bulk_load(sb, scores + x0, (unsigned)n * 4u, &wbar[t >> 5]);
                    mbar_wait_bounded(&wbar[t >> 5], wph);
                    wph ^= 1u;
                } else {
                    stage_in<W>(sb, scores + x0, n, lane, 32);
                }
                __syncwarp();
                const unsigned run_mask =
                    (i1 - i0 == 32 ? 0xffffffffu : ((1u << (i1 - i0)) - 1u)) << i0;
                const bool in_run = (run_mask >> lane) & 1u;
                if (tiers) {
                    const int n4 = deg_lane * Q;
                    const int need = (n4 + 3) >> 2;  // lanes at 4 float4s each
                    const int S_lane = need <= Q ? Q : 1 << (32 - __clz(need - 1));
                    // more than 8 float4s per lane: the whole warp through shared memory
                    for (unsigned lm = __ballot_sync(kFull, in_run && n4 > 256); lm; lm &= lm - 1u) {
                        const int i = __ffs(lm) - 1;
                        const int32_t ri0 = __shfl_sync(kFull, e0_lane, i);
                        const int32_t ri1 = __shfl_sync(kFull, e1_lane, i);
                        __syncwarp();
                        warp_row_softmax4(sb + (ri0 - base) * H, ri1 - ri0, H, lane);
                    }
                    // 5 .. 8 float4s per lane: the whole warp, in registers
                    const unsigned m8 = __ballot_sync(kFull, in_run && n4 > 128 && n4 <= 256);
                    if (m8)
                        softmax_tier4<8>(sb, base, H, Q, 32, m8, e0_lane, e1_lane, order, lane);
                    // up to 4 float4s per lane: tiers of S lanes per row
                    unsigned rest = __ballot_sync(kFull, in_run && n4 > 0 && n4 <= 128);
                    while (rest) {
                        const int S = __shfl_sync(kFull, S_lane, __ffs(rest) - 1);
                        const unsigned tm = __ballot_sync(kFull, ((rest >> lane) & 1u) && S_lane == S);
                        rest &= ~tm;
                        softmax_tier4<4>(sb, base, H, Q, S, tm, e0_lane, e1_lane, order, lane);
                    }
                } else {
                    if (in_run) order[lane - i0] = lane;
                    __syncwarp();
                    const int ns = i1 - i0;
                    for (int g0 = 0; g0 < ns; g0 += R) {
                        const int slot = g0 + r;
                        const bool has = r < R && slot < ns;
                        const int i = has ? order[slot] : 0;
                        const int32_t ri0 = __shfl_sync(kFull, e0_lane, i);
                        const int32_t ri1 = __shfl_sync(kFull, e1_lane, i);
                        if (has) segment_softmax<W>(sb + (ri0 - base) * H + q * W, ri1 - ri0, H);
                    }
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
        b = b_next;
    }
    if (W == 4 && lane == 0) bulk_wait_all();
    if (dyn) {
        // every warp of the block has taken its last batch index
        __syncthreads();
        if (t == 0) {
            __threadfence();
            if (atomicAdd(sched + 2, 1) == (int32_t)gridDim.x - 1) {
                sched[0] = 0;
                sched[1] = 0;
                sched[2] = 0;
                __threadfence();
            }
        }
    }
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
    // W = 4 heads per thread (16-byte accesses) when the layout allows it
    const bool vec4 = H % 4 == 0 && aligned16(scores) && aligned16(out);
    // H = 64 or 128 with 16-byte groups of four heads: Q = H/4 <= 32 head
    // groups, a power of two, as the one-launch kernel needs
    const bool wide4 = vec4 && (H == 64 || H == 128);
    const bool one_launch = H <= 32 || wide4;
    // a warp per batch of 32 rows (one launch) or per row (the others)
    const int64_t warps = one_launch ? (n_rows + 31) / 32 : n_rows;
    int64_t blocks = (warps + wpb - 1) / wpb;
    if (one_launch) {
        // one launch: the plan's heavy rows, then light batches; with a plan
        // the grid is exactly the resident blocks and batches are fetched
        // from the plan's counter
        auto kern = vec4 ? softmax_rows_kernel<4> : softmax_rows_kernel<1>;
        // the attribute and the resident-block count, once per device and kernel
        static std::atomic<int> attr_done[2][kMaxDevices];
        static std::atomic<int64_t> caps[2][kMaxDevices];
        cudaError_t err = allow_dynamic_smem(attr_done[vec4 ? 1 : 0], kern, kSpanSmemBytes);
        if (err != cudaSuccess) return cuda_fail(err, "gat_edge_softmax: shared memory attribute");
        const int64_t cap = device_blocks(caps[vec4 ? 1 : 0], kern, kSoftmaxThreads, kSpanSmemBytes);
        const int64_t n_heavy = plan ? plan->n_heavy : 0;
        if (blocks > cap || (plan && n_heavy > 0)) blocks = cap;
        kern<<<(unsigned)blocks, kSoftmaxThreads, kSpanSmemBytes, s>>>(
            row_ptr, n_rows, H, scores, out, T, plan ? plan->heavy_rows : nullptr, n_heavy,
            plan ? plan->sched : nullptr);
        return check_launch("gat_edge_softmax: rows");
    }
    {
        const int64_t cap = (int64_t)sm_count() * 8;
        if (blocks > cap) blocks = cap;
        softmax_rows_generic_kernel<<<(unsigned)blocks, kSoftmaxThreads, 0, s>>>(
            row_ptr, n_rows, H, scores, out, T);
    }
    gat_status_t st = check_launch("gat_edge_softmax: rows");
    if (st != GAT_OK) return st;
    if (plan && plan->n_heavy > 0) {
        int64_t hb = plan->n_heavy;
        const int64_t hcap = (int64_t)sm_count() * 8;
        if (hb > hcap) hb = hcap;
        softmax_heavy_kernel<<<(unsigned)hb, kSoftmaxThreads, 0, s>>>(
            row_ptr, plan->heavy_rows, plan->n_heavy, H, scores, out);
        st = check_launch("gat_edge_softmax: heavy rows");
    }
    return st;
}
