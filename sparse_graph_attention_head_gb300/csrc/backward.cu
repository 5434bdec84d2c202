// backward.cu - gradients of the fused layer (gat_fused_layer_backward).
//
// The forward computes, per row i, head h and edge e of the row (source
// j = col_idx[e]): s[e] = scale <q[i,h], k[j,h]>, a = softmax over the row's
// edges, out[i,h] = sum_e a[e] v[j,h]. Its chain rule, for the upstream
// gradient dout:
//   da[e] = <dout[i,h], v[j,h]>,  Delta = sum_e a[e] da[e],  ds[e] = a[e] (da[e] - Delta)
//   dq[i,h] = scale sum_e ds[e] k[j,h]
//   dk[j,h] = scale sum_{e reading j} ds[e] q[i(e),h]
//   dv[j,h] = sum_{e reading j} a[e] dout[i(e),h]
// dk and dv collect the contributions of every edge that reads source j;
// FW-GLM-5-1 l1_p10 (discussion of the backward pass) adds them with atomics.
// Here they are summed per source over the transposed view (transpose.cu),
// in edge order, so the result is the same on every call.
//
// Pass A (rows, CSR): one persistent kernel over the work items of the
// forward plan, the chunks of heavy rows first, then the light rows, one warp
// per item. The row's scores are recomputed in registers with the forward's
// lane layout (row_engine.cuh) and folded into an online state per head:
// m (running max, log2 units), l = sum p, S = sum p da, A = sum p da k,
// B = sum p k, with p = 2^(s - m) rescaled whenever m grows. At the row's end
// Delta = S / l and dq = scale (A - Delta B) / l, so k is gathered once. A
// heavy row's chunks write their states to the workspace and the chunk that
// finishes last (arrival counter) merges them in chunk order, as in the
// forward. Each edge's score (log2 units) and da go to the workspace, and
// each row's lse (log2 units) and Delta to a per-row table.
// Pass B (sources, CSC): one warp per light source (a block per heavy one);
// per edge it gathers dout[i] and q[i], the edge's score and da and the
// row's lse and Delta: a = 2^(s - lse), ds = a (da - Delta),
// dv += a dout[i], dk += ds q[i]; dk is scaled at the end.
// Shapes outside the vector lanes take the scalar kernels at the end.
#include <climits>
#include <type_traits>

#include "row_engine.cuh"

namespace gat {

constexpr int kBwdThreads = 128;       // light-row / light-source kernels
constexpr int kBwdHeavyThreads = 256;  // one block per heavy row or source
constexpr float kLog2eB = 1.4426950408889634f;

struct BwdParams {
    const int32_t *row_ptr, *col_idx;
    const void *q, *k, *v, *dout;
    void *dq, *dk, *dv;
    int64_t n_rows, n_src;
    int32_t H, Dh;
    int32_t hgroups;  // pass A: head groups per row (32 vectors each)
    float scale;   // the layer's score scale
    float qscale;  // scale * log2(e)
    float2 *ws;     // [E, H] (score in log2 units, da)
    float2 *stats;  // [n_rows, H] (lse in log2 units, Delta)
    // forward plan (rows): light threshold and heavy-row chunks
    int32_t row_threshold;
    int64_t n_chunks;
    const int4 *chunk_desc;      // {row, e0, e1, heavy index}
    const int32_t *chunk_start;  // [n_heavy + 1]
    int32_t *counters;           // [n_heavy], zero between calls
    float *partials;             // [n_chunks][hgroups][slot_floats]
    int64_t slot_floats;         // one head group's state, multiple of 4
    // transposed view (sources)
    const int32_t *src_ptr, *perm, *dst;
    int32_t src_threshold;
    const int32_t *heavy_src;
    int64_t n_heavy_src;
};

// 2^x by the hardware approximation (as in the forward)
__device__ __forceinline__ float bexp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ---------------------------------------------------------------------------
// pass A: rows
// ---------------------------------------------------------------------------
// Pass A works on head groups: a row's H*Dh elements are cut into HG groups
// of 32 16-byte vectors (HG = the forward's V), and one warp takes one
// (item, group) pair, lane l owning vector l of the group. A group holds
// HL = H / HG whole heads, G lanes each.
constexpr float kRescale = 8.f;  // the running max is moved only by more than this (log2 units)

// packed fp32 FMA on a pair, (a.x b.x + c.x, a.y b.y + c.y), each rounded once
__device__ __forceinline__ float2 fma_x2(float2 a, float2 b, float2 c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;"
        : "=l"(r)
        : "l"(*reinterpret_cast<uint64_t *>(&a)), "l"(*reinterpret_cast<uint64_t *>(&b)),
          "l"(*reinterpret_cast<uint64_t *>(&c)));
    return *reinterpret_cast<float2 *>(&r);
}

template <typename T, int U>
struct BwdRow {
    static constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
    using L = Lanes<T, 1, 32>;
    static constexpr int VE = L::VE;
    float qf[VE], gf[VE];  // q * qscale and dout of the row's group
    uint4 qpk, gpk;        // q and dout as stored (bf16: the dot products on the packed pairs)
    float A[VE], B[VE];
    float m, l, S;

    // this lane's q and dout vectors of (row, group g)
    __device__ __forceinline__ static void load_qg(const BwdParams &p, const L &ln, int64_t row,
                                                   int g, uint4 &qr, uint4 &gr) {
        const int64_t rb = (int64_t)p.H * p.Dh * sizeof(T);
        const int64_t off = row * rb + (int64_t)(g * 32 + ln.lane) * 16;
        qr = ld_stream16(static_cast<const char *>(p.q) + off);
        gr = ld_stream16(static_cast<const char *>(p.dout) + off);
    }

    __device__ __forceinline__ void begin(const BwdParams &p, const uint4 &qr, const uint4 &gr) {
        if (kBf16) {
            qpk = qr;
            gpk = gr;
        } else {
            Vec<T>::unpack(qr, qf);
            Vec<T>::unpack(gr, gf);
#pragma unroll
            for (int t = 0; t < VE; ++t) qf[t] *= p.qscale;
        }
#pragma unroll
        for (int t = 0; t < VE; ++t) A[t] = B[t] = 0.f;
        m = -INFINITY;
        l = 0.f;
        S = 0.f;
    }

    // edges [e0, e1) of the row, one 32-edge tile after another
    __device__ __forceinline__ void run(const BwdParams &p, const L &ln, int e0, int e1, int g) {
        const int64_t rb = (int64_t)p.H * p.Dh * sizeof(T);
        const int64_t goff = (int64_t)(g * 32 + ln.lane) * 16;
        const char *kb = static_cast<const char *>(p.k) + goff;
        const char *vb = static_cast<const char *>(p.v) + goff;
        const int HL = p.H / p.hgroups;
        const int head = g * HL + ln.head[0];
        const bool leader = ln.lane % ln.G == 0;
        for (int base = e0; base < e1; base += 32) {
            const int n = min(32, e1 - base);
            const int my_ci = ln.lane < n ? __ldg(p.col_idx + base + ln.lane) : 0;
            for (int j0 = 0; j0 < n; j0 += U) {
                uint4 kr[U], vr[U];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int64_t src = __shfl_sync(kFull, my_ci, (j0 + u) & 31);
                    if (j0 + u < n) {
                        kr[u] = ld_stream16(kb + src * rb);
                        vr[u] = ld_stream16(vb + src * rb);
                    } else {
                        kr[u] = vr[u] = make_uint4(0, 0, 0, 0);
                    }
                }
                float sc[U], da[U];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    float a = 0.f, b = 0.f;
                    if constexpr (kBf16) {
                        a = dot_bf16x8(qpk, kr[u]);  // scaled after the head's sum
                        b = dot_bf16x8(gpk, vr[u]);
                    } else {
                        float kf[VE], vf[VE];
                        Vec<T>::unpack(kr[u], kf);
                        Vec<T>::unpack(vr[u], vf);
#pragma unroll
                        for (int t = 0; t < VE; ++t) {
                            a = fmaf(qf[t], kf[t], a);
                            b = fmaf(gf[t], vf[t], b);
                        }
                    }
                    sc[u] = a;
                    da[u] = b;
                }
                for (int o = 1; o < ln.G; o <<= 1) {
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        sc[u] += __shfl_xor_sync(kFull, sc[u], o);
                        da[u] += __shfl_xor_sync(kFull, da[u], o);
                    }
                }
                if (kBf16)
#pragma unroll
                    for (int u = 0; u < U; ++u) sc[u] *= p.qscale;
                // the head's first lane records the edge's score and da
                if (leader)
#pragma unroll
                    for (int u = 0; u < U; ++u)
                        if (j0 + u < n)
                            p.ws[(int64_t)(base + j0 + u) * p.H + head] = make_float2(sc[u], da[u]);
                float mx = -INFINITY;
#pragma unroll
                for (int u = 0; u < U; ++u)
                    if (j0 + u < n) mx = fmaxf(mx, sc[u]);
                // terms are 2^(s - m) <= 2^kRescale, so the state is rescaled
                // only when a score passes the running max by more than that
                if (mx > m + kRescale) {
                    const float c = bexp2(m - mx);  // m = -inf at the start: c = 0
                    l *= c;
                    S *= c;
#pragma unroll
                    for (int t = 0; t < VE; ++t) {
                        A[t] *= c;
                        B[t] *= c;
                    }
                    m = mx;
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    if (j0 + u >= n) continue;
                    const float pe = bexp2(sc[u] - m), pd = pe * da[u];
                    l += pe;
                    S += pd;
                    float kf[VE];
                    Vec<T>::unpack(kr[u], kf);
                    const float2 pd2 = make_float2(pd, pd), pe2 = make_float2(pe, pe);
#pragma unroll
                    for (int t = 0; t < VE; t += 2) {
                        const float2 k2 = make_float2(kf[t], kf[t + 1]);
                        const float2 a2 = fma_x2(pd2, k2, make_float2(A[t], A[t + 1]));
                        const float2 b2 = fma_x2(pe2, k2, make_float2(B[t], B[t + 1]));
                        A[t] = a2.x;
                        A[t + 1] = a2.y;
                        B[t] = b2.x;
                        B[t + 1] = b2.y;
                    }
                }
            }
        }
    }

    // dq of the row's group and its heads' (lse, Delta)
    __device__ __forceinline__ void finish(const BwdParams &p, const L &ln, int64_t row, int g) {
        const int64_t rb = (int64_t)p.H * p.Dh * sizeof(T);
        const float inv = l > 0.f ? 1.f / l : 0.f;
        const float delta = S * inv;
        float o[VE];
#pragma unroll
        for (int t = 0; t < VE; ++t) o[t] = p.scale * (A[t] - delta * B[t]) * inv;
        st_stream16(static_cast<char *>(p.dq) + row * rb + (int64_t)(g * 32 + ln.lane) * 16,
                    Vec<T>::pack(o));
        if (ln.lane % ln.G == 0)
            p.stats[row * p.H + g * (p.H / p.hgroups) + ln.head[0]] =
                make_float2(m + log2f(l), delta);
    }

    // A chunk of a heavy row: publish the group's state; the warp that
    // completes the row's last (chunk, group) pair merges every group of the
    // row over its chunks in chunk order and finishes the row.
    __device__ __forceinline__ void chunk_epilogue(const BwdParams &p, const L &ln, int64_t row,
                                                   int hr, int64_t chunk, int g) {
        constexpr int HDL = 32 * VE;  // elements of a group
        const int HL = p.H / p.hgroups;
        float *slot = p.partials + (chunk * p.hgroups + g) * p.slot_floats;
#pragma unroll
        for (int t = 0; t < VE; t += 4) {
            __stcg(reinterpret_cast<float4 *>(slot + ln.lane * VE + t),
                   make_float4(A[t], A[t + 1], A[t + 2], A[t + 3]));
            __stcg(reinterpret_cast<float4 *>(slot + HDL + ln.lane * VE + t),
                   make_float4(B[t], B[t + 1], B[t + 2], B[t + 3]));
        }
        if (ln.lane % ln.G == 0) {
            __stcg(slot + 2 * HDL + ln.head[0], m);
            __stcg(slot + 2 * HDL + HL + ln.head[0], l);
            __stcg(slot + 2 * HDL + 2 * HL + ln.head[0], S);
        }
        __threadfence();
        __syncwarp();
        int old = 0;
        if (ln.lane == 0) old = atomicAdd(p.counters + hr, 1);
        old = __shfl_sync(kFull, old, 0);
        const int c0 = __ldg(p.chunk_start + hr), c1 = __ldg(p.chunk_start + hr + 1);
        if (old != (c1 - c0) * p.hgroups - 1) return;  // not the row's last piece
        __threadfence();
        for (int g2 = 0; g2 < p.hgroups; ++g2) {
            float mx = -INFINITY;
            for (int c = c0; c < c1; ++c)
                mx = fmaxf(mx, __ldcg(p.partials + ((int64_t)c * p.hgroups + g2) * p.slot_floats +
                                      2 * HDL + ln.head[0]));
            float ls = 0.f, ss = 0.f;
#pragma unroll
            for (int t = 0; t < VE; ++t) A[t] = B[t] = 0.f;
            for (int c = c0; c < c1; ++c) {
                const float *sl = p.partials + ((int64_t)c * p.hgroups + g2) * p.slot_floats;
                const float mc = __ldcg(sl + 2 * HDL + ln.head[0]);
                if (mc == -INFINITY) continue;
                const float w = bexp2(mc - mx);
                ls += w * __ldcg(sl + 2 * HDL + HL + ln.head[0]);
                ss += w * __ldcg(sl + 2 * HDL + 2 * HL + ln.head[0]);
#pragma unroll
                for (int t = 0; t < VE; t += 4) {
                    const float4 fa = ld_cg_f4(sl + ln.lane * VE + t);
                    const float4 fb = ld_cg_f4(sl + HDL + ln.lane * VE + t);
                    A[t] += w * fa.x;
                    A[t + 1] += w * fa.y;
                    A[t + 2] += w * fa.z;
                    A[t + 3] += w * fa.w;
                    B[t] += w * fb.x;
                    B[t + 1] += w * fb.y;
                    B[t + 2] += w * fb.z;
                    B[t + 3] += w * fb.w;
                }
            }
            m = mx;
            l = ls;
            S = ss;
            finish(p, ln, row, g2);
        }
        if (ln.lane == 0) p.counters[hr] = 0;  // ready for the next call
    }
};

// Persistent: warp w takes items w, w + W, ...: (chunk, group) pairs of the
// heavy rows (plan order), then (row, group) pairs of every row (heavy rows
// skipped: their chunks did them). The groups of one row go to adjacent warps.
template <typename T, int U>
__global__ void __launch_bounds__(kBwdThreads, 8)
bwd_rows_kernel(const BwdParams p) {
    using L = Lanes<T, 1, 32>;
    const L ln(p.Dh);
    BwdRow<T, U> st;
    const int64_t wpb = blockDim.x >> 5;
    const int64_t n_warps = (int64_t)gridDim.x * wpb;
    const int64_t n_items = (p.n_chunks + p.n_rows) * p.hgroups;
    for (int64_t item = (int64_t)blockIdx.x * wpb + (threadIdx.x >> 5); item < n_items;
         item += n_warps) {
        const int64_t it = item / p.hgroups;
        const int g = (int)(item - it * p.hgroups);
        int64_t row;
        int e0, e1, hr = -1;
        if (it < p.n_chunks) {
            const int4 d = __ldg(p.chunk_desc + it);
            row = d.x;
            e0 = d.y;
            e1 = d.z;
            hr = d.w;
        } else {
            row = it - p.n_chunks;
            e0 = __ldg(p.row_ptr + row);
            e1 = __ldg(p.row_ptr + row + 1);
            if (e1 - e0 > p.row_threshold) continue;
        }
        uint4 qr, gr;
        BwdRow<T, U>::load_qg(p, ln, row, g, qr, gr);
        st.begin(p, qr, gr);
        st.run(p, ln, e0, e1, g);
        if (hr >= 0)
            st.chunk_epilogue(p, ln, row, hr, it, g);
        else
            st.finish(p, ln, row, g);
    }
}

// ---------------------------------------------------------------------------
// pass B: sources
// ---------------------------------------------------------------------------
template <typename T, int V, int U>
struct BwdSrc {
    using L = Lanes<T, V, 32>;
    static constexpr int VE = L::VE;
    float dkf[V][VE], dvf[V][VE];

    __device__ __forceinline__ void zero() {
#pragma unroll
        for (int s = 0; s < V; ++s)
#pragma unroll
            for (int t = 0; t < VE; ++t) dkf[s][t] = dvf[s][t] = 0.f;
    }

    // CSC positions k0 + 32*tile0, ... below k1
    __device__ __forceinline__ void run(const BwdParams &p, const L &ln, int k0, int k1, int tile0,
                                        int step) {
        const int64_t rb = (int64_t)p.H * p.Dh * sizeof(T);
        const char *qb = static_cast<const char *>(p.q);
        const char *gb = static_cast<const char *>(p.dout);
        for (int base = k0 + tile0 * 32; base < k1; base += step * 32) {
            const int n = min(32, k1 - base);
            const int my_e = ln.lane < n ? __ldg(p.perm + base + ln.lane) : 0;
            const int my_i = ln.lane < n ? __ldg(p.dst + base + ln.lane) : 0;
            for (int j0 = 0; j0 < n; j0 += U) {
                uint4 qr[U][V], gr[U][V];
                float2 sd[U][V], ld[U][V];
                // every load of the group first, the weights after
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int64_t e = __shfl_sync(kFull, my_e, (j0 + u) & 31);
                    const int64_t i = __shfl_sync(kFull, my_i, (j0 + u) & 31);
#pragma unroll
                    for (int s = 0; s < V; ++s) {
                        if (j0 + u < n) {
                            qr[u][s] = ld_stream16(qb + i * rb + ln.vi[s] * 16);
                            gr[u][s] = ld_stream16(gb + i * rb + ln.vi[s] * 16);
                            sd[u][s] = __ldcg(p.ws + e * p.H + ln.head[s]);
                            ld[u][s] = __ldcg(p.stats + i * p.H + ln.head[s]);
                        } else {
                            qr[u][s] = gr[u][s] = make_uint4(0, 0, 0, 0);
                            sd[u][s] = make_float2(-INFINITY, 0.f);
                            ld[u][s] = make_float2(0.f, 0.f);
                        }
                    }
                }
                float wa[U][V], wd[U][V];
#pragma unroll
                for (int u = 0; u < U; ++u)
#pragma unroll
                    for (int s = 0; s < V; ++s) {
                        const float a = bexp2(sd[u][s].x - ld[u][s].x);  // invalid: 2^-inf = 0
                        wa[u][s] = a;
                        wd[u][s] = a * (sd[u][s].y - ld[u][s].y);
                    }
#pragma unroll
                for (int u = 0; u < U; ++u)
#pragma unroll
                    for (int s = 0; s < V; ++s) {
                        float qv[VE], gv[VE];
                        Vec<T>::unpack(qr[u][s], qv);
                        Vec<T>::unpack(gr[u][s], gv);
#pragma unroll
                        for (int t = 0; t < VE; ++t) {
                            dkf[s][t] = fmaf(wd[u][s], qv[t], dkf[s][t]);
                            dvf[s][t] = fmaf(wa[u][s], gv[t], dvf[s][t]);
                        }
                    }
            }
        }
    }

    __device__ __forceinline__ void store(const BwdParams &p, const L &ln, int64_t j) {
        const int64_t rb = (int64_t)p.H * p.Dh * sizeof(T);
        char *krow = static_cast<char *>(p.dk) + j * rb;
        char *vrow = static_cast<char *>(p.dv) + j * rb;
#pragma unroll
        for (int s = 0; s < V; ++s) {
            float o[VE];
#pragma unroll
            for (int t = 0; t < VE; ++t) o[t] = p.scale * dkf[s][t];
            st_stream16(krow + ln.vi[s] * 16, Vec<T>::pack(o));
            st_stream16(vrow + ln.vi[s] * 16, Vec<T>::pack(dvf[s]));
        }
    }
};

template <typename T, int V, int U>
__global__ void __launch_bounds__(kBwdThreads)
bwd_src_kernel(const BwdParams p) {
    using L = Lanes<T, V, 32>;
    const L ln(p.Dh);
    BwdSrc<T, V, U> st;
    const int64_t wpb = blockDim.x >> 5;
    const int64_t n_warps = (int64_t)gridDim.x * wpb;
    for (int64_t j = (int64_t)blockIdx.x * wpb + (threadIdx.x >> 5); j < p.n_src; j += n_warps) {
        const int k0 = __ldg(p.src_ptr + j), k1 = __ldg(p.src_ptr + j + 1);
        if (k1 - k0 > p.src_threshold) continue;  // a heavy source: the block kernel's
        st.zero();
        st.run(p, ln, k0, k1, 0, 1);
        st.store(p, ln, j);
    }
}

template <typename T, int V, int U>
__global__ void __launch_bounds__(kBwdHeavyThreads)
bwd_heavy_src_kernel(const BwdParams p) {
    using L = Lanes<T, V, 32>;
    constexpr int VE = L::VE;
    constexpr int NW = kBwdHeavyThreads / 32;
    constexpr int SF = 2 * V * VE;
    extern __shared__ float sm[];  // [NW][SF][32]
    const L ln(p.Dh);
    const int warp = threadIdx.x >> 5;
    BwdSrc<T, V, U> st;
    for (int64_t b = blockIdx.x; b < p.n_heavy_src; b += gridDim.x) {
        const int64_t j = __ldg(p.heavy_src + b);
        const int k0 = __ldg(p.src_ptr + j), k1 = __ldg(p.src_ptr + j + 1);
        st.zero();
        st.run(p, ln, k0, k1, warp, NW);
        float *my = sm + warp * SF * 32 + ln.lane;
#pragma unroll
        for (int s = 0; s < V; ++s)
#pragma unroll
            for (int t = 0; t < VE; ++t) {
                my[((s * VE + t) * 2) * 32] = st.dkf[s][t];
                my[((s * VE + t) * 2 + 1) * 32] = st.dvf[s][t];
            }
        __syncthreads();
        if (warp == 0) {
#pragma unroll
            for (int s = 0; s < V; ++s)
#pragma unroll
                for (int t = 0; t < VE; ++t) {
                    float a = 0.f, c = 0.f;
                    for (int w = 0; w < NW; ++w) {
                        a += sm[w * SF * 32 + ((s * VE + t) * 2) * 32 + ln.lane];
                        c += sm[w * SF * 32 + ((s * VE + t) * 2 + 1) * 32 + ln.lane];
                    }
                    st.dkf[s][t] = a;
                    st.dvf[s][t] = c;
                }
            st.store(p, ln, j);
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------
// scalar kernels (any H, Dh, alignment): one warp per row / source, lanes
// over a head's Dh elements, heads one at a time
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(kBwdThreads)
bwd_rows_generic_kernel(const BwdParams p) {
    const int lane = threadIdx.x & 31;
    const int64_t wpb = blockDim.x >> 5;
    const int64_t n_warps = (int64_t)gridDim.x * wpb;
    const T *q = static_cast<const T *>(p.q), *k = static_cast<const T *>(p.k);
    const T *v = static_cast<const T *>(p.v), *g = static_cast<const T *>(p.dout);
    T *dq = static_cast<T *>(p.dq);
    const int64_t HD = (int64_t)p.H * p.Dh;
    for (int64_t row = (int64_t)blockIdx.x * wpb + (threadIdx.x >> 5); row < p.n_rows;
         row += n_warps) {
        const int64_t e0 = __ldg(p.row_ptr + row), e1 = __ldg(p.row_ptr + row + 1);
        for (int h = 0; h < p.H; ++h) {
            const int64_t qo = row * HD + (int64_t)h * p.Dh;
            float m = -INFINITY;
            for (int64_t e = e0; e < e1; ++e) {  // scores (log2 units) and da
                const int64_t ko = (int64_t)__ldg(p.col_idx + e) * HD + (int64_t)h * p.Dh;
                float a = 0.f, b = 0.f;
                for (int d = lane; d < p.Dh; d += 32) {
                    a = fmaf(load_elem(q, qo + d), load_elem(k, ko + d), a);
                    b = fmaf(load_elem(g, qo + d), load_elem(v, ko + d), b);
                }
                a = warp_sum(a) * p.qscale;
                b = warp_sum(b);
                if (lane == 0) p.ws[e * p.H + h] = make_float2(a, b);
                m = fmaxf(m, a);
            }
            __syncwarp();
            float l = 0.f, sd = 0.f;
            for (int64_t e = e0 + lane; e < e1; e += 32) {
                const float2 w = p.ws[e * p.H + h];
                const float pe = bexp2(w.x - m);
                l += pe;
                sd += pe * w.y;
            }
            l = warp_sum(l);
            sd = warp_sum(sd);
            const float lse = m + log2f(l), delta = l > 0.f ? sd / l : 0.f;
            if (lane == 0) p.stats[row * p.H + h] = make_float2(lse, delta);
            for (int d = lane; d < p.Dh; d += 32) {
                float acc = 0.f;
                for (int64_t e = e0; e < e1; ++e) {
                    const float2 w = p.ws[e * p.H + h];
                    const float a = bexp2(w.x - lse);
                    const float ds = a * (w.y - delta);
                    acc = fmaf(ds,
                               load_elem(k, (int64_t)__ldg(p.col_idx + e) * HD + (int64_t)h * p.Dh + d),
                               acc);
                }
                store_elem(dq, qo + d, p.scale * acc);
            }
            __syncwarp();
        }
    }
}

template <typename T>
__global__ void __launch_bounds__(kBwdThreads)
bwd_src_generic_kernel(const BwdParams p) {
    const int lane = threadIdx.x & 31;
    const int64_t wpb = blockDim.x >> 5;
    const int64_t n_warps = (int64_t)gridDim.x * wpb;
    const T *q = static_cast<const T *>(p.q), *g = static_cast<const T *>(p.dout);
    T *dk = static_cast<T *>(p.dk), *dv = static_cast<T *>(p.dv);
    const int64_t HD = (int64_t)p.H * p.Dh;
    for (int64_t j = (int64_t)blockIdx.x * wpb + (threadIdx.x >> 5); j < p.n_src; j += n_warps) {
        const int64_t k0 = __ldg(p.src_ptr + j), k1 = __ldg(p.src_ptr + j + 1);
        for (int64_t x = lane; x < HD; x += 32) {
            const int h = (int)(x / p.Dh);
            float ak = 0.f, av = 0.f;
            for (int64_t kk = k0; kk < k1; ++kk) {
                const int64_t e = __ldg(p.perm + kk), i = __ldg(p.dst + kk);
                const float2 w = __ldcg(p.ws + e * p.H + h), st = p.stats[i * p.H + h];
                const float a = bexp2(w.x - st.x);
                const float ds = a * (w.y - st.y);
                ak = fmaf(ds, load_elem(q, i * HD + x), ak);
                av = fmaf(a, load_elem(g, i * HD + x), av);
            }
            store_elem(dk, j * HD + x, p.scale * ak);
            store_elem(dv, j * HD + x, av);
        }
    }
}

// ---------------------------------------------------------------------------
// launch
// ---------------------------------------------------------------------------
template <typename K>
static int64_t resident(K kern, int threads, int smem) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, smem) != cudaSuccess ||
        per_sm < 1)
        per_sm = 1;
    return (int64_t)sm_count() * per_sm;
}

template <typename K>
static gat_status_t launch_grid(K kern, int64_t items, int threads, int smem, const BwdParams &p,
                                cudaStream_t s, const char *what) {
    if (items <= 0) return GAT_OK;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return cuda_fail(e, what);
    }
    int64_t blocks = items;
    const int64_t cap = resident(kern, threads, smem);
    if (blocks > cap) blocks = cap;
    kern<<<(unsigned)blocks, threads, smem, s>>>(p);
    return check_launch(what);
}

template <typename T, int V>
static gat_status_t launch_bwd_fast(const BwdParams &p, cudaStream_t s) {
    constexpr int UA = 2;                              // edges in flight, pass A
    constexpr int UB = V == 4 ? 1 : (V == 2 ? 3 : 4);  // pass B
    constexpr int VE = 16 / (int)sizeof(T);
    const int wpb = kBwdThreads / 32;
    gat_status_t st = launch_grid(bwd_rows_kernel<T, UA>,
                                  ((p.n_chunks + p.n_rows) * p.hgroups + wpb - 1) / wpb,
                                  kBwdThreads, 0, p, s, "backward rows");
    if (st != GAT_OK) return st;
    st = launch_grid(bwd_src_kernel<T, V, UB>, (p.n_src + wpb - 1) / wpb, kBwdThreads, 0, p, s,
                     "backward sources");
    if (st != GAT_OK) return st;
    const int hsm_b = kBwdHeavyThreads / 32 * 2 * V * VE * 32 * (int)sizeof(float);
    return launch_grid(bwd_heavy_src_kernel<T, V, UB>, p.n_heavy_src, kBwdHeavyThreads, hsm_b, p, s,
                       "backward heavy sources");
}

template <typename T>
static gat_status_t launch_bwd(BwdParams p, bool vec_ok, cudaStream_t s) {
    int V = 0, LE = 0;
    if (vec_ok && engine_shape(p.H, p.Dh, sizeof(T), V, LE) && LE == 32) {
        if (V == 1) return launch_bwd_fast<T, 1>(p, s);
        if (V == 2) return launch_bwd_fast<T, 2>(p, s);
        if (V == 4) return launch_bwd_fast<T, 4>(p, s);
    }
    const int wpb = kBwdThreads / 32;
    gat_status_t st = launch_grid(bwd_rows_generic_kernel<T>, (p.n_rows + wpb - 1) / wpb,
                                  kBwdThreads, 0, p, s, "backward rows (scalar)");
    if (st != GAT_OK) return st;
    return launch_grid(bwd_src_generic_kernel<T>, (p.n_src + wpb - 1) / wpb, kBwdThreads, 0, p, s,
                       "backward sources (scalar)");
}

static size_t round256(size_t x) { return (x + 255) & ~(size_t)255; }

// Workspace: (score, da) [E,H], row (lse, Delta) [n_rows,H], then (with a
// plan of heavy rows on the vector path) one chunk state per chunk.
struct BwdLayout {
    size_t ws_off, st_off, part_off, total;
};

static BwdLayout bwd_layout(int64_t n_rows, int64_t n_edges, int32_t H, int32_t Dh,
                            int64_t n_chunks) {
    BwdLayout L{};
    L.ws_off = 0;
    L.st_off = round256((size_t)n_edges * (size_t)H * sizeof(float2));
    L.part_off = L.st_off + round256((size_t)n_rows * 2 * (size_t)H * sizeof(float));
    // head groups of 32 vectors: at most H*Dh/128 of them (fp32), each state
    // 2*(elements) + 3*(heads) floats rounded up to a multiple of 4
    const int64_t hg_max = ((int64_t)H * Dh + 127) / 128;
    const int64_t per_chunk = 2 * (int64_t)H * Dh + 3 * (int64_t)H + 3 * hg_max;
    L.total = L.part_off + round256((size_t)n_chunks * (size_t)per_chunk * sizeof(float));
    return L;
}

}  // namespace gat

using namespace gat;

extern "C" gat_status_t gat_fused_layer_backward_workspace_size(gat_plan_t plan, int64_t n_rows,
                                                                int64_t n_edges, int32_t H,
                                                                int32_t Dh, size_t *bytes) {
    if (!bytes) return fail(GAT_ERR_INVALID_ARG, "gat_fused_layer_backward_workspace_size: NULL");
    if (n_rows < 0 || n_edges < 0 || H < 1 || Dh < 1)
        return fail(GAT_ERR_INVALID_ARG, "gat_fused_layer_backward_workspace_size: bad sizes");
    if (plan && (plan->n_rows != n_rows || plan->n_edges != n_edges))
        return fail(GAT_ERR_PLAN_MISMATCH, "gat_fused_layer_backward_workspace_size: plan mismatch");
    *bytes = bwd_layout(n_rows, n_edges, H, Dh, plan ? plan->n_chunks : 0).total;
    return GAT_OK;
}

extern "C" gat_status_t gat_fused_layer_backward(
    const int32_t *row_ptr, const int32_t *col_idx, int64_t n_rows, int64_t n_src,
    int64_t n_edges, int32_t H, int32_t Dh, float scale, const void *q, const void *k,
    const void *v, const void *dout, gat_dtype_t dtype, void *dq, void *dk, void *dv,
    gat_plan_t plan, gat_transpose_t transpose, void *workspace, size_t workspace_bytes,
    void *stream) {
    if (n_rows < 0 || n_src < 0 || n_edges < 0 || H < 1 || Dh < 1)
        return fail(GAT_ERR_INVALID_ARG, "gat_fused_layer_backward: bad sizes");
    if (dtype != GAT_F32 && dtype != GAT_BF16)
        return fail(GAT_ERR_UNSUPPORTED, "gat_fused_layer_backward: unknown dtype %d", (int)dtype);
    if (!transpose)
        return fail(GAT_ERR_INVALID_ARG, "gat_fused_layer_backward: a transpose is required");
    if (transpose->n_rows != n_rows || transpose->n_src != n_src || transpose->n_edges != n_edges)
        return fail(GAT_ERR_PLAN_MISMATCH,
                    "gat_fused_layer_backward: transpose is for n_rows=%lld n_src=%lld n_edges=%lld",
                    (long long)transpose->n_rows, (long long)transpose->n_src,
                    (long long)transpose->n_edges);
    if (plan && (plan->n_rows != n_rows || plan->n_edges != n_edges))
        return fail(GAT_ERR_PLAN_MISMATCH, "gat_fused_layer_backward: plan is for n_rows=%lld n_edges=%lld",
                    (long long)plan->n_rows, (long long)plan->n_edges);
    if (n_rows == 0 && n_src == 0) return GAT_OK;
    if (!row_ptr || (n_rows > 0 && (!q || !dout || !dq)) || (n_src > 0 && (!dk || !dv)) ||
        (n_edges > 0 && (!col_idx || !k || !v)))
        return fail(GAT_ERR_INVALID_ARG, "gat_fused_layer_backward: NULL pointer");
    const BwdLayout lay = bwd_layout(n_rows, n_edges, H, Dh, plan ? plan->n_chunks : 0);
    if (lay.total > 0 && (!workspace || workspace_bytes < lay.total ||
                          (reinterpret_cast<uintptr_t>(workspace) & 15u)))
        return fail(GAT_ERR_WORKSPACE,
                    "gat_fused_layer_backward: workspace of %zu bytes (16-byte aligned) needed",
                    lay.total);
    BwdParams p{};
    p.row_ptr = row_ptr;
    p.col_idx = col_idx;
    p.q = q;
    p.k = k;
    p.v = v;
    p.dout = dout;
    p.dq = dq;
    p.dk = dk;
    p.dv = dv;
    p.n_rows = n_rows;
    p.n_src = n_src;
    p.H = H;
    p.Dh = Dh;
    p.hgroups = 1;
    p.scale = scale;
    p.qscale = scale * kLog2eB;
    char *wsb = static_cast<char *>(workspace);
    p.ws = reinterpret_cast<float2 *>(wsb + lay.ws_off);
    p.stats = reinterpret_cast<float2 *>(wsb + lay.st_off);
    p.row_threshold = INT_MAX;
    p.src_threshold = INT_MAX;
    p.src_ptr = transpose->src_ptr;
    p.perm = transpose->perm;
    p.dst = transpose->dst;
    const int eb = dtype == GAT_F32 ? 4 : 2;
    const bool vec_ok = aligned16(q) && aligned16(dout) && aligned16(dq) &&
                        (n_edges == 0 || (aligned16(k) && aligned16(v))) &&
                        (n_src == 0 || (aligned16(dk) && aligned16(dv)));
    int V, LE;
    if (vec_ok && engine_shape(H, Dh, eb, V, LE) && LE == 32) {
        p.hgroups = V;
        if (plan && plan->n_chunks > 0) {
            p.row_threshold = plan->heavy_threshold;
            p.n_chunks = plan->n_chunks;
            p.chunk_desc = plan->chunk_desc;
            p.chunk_start = plan->chunk_start;
            p.counters = plan->counters;
            p.partials = reinterpret_cast<float *>(wsb + lay.part_off);
            const int64_t hl = H / V, hdl = (int64_t)H * Dh / V;
            p.slot_floats = (2 * hdl + 3 * hl + 3) & ~(int64_t)3;
        }
        if (transpose->src_plan && transpose->src_plan->n_heavy > 0) {
            p.src_threshold = transpose->src_plan->heavy_threshold;
            p.heavy_src = transpose->src_plan->heavy_rows;
            p.n_heavy_src = transpose->src_plan->n_heavy;
        }
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (dtype == GAT_F32) return launch_bwd<float>(p, vec_ok, s);
    return launch_bwd<__nv_bfloat16>(p, vec_ok, s);
}
