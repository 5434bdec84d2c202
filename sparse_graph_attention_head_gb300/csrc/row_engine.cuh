// row_engine.cuh - the gather/aggregate engine behind gat_fused_layer and
// gat_spmm_weighted.
//
// Layout of the work: one warp owns one destination row (or one fixed-size
// edge chunk of a heavy row). The row's H*Dh features are spread over the
// warp's lanes in 16-byte vectors, so every gathered feature row of a source
// node is read as full, coalesced 16-byte accesses (the float4 idea of the
// spmm page's vectorised draft, taken to bf16 and to all heads at once).
//
//   LE == 32: a row has V*32 vectors; lane l owns vectors l, l+32, ...,
//             l+32(V-1) ("slots"); the warp walks the row's edges one by one.
//   LE <  32: a row has LE vectors (V == 1); the warp is split into 32/LE
//             edge subgroups, each walking every (32/LE)-th edge, and the
//             subgroups' states are merged at the end of the row.
// A head's Dh elements are G = Dh/VE consecutive vectors, i.e. G adjacent
// lanes of one slot, so a per-head dot product is a G-lane xor-shuffle sum.
//
// Fused mode (SDDMM -> softmax -> SpMM, single pass): the score of each edge
// is formed in registers and folded into an online softmax state (m, l, acc)
// per head: m' = max(m, s), c = 2^(m-m'), l = l c + 2^(s-m'),
// acc = acc c + 2^(s-m') v. Scores are pre-scaled by log2(e) so the
// exponentials are exp2. Nothing per edge ever reaches memory.
// Given-score mode (gat_softmax_aggregate): the same online softmax over
// scores read from w[e,h] (scaled by qscale = log2(e)) instead of q.k.
// SpMM mode (spmm.cu): acc += w[e,h] * feat[src].
//
// Heavy rows (fused mode, with a plan) arrive as chunks; each chunk warp
// writes its (m, l, acc) to a workspace slot, and the warp that finishes a
// row's last chunk (arrival counter) merges all of that row's chunk states in
// chunk order - deterministic, and without any spin-wait.
#pragma once

#include <climits>

#include "common.cuh"

namespace gat {

constexpr int kEngineThreads = 256;  // 8 warps per block

struct EngineParams {
    const int32_t *row_ptr;
    const int32_t *col_idx;
    const void *q;    // fused: [n_rows, H, Dh]
    const void *k;    // fused: [n_src, H, Dh]
    const void *v;    // [n_src, H, Dh] (fused: values; spmm: features)
    const float *w;   // spmm: [n_edges, w_stride], this call's heads from column 0
    int32_t w_stride; // spmm: weights per edge (H, or more for a head group)
    void *out;        // [n_rows, H, Dh]
    int64_t n_rows;
    int32_t H, Dh;
    int64_t row_elems;  // fused: elements per q/k/v/out row (H * Dh, or more for a head group)
    float qscale;     // fused: scale * log2(e)
    // light/heavy split (no plan: heavy_threshold = INT_MAX, n_chunks = 0)
    int32_t heavy_threshold;
    int32_t chunk_edges;
    int64_t n_chunks;
    const int32_t *heavy_rows;
    const int32_t *chunk_start;
    const int32_t *chunk_row;
    const int4 *chunk_desc;  // [n_chunks] {row, e0, e1, heavy index}
    int32_t *counters;
    float *partials;       // [n_chunks][slot_floats]
    int64_t slot_floats;   // >= H*Dh + 2H, multiple of 4
    // spmm heavy-row kernel: list of rows handled one block per row
    int64_t n_block_rows;
};

// Vector-engine shape selection (shared by the fused layer and the SpMM):
// V vectors per lane and LE lanes per edge for H heads of Dh elements of
// elem_bytes each; false when the shape needs the scalar fallback.
bool engine_shape(int H, int Dh, int elem_bytes, int &V, int &LE);

// Bytes-per-chunk-slot helper: floats in one chunk state (acc, m, l), padded
// to a multiple of four.
int64_t slot_floats(int H, int Dh);

// Grid size for a persistent kernel: at most `want` blocks, at most as many
// as can be resident on the device at once.
template <typename K>
inline int64_t persistent_blocks(K kernel, int64_t want) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kEngineThreads, 0) !=
            cudaSuccess ||
        per_sm < 1)
        per_sm = 1;
    const int64_t cap = (int64_t)sm_count() * per_sm;
    if (want > cap) want = cap;
    return want < 1 ? 1 : want;
}

template <typename T, int V, int LE>
struct Lanes {
    static constexpr int VE = Vec<T>::N;
    static constexpr int ES = 32 / LE;  // edge subgroups per warp
    int lane, sub, vi[V], head[V], G;
    __device__ __forceinline__ Lanes(int Dh) {
        lane = threadIdx.x & 31;
        sub = lane / LE;
        G = Dh / VE;
#pragma unroll
        for (int s = 0; s < V; ++s) {
            vi[s] = (LE == 32) ? s * 32 + lane : (lane % LE);
            head[s] = vi[s] / G;
        }
    }
};

// 2^x with the hardware's approximate exp2 (relative error about 2^-22;
// subnormal results flush to zero, far below any softmax weight that matters;
// 2^-inf = 0).
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Work item metadata {row, e0, e1, heavy index or -1}, issued as loads whose
// results are only needed when the item starts (so they overlap the previous
// item): one 16-byte descriptor for a chunk, two row_ptr entries for a row.
__device__ __forceinline__ int4 item_meta(const EngineParams &p, int64_t item) {
    if (item < p.n_chunks) return __ldg(p.chunk_desc + item);
    const int64_t row = item - p.n_chunks;
    return make_int4((int)row, __ldg(p.row_ptr + row), __ldg(p.row_ptr + row + 1), -1);
}

// ---------------------------------------------------------------------------
// fused mode
// ---------------------------------------------------------------------------
template <typename T, int V, int LE, int U>
struct FusedRow {
    using L = Lanes<T, V, LE>;
    static constexpr int VE = L::VE;
    static constexpr int ES = L::ES;
    static constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
    float qf[V][VE];  // q * qscale (bf16: q as stored in qpk, scaled after the dot)
    uint4 qpk[V];
    float acc[V][VE];
    float m[V], l[V];

    __device__ __forceinline__ void load_q(const EngineParams &p, const L &ln, int64_t row) {
        const char *qrow = static_cast<const char *>(p.q) + row * p.row_elems * (int64_t)sizeof(T);
#pragma unroll
        for (int s = 0; s < V; ++s) {
            uint4 u = ld_stream16(qrow + ln.vi[s] * 16);
            if (kBf16) {
                qpk[s] = u;
            } else {
                Vec<T>::unpack(u, qf[s]);
#pragma unroll
                for (int t = 0; t < VE; ++t) qf[s][t] *= p.qscale;
            }
        }
    }

    // Walk edges [e0, e1). first_ci is this lane's col_idx[e0 + lane] (already
    // loaded). Right after the first batch's gathers are issued, the col_idx
    // tile of the warp's next item [ne0, ne1) is fetched into next_ci
    // (next_ready), so the next item can start gathering at once; a next
    // item that is a light-row slot beyond the threshold is not fetched.
    // GIVEN: the edges' scores are read from w (no k rows, no q).
    template <bool GIVEN>
    __device__ __forceinline__ void run(const EngineParams &p, const L &ln, int e0, int e1,
                                        int first_ci, int ne0, int ne1, bool next_is_row,
                                        int &next_ci, bool &next_ready) {
#pragma unroll
        for (int s = 0; s < V; ++s) {
            m[s] = -INFINITY;
            l[s] = 0.f;
#pragma unroll
            for (int t = 0; t < VE; ++t) acc[s][t] = 0.f;
        }
        const int64_t row_bytes = p.row_elems * (int64_t)sizeof(T);
        const char *kb = static_cast<const char *>(p.k);
        const char *vb = static_cast<const char *>(p.v);
        for (int base = e0; base < e1; base += 32) {
            const int n = min(32, e1 - base);
            const int my_ci =
                base == e0 ? first_ci : (ln.lane < n ? __ldg(p.col_idx + base + ln.lane) : 0);
            for (int j0 = 0; j0 < n; j0 += U * ES) {
                uint4 kr[U][V], vr[U][V];
                bool valid[U];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int j = j0 + u * ES + ln.sub;
                    valid[u] = j < n;
                    const int64_t src = __shfl_sync(kFull, my_ci, j & 31);
                    if (valid[u]) {
#pragma unroll
                        for (int s = 0; s < V; ++s) {
                            if (!GIVEN) kr[u][s] = ld_stream16(kb + src * row_bytes + ln.vi[s] * 16);
                            vr[u][s] = ld_stream16(vb + src * row_bytes + ln.vi[s] * 16);
                        }
                    } else {
#pragma unroll
                        for (int s = 0; s < V; ++s) {
                            kr[u][s] = make_uint4(0, 0, 0, 0);
                            vr[u][s] = make_uint4(0, 0, 0, 0);
                        }
                    }
                }
                if (base == e0 && j0 == 0 && !next_ready) {
                    const int nn = ne1 - ne0;
                    if (nn > 0 && !(next_is_row && nn > p.heavy_threshold)) {
                        next_ci = ln.lane < nn ? __ldg(p.col_idx + ne0 + ln.lane) : 0;
                        next_ready = true;
                    }
                }
                float sc[U][V];
                if constexpr (GIVEN) {
                    // every lane of a head reads the edge's score of that head
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        const int64_t e = base + j0 + u * ES + ln.sub;
#pragma unroll
                        for (int s = 0; s < V; ++s)
                            sc[u][s] = valid[u] ? __ldg(p.w + e * p.w_stride + ln.head[s]) * p.qscale
                                                : 0.f;
                    }
                } else {
#pragma unroll
                    for (int u = 0; u < U; ++u)
#pragma unroll
                        for (int s = 0; s < V; ++s) {
                            if constexpr (kBf16) {
                                sc[u][s] = dot_bf16x8(qpk[s], kr[u][s]);
                            } else {
                                float kf[VE];
                                Vec<T>::unpack(kr[u][s], kf);
                                float d = 0.f;
#pragma unroll
                                for (int t = 0; t < VE; ++t) d = fmaf(qf[s][t], kf[t], d);
                                sc[u][s] = d;
                            }
                        }
                    // per-head sums over the head's G lanes (uniform across the warp)
                    for (int o = 1; o < ln.G; o <<= 1) {
#pragma unroll
                        for (int u = 0; u < U; ++u)
#pragma unroll
                            for (int s = 0; s < V; ++s)
                                sc[u][s] += __shfl_xor_sync(kFull, sc[u][s], o);
                    }
                    if (kBf16)
#pragma unroll
                        for (int u = 0; u < U; ++u)
#pragma unroll
                            for (int s = 0; s < V; ++s) sc[u][s] *= p.qscale;
                }
#pragma unroll
                for (int s = 0; s < V; ++s) {
                    float mx = m[s];
#pragma unroll
                    for (int u = 0; u < U; ++u)
                        if (valid[u]) mx = fmaxf(mx, sc[u][s]);
                    if (mx == -INFINITY) continue;  // no edge for this subgroup yet
                    const float c = fast_exp2(m[s] - mx);
                    l[s] *= c;
#pragma unroll
                    for (int t = 0; t < VE; ++t) acc[s][t] *= c;
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        const float pe = valid[u] ? fast_exp2(sc[u][s] - mx) : 0.f;
                        l[s] += pe;
                        float vf[VE];
                        Vec<T>::unpack(vr[u][s], vf);
#pragma unroll
                        for (int t = 0; t < VE; ++t) acc[s][t] = fmaf(pe, vf[t], acc[s][t]);
                    }
                    m[s] = mx;
                }
            }
        }
        // merge the edge subgroups' states (LE < 32)
#pragma unroll
        for (int o = LE; o < 32; o <<= 1) {
#pragma unroll
            for (int s = 0; s < V; ++s) {
                const float m2 = __shfl_xor_sync(kFull, m[s], o);
                const float l2 = __shfl_xor_sync(kFull, l[s], o);
                float a2[VE];
#pragma unroll
                for (int t = 0; t < VE; ++t) a2[t] = __shfl_xor_sync(kFull, acc[s][t], o);
                const float mx = fmaxf(m[s], m2);
                if (mx == -INFINITY) continue;
                const float c1 = fast_exp2(m[s] - mx), c2 = fast_exp2(m2 - mx);
                l[s] = l[s] * c1 + l2 * c2;
#pragma unroll
                for (int t = 0; t < VE; ++t) acc[s][t] = acc[s][t] * c1 + a2[t] * c2;
                m[s] = mx;
            }
        }
    }

    // masked_nan: the row has edges, so a head with no finite score (l = 0,
    // possible only with given scores of -inf) is NaN, as the two-pass softmax
    __device__ __forceinline__ void store_out(const EngineParams &p, const L &ln, int64_t row,
                                              bool masked_nan = false) {
        if (ln.sub != 0) return;
        char *orow = static_cast<char *>(p.out) + row * p.row_elems * (int64_t)sizeof(T);
#pragma unroll
        for (int s = 0; s < V; ++s) {
            const float inv = l[s] > 0.f ? 1.f / l[s] : (masked_nan ? NAN : 0.f);
            float o[VE];
#pragma unroll
            for (int t = 0; t < VE; ++t) o[t] = acc[s][t] * inv;
            st_stream16(orow + ln.vi[s] * 16, Vec<T>::pack(o));
        }
    }

    // chunk of a heavy row: publish the state; the last chunk merges the row
    __device__ __forceinline__ void chunk_epilogue(const EngineParams &p, const L &ln, int64_t row,
                                                   int hr, int64_t chunk, bool masked_nan = false) {
        const int HD = p.H * p.Dh;
        if (ln.sub == 0) {
            float *slot = p.partials + chunk * p.slot_floats;
#pragma unroll
            for (int s = 0; s < V; ++s) {
                float *a = slot + ln.vi[s] * VE;
#pragma unroll
                for (int t = 0; t < VE; t += 4)
                    __stcg(reinterpret_cast<float4 *>(a + t),
                           make_float4(acc[s][t], acc[s][t + 1], acc[s][t + 2], acc[s][t + 3]));
                if (ln.vi[s] % ln.G == 0) {
                    __stcg(slot + HD + ln.head[s], m[s]);
                    __stcg(slot + HD + p.H + ln.head[s], l[s]);
                }
            }
        }
        __threadfence();
        __syncwarp();
        int old = 0;
        if (ln.lane == 0) old = atomicAdd(p.counters + hr, 1);
        old = __shfl_sync(kFull, old, 0);
        const int c0 = __ldg(p.chunk_start + hr), c1 = __ldg(p.chunk_start + hr + 1);
        if (old != c1 - c0 - 1) return;  // not the last chunk of this row
        __threadfence();
        // merge all chunk states of the row in chunk order
#pragma unroll
        for (int s = 0; s < V; ++s) {
            m[s] = -INFINITY;
            l[s] = 0.f;
#pragma unroll
            for (int t = 0; t < VE; ++t) acc[s][t] = 0.f;
        }
        for (int c = c0; c < c1; ++c) {
            const float *slot = p.partials + (int64_t)c * p.slot_floats;
#pragma unroll
            for (int s = 0; s < V; ++s) {
                const float mc = __ldcg(slot + HD + ln.head[s]);
                const float lc = __ldcg(slot + HD + p.H + ln.head[s]);
                float ac[VE];
#pragma unroll
                for (int t = 0; t < VE; t += 4) {
                    float4 f = ld_cg_f4(slot + ln.vi[s] * VE + t);
                    ac[t] = f.x;
                    ac[t + 1] = f.y;
                    ac[t + 2] = f.z;
                    ac[t + 3] = f.w;
                }
                const float mx = fmaxf(m[s], mc);
                if (mx == -INFINITY) continue;
                const float a1 = fast_exp2(m[s] - mx), a2 = fast_exp2(mc - mx);
                l[s] = l[s] * a1 + lc * a2;
#pragma unroll
                for (int t = 0; t < VE; ++t) acc[s][t] = acc[s][t] * a1 + ac[t] * a2;
                m[s] = mx;
            }
        }
        store_out(p, ln, row, masked_nan);
        if (ln.lane == 0) p.counters[hr] = 0;  // ready for the next call
    }
};

// Persistent: warp w takes items w, w + W, w + 2W, ... (chunks of heavy rows
// first, then rows). While an item is processed, the next item's metadata
// (and, once that arrives, its first col_idx tile) is already being fetched.
// Blocks of 4 warps, MINB resident per SM (5 -> 96 registers, 20 warps/SM).
constexpr int kFusedThreads = 128;

template <typename T, int V, int LE, int U, int MINB, bool GIVEN = false>
__global__ void __launch_bounds__(kFusedThreads, MINB)
fused_engine_kernel(const EngineParams p) {
    using L = Lanes<T, V, LE>;
    const L ln(p.Dh);
    FusedRow<T, V, LE, U> st;
    const int64_t wpb = blockDim.x >> 5;
    const int64_t n_warps = (int64_t)gridDim.x * wpb;
    const int64_t n_items = p.n_chunks + p.n_rows;
    int64_t item = (int64_t)blockIdx.x * wpb + (threadIdx.x >> 5);
    if (item >= n_items) return;
    int4 meta = item_meta(p, item);
    int ci_tile = 0;
    bool ci_ready = false;
    for (; item < n_items; item += n_warps) {
        const int4 cur = meta;  // {row, e0, e1, heavy index or -1}
        const int64_t nxt = item + n_warps;
        const bool has_next = nxt < n_items;
        meta = has_next ? item_meta(p, nxt) : make_int4(0, 0, 0, -1);
        const bool is_chunk = item < p.n_chunks;
        if (!is_chunk && cur.z - cur.y > p.heavy_threshold) {  // a heavy row: done as chunks
            ci_ready = false;
            continue;
        }
        const int first_ci =
            ci_ready ? ci_tile : (ln.lane < cur.z - cur.y ? __ldg(p.col_idx + cur.y + ln.lane) : 0);
        bool next_ready = false;
        if (!GIVEN) st.load_q(p, ln, cur.x);
        st.template run<GIVEN>(p, ln, cur.y, cur.z, first_ci, has_next ? meta.y : 0, has_next ? meta.z : 0,
               nxt >= p.n_chunks, ci_tile, next_ready);
        ci_ready = next_ready;
        if (!is_chunk)
            st.store_out(p, ln, cur.x, GIVEN && cur.z > cur.y);
        else
            st.chunk_epilogue(p, ln, cur.x, cur.w, item, GIVEN);
    }
}

// Host-side launch of the fused engine for one (T, V, LE): U edges in flight
// per warp (V=1: 4, V=2: 3, V=4: 1), five resident 4-warp blocks per SM.
template <typename T, int V, int LE, bool GIVEN = false>
inline gat_status_t launch_fused_engine(const EngineParams &p, cudaStream_t s) {
    constexpr int U = V == 1 ? 4 : (V == 2 ? 3 : 1);
    auto kern = fused_engine_kernel<T, V, LE, U, 5, GIVEN>;
    static std::atomic<int64_t> caps[kMaxDevices];
    const int64_t cap = device_blocks(caps, kern, kFusedThreads, 0);
    const int64_t items = p.n_chunks + p.n_rows;
    const int64_t wpb = kFusedThreads / 32;
    int64_t blocks = (items + wpb - 1) / wpb;
    if (blocks > cap) blocks = cap;
    kern<<<(unsigned)blocks, kFusedThreads, 0, s>>>(p);
    return check_launch("fused_engine_kernel");
}

}  // namespace gat
