// spmm.cu - gat_spmm_weighted: out[i,h,:] = sum_e w[e,h] * feat[col_idx[e],h,:]
// (FW-GLM-5-1 l1_p18, reference model; Kimi-K2.6 l2_p37: a destination with
// no edges stays zero). One warp per row, persistent, with the next item's
// metadata prefetched. Heavy rows of a plan: with a workspace, cut into
// chunks in the same launch and summed by the last chunk in chunk order;
// without one, one 8-warp block per row in a second launch, warps summed in
// warp order. Lane layout: row_engine.cuh. A shape the vector kernels do not
// take whole runs as groups of heads they take, one launch per group.
#include <climits>

#include "row_engine.cuh"

namespace gat {

// Scalar fallback: one warp per row; lanes over the row's H*Dh elements in
// groups of 32 * MAXT.
template <typename T>
__global__ void __launch_bounds__(kEngineThreads)
spmm_generic_kernel(const EngineParams p) {
    constexpr int MAXT = 8;
    const int lane = threadIdx.x & 31;
    const int64_t wpb = blockDim.x >> 5;
    const int64_t n_warps = (int64_t)gridDim.x * wpb;
    const T *feat = static_cast<const T *>(p.v);
    T *out = static_cast<T *>(p.out);
    const int64_t HD = (int64_t)p.H * p.Dh;
    for (int64_t row = (int64_t)blockIdx.x * wpb + (threadIdx.x >> 5); row < p.n_rows;
         row += n_warps) {
        const int e0 = __ldg(p.row_ptr + row), e1 = __ldg(p.row_ptr + row + 1);
        for (int64_t x0 = 0; x0 < HD; x0 += 32 * MAXT) {
            float acc[MAXT];
#pragma unroll
            for (int t = 0; t < MAXT; ++t) acc[t] = 0.f;
            for (int e = e0; e < e1; ++e) {
                const int64_t src = __ldg(p.col_idx + e);
#pragma unroll
                for (int t = 0; t < MAXT; ++t) {
                    const int64_t x = x0 + lane + 32 * t;
                    if (x < HD)
                        acc[t] = fmaf(__ldg(p.w + (int64_t)e * p.H + x / p.Dh),
                                      load_elem(feat, src * HD + x), acc[t]);
                }
            }
#pragma unroll
            for (int t = 0; t < MAXT; ++t) {
                const int64_t x = x0 + lane + 32 * t;
                if (x < HD) store_elem(out, row * HD + x, acc[t]);
            }
        }
    }
}

// Accumulator of one warp: acc += w[e,h] * feat[col_idx[e],h,:] over 32-edge
// tiles, U edges (per edge subgroup) in flight at a time.
template <typename T, int V, int LE, int U>
struct SpmmAcc {
    using L = Lanes<T, V, LE>;
    static constexpr int VE = L::VE;
    static constexpr int ES = L::ES;
    float acc[V][VE];

    __device__ __forceinline__ void zero() {
#pragma unroll
        for (int s = 0; s < V; ++s)
#pragma unroll
            for (int t = 0; t < VE; ++t) acc[s][t] = 0.f;
    }

    // Tiles e0 + 32*tile0, e0 + 32*(tile0 + tile_step), ... below e1. first_ci
    // is this lane's col_idx entry of the first tile when have_first. Right
    // after the first gathers are issued, the col_idx tile of [ne0, ne1) is
    // fetched into next_ci when want_next (so the warp's next row can start
    // gathering at once).
    __device__ __forceinline__ void run(const EngineParams &p, const L &ln, int e0, int e1,
                                        int tile0, int tile_step, int first_ci, bool have_first,
                                        int ne0, int ne1, bool want_next, int &next_ci,
                                        bool &next_ready) {
        const int64_t row_bytes = p.row_elems * (int64_t)sizeof(T);
        const char *fb = static_cast<const char *>(p.v);
        const int first = e0 + tile0 * 32;
        for (int base = first; base < e1; base += tile_step * 32) {
            const int n = min(32, e1 - base);
            const int my_ci = (have_first && base == first)
                                  ? first_ci
                                  : (ln.lane < n ? __ldg(p.col_idx + base + ln.lane) : 0);
            for (int j0 = 0; j0 < n; j0 += U * ES) {
                uint4 vr[U][V];
                float wv[U][V];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int j = j0 + u * ES + ln.sub;
                    const bool valid = j < n;
                    const int64_t src = __shfl_sync(kFull, my_ci, j & 31);
#pragma unroll
                    for (int s = 0; s < V; ++s) {
                        if (valid) {
                            vr[u][s] = ld_stream16(fb + src * row_bytes + ln.vi[s] * 16);
                            wv[u][s] = __ldg(p.w + (int64_t)(base + j) * p.w_stride + ln.head[s]);
                        } else {
                            vr[u][s] = make_uint4(0, 0, 0, 0);
                            wv[u][s] = 0.f;
                        }
                    }
                }
                if (want_next && !next_ready) {
                    const int nn = ne1 - ne0;
                    next_ci = ln.lane < nn ? __ldg(p.col_idx + ne0 + ln.lane) : 0;
                    next_ready = true;
                }
#pragma unroll
                for (int u = 0; u < U; ++u)
#pragma unroll
                    for (int s = 0; s < V; ++s) {
                        float vf[VE];
                        Vec<T>::unpack(vr[u][s], vf);
#pragma unroll
                        for (int t = 0; t < VE; ++t) acc[s][t] = fmaf(wv[u][s], vf[t], acc[s][t]);
                    }
            }
        }
    }

    // sum the edge subgroups (LE < 32) in a fixed butterfly order
    __device__ __forceinline__ void merge_subgroups() {
#pragma unroll
        for (int o = LE; o < 32; o <<= 1)
#pragma unroll
            for (int s = 0; s < V; ++s)
#pragma unroll
                for (int t = 0; t < VE; ++t) acc[s][t] += __shfl_xor_sync(kFull, acc[s][t], o);
    }

    __device__ __forceinline__ void store_out(const EngineParams &p, const L &ln, int64_t row) {
        if (ln.sub != 0) return;
        char *orow = static_cast<char *>(p.out) + row * p.row_elems * (int64_t)sizeof(T);
#pragma unroll
        for (int s = 0; s < V; ++s) st_stream16(orow + ln.vi[s] * 16, Vec<T>::pack(acc[s]));
    }

    // A chunk of a heavy row: publish the chunk's sum; the warp that finishes
    // the row's last chunk (arrival counter) adds the row's chunk sums in
    // chunk order and writes the row.
    __device__ __forceinline__ void chunk_epilogue(const EngineParams &p, const L &ln, int64_t row,
                                                   int hr, int64_t chunk) {
        if (ln.sub == 0) {
            float *slot = p.partials + chunk * p.slot_floats;
#pragma unroll
            for (int s = 0; s < V; ++s)
#pragma unroll
                for (int t = 0; t < VE; t += 4)
                    __stcg(reinterpret_cast<float4 *>(slot + ln.vi[s] * VE + t),
                           make_float4(acc[s][t], acc[s][t + 1], acc[s][t + 2], acc[s][t + 3]));
        }
        __threadfence();
        __syncwarp();
        int old = 0;
        if (ln.lane == 0) old = atomicAdd(p.counters + hr, 1);
        old = __shfl_sync(kFull, old, 0);
        const int c0 = __ldg(p.chunk_start + hr), c1 = __ldg(p.chunk_start + hr + 1);
        if (old != c1 - c0 - 1) return;  // not the row's last chunk
        __threadfence();
        zero();
        for (int c = c0; c < c1; ++c) {
            const float *slot = p.partials + (int64_t)c * p.slot_floats;
#pragma unroll
            for (int s = 0; s < V; ++s)
#pragma unroll
                for (int t = 0; t < VE; t += 4) {
                    const float4 f = ld_cg_f4(slot + ln.vi[s] * VE + t);
                    acc[s][t] += f.x;
                    acc[s][t + 1] += f.y;
                    acc[s][t + 2] += f.z;
                    acc[s][t + 3] += f.w;
                }
        }
        store_out(p, ln, row);
        if (ln.lane == 0) p.counters[hr] = 0;  // ready for the next call
    }
};

// Persistent warps, warp w takes items w, w + W, ...: with a plan and a
// workspace, the chunks of heavy rows first, then every row (heavy rows
// skipped: their chunks or the heavy-row kernel do them). While an item is
// processed, the next item's metadata and then its first col_idx tile are
// already being fetched.
constexpr int kSpmmThreads = 128;

template <typename T, int V, int LE, int U>
__global__ void __launch_bounds__(kSpmmThreads, V == 4 ? 4 : (V == 2 && sizeof(T) == 2 ? 6 : 8))
spmm_rows_kernel(const EngineParams p) {
    using L = Lanes<T, V, LE>;
    const L ln(p.Dh);
    SpmmAcc<T, V, LE, U> st;
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
        if (!is_chunk && cur.z - cur.y > p.heavy_threshold) {
            ci_ready = false;
            continue;
        }
        const int first_ci =
            ci_ready ? ci_tile : (ln.lane < cur.z - cur.y ? __ldg(p.col_idx + cur.y + ln.lane) : 0);
        const int nn = meta.z - meta.y;
        const bool want_next =
            has_next && nn > 0 && (nxt < p.n_chunks || nn <= p.heavy_threshold);
        bool next_ready = false;
        st.zero();
        st.run(p, ln, cur.y, cur.z, 0, 1, first_ci, true, meta.y, meta.z, want_next, ci_tile,
               next_ready);
        ci_ready = next_ready;
        st.merge_subgroups();
        if (is_chunk)
            st.chunk_epilogue(p, ln, cur.x, cur.w, item);
        else
            st.store_out(p, ln, cur.x);
    }
}

// Heavy rows: one block of kSpmmHeavyThreads per row (8 warps); warp w takes
// 32-edge tiles w, w + 8, ... The warps' sums meet in shared memory and each
// output element is summed over the warps in warp order (deterministic).
constexpr int kSpmmHeavyThreads = 256;

template <typename T, int V, int LE, int U>
__global__ void __launch_bounds__(kSpmmHeavyThreads)
spmm_heavy_kernel(const EngineParams p) {
    using L = Lanes<T, V, LE>;
    constexpr int VE = L::VE;
    constexpr int NW = kSpmmHeavyThreads / 32;
    constexpr int PER_WARP = V * VE * 32;  // floats of one warp's row sum
    extern __shared__ float red[];          // [NW][PER_WARP]
    const L ln(p.Dh);
    const int warp = threadIdx.x >> 5;
    SpmmAcc<T, V, LE, U> st;
    int dummy_ci = 0;
    bool dummy_ready = false;
    for (int64_t b = blockIdx.x; b < p.n_block_rows; b += gridDim.x) {
        const int64_t row = __ldg(p.heavy_rows + b);
        const int e0 = __ldg(p.row_ptr + row), e1 = __ldg(p.row_ptr + row + 1);
        st.zero();
        st.run(p, ln, e0, e1, warp, NW, 0, false, 0, 0, false, dummy_ci, dummy_ready);
        st.merge_subgroups();
#pragma unroll
        for (int s = 0; s < V; ++s)
#pragma unroll
            for (int t = 0; t < VE; ++t) red[warp * PER_WARP + (s * VE + t) * 32 + ln.lane] = st.acc[s][t];
        __syncthreads();
        for (int i = threadIdx.x; i < PER_WARP; i += kSpmmHeavyThreads) {
            float a = red[i];
            for (int w2 = 1; w2 < NW; ++w2) a += red[w2 * PER_WARP + i];
            red[i] = a;
        }
        __syncthreads();
        if (warp == 0) {
#pragma unroll
            for (int s = 0; s < V; ++s)
#pragma unroll
                for (int t = 0; t < VE; ++t) st.acc[s][t] = red[(s * VE + t) * 32 + ln.lane];
            st.store_out(p, ln, row);
        }
        __syncthreads();
    }
}

// The widest head group g (g divides H) whose (g, Dh) the vector kernels
// cover; 0 when there is none. Heads are independent, so a row is summed
// group by group, each group a slice of every feature / output row and of
// every edge's weights.
static int spmm_group(int H, int Dh, int elem_bytes) {
    int V, LE;
    for (int g = H; g >= 1; --g)
        if (H % g == 0 && engine_shape(g, Dh, elem_bytes, V, LE)) return g;
    return 0;
}

template <typename T, int V, int LE>
static gat_status_t launch_spmm_fast(const EngineParams &p, cudaStream_t s) {
    constexpr int U = V == 4 ? 2 : 3;  // edges in flight per warp (3 KB at V = 2, fp32)
    auto kern = spmm_rows_kernel<T, V, LE, U>;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kSpmmThreads, 0) !=
            cudaSuccess ||
        per_sm < 1)
        per_sm = 1;
    const int64_t wpb = kSpmmThreads / 32;
    int64_t blocks = (p.n_chunks + p.n_rows + wpb - 1) / wpb;
    const int64_t cap = (int64_t)sm_count() * per_sm;
    if (blocks > cap) blocks = cap;
    kern<<<(unsigned)blocks, kSpmmThreads, 0, s>>>(p);
    gat_status_t st = check_launch("gat_spmm_weighted");
    if (st != GAT_OK || p.n_block_rows == 0) return st;
    auto hk = spmm_heavy_kernel<T, V, LE, U>;
    const int smem = kSpmmHeavyThreads / 32 * V * Vec<T>::N * 32 * (int)sizeof(float);
    cudaError_t err = cudaFuncSetAttribute(hk, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return cuda_fail(err, "gat_spmm_weighted: shared memory attribute");
    int hper_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&hper_sm, hk, kSpmmHeavyThreads, smem) !=
            cudaSuccess ||
        hper_sm < 1)
        hper_sm = 1;
    const int64_t hcap = (int64_t)sm_count() * hper_sm;
    const int64_t hb = p.n_block_rows < hcap ? p.n_block_rows : hcap;
    hk<<<(unsigned)hb, kSpmmHeavyThreads, smem, s>>>(p);
    return check_launch("gat_spmm_weighted: heavy rows");
}

template <typename T>
static gat_status_t launch_spmm(EngineParams p, bool vec_ok, cudaStream_t s) {
    int V = 0, LE = 0;
    if (vec_ok && engine_shape(p.H, p.Dh, sizeof(T), V, LE)) {
        if (V == 1 && LE == 4) return launch_spmm_fast<T, 1, 4>(p, s);
        if (V == 1 && LE == 8) return launch_spmm_fast<T, 1, 8>(p, s);
        if (V == 1 && LE == 16) return launch_spmm_fast<T, 1, 16>(p, s);
        if (V == 1 && LE == 32) return launch_spmm_fast<T, 1, 32>(p, s);
        if (V == 2) return launch_spmm_fast<T, 2, 32>(p, s);
        if (V == 4) return launch_spmm_fast<T, 4, 32>(p, s);
    }
    static std::atomic<int64_t> caps[kMaxDevices];
    const int64_t cap = device_blocks(caps, spmm_generic_kernel<T>, kEngineThreads, 0);
    const int64_t wpb = kEngineThreads / 32;
    int64_t blocks = (p.n_rows + wpb - 1) / wpb;
    if (blocks > cap) blocks = cap;
    spmm_generic_kernel<T><<<(unsigned)blocks, kEngineThreads, 0, s>>>(p);
    return check_launch("gat_spmm_weighted (scalar)");
}

}  // namespace gat

using namespace gat;

extern "C" gat_status_t gat_spmm_weighted_workspace_size(gat_plan_t plan, int32_t H, int32_t Dh,
                                                         size_t *bytes) {
    if (!bytes || H < 1 || Dh < 1)
        return fail(GAT_ERR_INVALID_ARG, "gat_spmm_weighted_workspace_size: bad arguments");
    const int64_t slot = ((int64_t)H * Dh + 3) / 4 * 4;
    *bytes = plan ? (size_t)plan->n_chunks * (size_t)slot * sizeof(float) : 0;
    return GAT_OK;
}

extern "C" gat_status_t gat_spmm_weighted(const int32_t *row_ptr, const int32_t *col_idx,
                                          int64_t n_rows, int64_t n_src, int64_t n_edges,
                                          int32_t H, int32_t Dh, const float *w, const void *feat,
                                          gat_dtype_t dtype, void *out, gat_plan_t plan,
                                          void *workspace, size_t workspace_bytes, void *stream) {
    if (n_rows < 0 || n_src < 0 || n_edges < 0 || H < 1 || Dh < 1)
        return fail(GAT_ERR_INVALID_ARG, "gat_spmm_weighted: bad sizes");
    if (dtype != GAT_F32 && dtype != GAT_BF16)
        return fail(GAT_ERR_UNSUPPORTED, "gat_spmm_weighted: unknown dtype %d", (int)dtype);
    if (n_rows == 0) return GAT_OK;
    if (!row_ptr || !out || (n_edges > 0 && (!col_idx || !w || !feat)))
        return fail(GAT_ERR_INVALID_ARG, "gat_spmm_weighted: NULL pointer");
    if (plan && (plan->n_rows != n_rows || plan->n_edges != n_edges))
        return fail(GAT_ERR_PLAN_MISMATCH,
                    "gat_spmm_weighted: plan is for n_rows=%lld n_edges=%lld",
                    (long long)plan->n_rows, (long long)plan->n_edges);
    EngineParams p{};
    p.row_ptr = row_ptr;
    p.col_idx = col_idx;
    p.v = feat;
    p.w = w;
    p.out = out;
    p.n_rows = n_rows;
    p.H = H;
    p.Dh = Dh;
    p.row_elems = (int64_t)H * Dh;
    p.w_stride = H;
    p.heavy_threshold = INT_MAX;
    p.slot_floats = ((int64_t)H * Dh + 3) / 4 * 4;
    const bool vec_ok = aligned16(out) && (n_edges == 0 || aligned16(feat));
    const int eb = dtype == GAT_F32 ? 4 : 2;
    const int Hg = vec_ok ? spmm_group(H, Dh, eb) : 0;
    if (plan && Hg > 0 && plan->n_heavy > 0) {
        p.heavy_threshold = plan->heavy_threshold;
        const size_t need = (size_t)plan->n_chunks * (size_t)p.slot_floats * sizeof(float);
        if (workspace && workspace_bytes >= need && aligned16(workspace)) {
            // heavy rows as chunks in the same launch
            p.n_chunks = plan->n_chunks;
            p.chunk_desc = plan->chunk_desc;
            p.chunk_start = plan->chunk_start;
            p.counters = plan->counters;
            p.partials = static_cast<float *>(workspace);
        } else if (workspace) {
            return fail(GAT_ERR_WORKSPACE,
                        "gat_spmm_weighted: workspace needs %zu bytes (16-byte aligned), got %zu",
                        need, workspace_bytes);
        } else {
            // no workspace: one thread block per heavy row, second launch
            p.heavy_rows = plan->heavy_rows;
            p.n_block_rows = plan->n_heavy;
        }
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (Hg > 0 && Hg < H) {
        // one launch (or two, with block-per-row heavy rows) per group of Hg
        // heads over the slices at head h0: rows keep their full stride
        // (row_elems), weights theirs (w_stride = H); Dh * elem_bytes is a
        // multiple of 16, so every slice stays 16-byte aligned
        for (int h0 = 0; h0 < H; h0 += Hg) {
            EngineParams pg = p;
            const size_t off = (size_t)h0 * Dh * eb;
            pg.H = Hg;
            pg.out = static_cast<char *>(out) + off;
            if (n_edges > 0) {
                pg.v = static_cast<const char *>(feat) + off;
                pg.w = w + h0;
            }
            const gat_status_t st = dtype == GAT_F32 ? launch_spmm<float>(pg, true, s)
                                                     : launch_spmm<__nv_bfloat16>(pg, true, s);
            if (st != GAT_OK) return st;
        }
        return GAT_OK;
    }
    if (dtype == GAT_F32) return launch_spmm<float>(p, vec_ok, s);
    return launch_spmm<__nv_bfloat16>(p, vec_ok, s);
}
