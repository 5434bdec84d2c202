// fused_layer.cu - gat_fused_layer: SDDMM -> segmented softmax -> weighted
// SpMM in one pass over the CSR graph (see row_engine.cuh for the layout and
// the online-softmax recurrence). This file holds the launch logic (a shape
// the vector engine does not cover whole runs as groups of heads it does
// cover, one launch per group) and the scalar fallback for the rest.
#include <climits>

#include "row_engine.cuh"

namespace gat {

constexpr float kLog2e = 1.4426950408889634f;

// Scalar fallback: one warp per row, one head at a time, lanes over Dh.
template <typename T>
__global__ void __launch_bounds__(kEngineThreads)
fused_generic_kernel(const EngineParams p) {
    constexpr int MAXT = 16;  // Dh <= 32 * MAXT
    const int lane = threadIdx.x & 31;
    const int64_t wpb = blockDim.x >> 5;
    const int64_t n_warps = (int64_t)gridDim.x * wpb;
    const T *q = static_cast<const T *>(p.q);
    const T *k = static_cast<const T *>(p.k);
    const T *v = static_cast<const T *>(p.v);
    T *out = static_cast<T *>(p.out);
    const int64_t HD = (int64_t)p.H * p.Dh;
    for (int64_t row = (int64_t)blockIdx.x * wpb + (threadIdx.x >> 5); row < p.n_rows;
         row += n_warps) {
        const int e0 = __ldg(p.row_ptr + row), e1 = __ldg(p.row_ptr + row + 1);
        for (int h = 0; h < p.H; ++h) {
            float qv[MAXT], acc[MAXT];
#pragma unroll
            for (int t = 0; t < MAXT; ++t) {
                const int d = lane + 32 * t;
                qv[t] = d < p.Dh ? load_elem(q, row * HD + h * p.Dh + d) * p.qscale : 0.f;
                acc[t] = 0.f;
            }
            float m = -INFINITY, l = 0.f;
            for (int e = e0; e < e1; ++e) {
                const int64_t src = __ldg(p.col_idx + e);
                const int64_t base = src * HD + (int64_t)h * p.Dh;
                float dot = 0.f;
#pragma unroll
                for (int t = 0; t < MAXT; ++t) {
                    const int d = lane + 32 * t;
                    if (d < p.Dh) dot = fmaf(qv[t], load_elem(k, base + d), dot);
                }
                dot = warp_sum(dot);
                const float mx = fmaxf(m, dot);
                const float c = exp2f(m - mx), pe = exp2f(dot - mx);
                l = l * c + pe;
#pragma unroll
                for (int t = 0; t < MAXT; ++t) {
                    const int d = lane + 32 * t;
                    acc[t] = acc[t] * c + (d < p.Dh ? pe * load_elem(v, base + d) : 0.f);
                }
                m = mx;
            }
            const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
            for (int t = 0; t < MAXT; ++t) {
                const int d = lane + 32 * t;
                if (d < p.Dh) store_elem(out, row * HD + h * p.Dh + d, acc[t] * inv);
            }
        }
    }
}

template <typename T, int V, int LE>
static gat_status_t launch_fused_fast(const EngineParams &p, cudaStream_t s) {
    return launch_fused_engine<T, V, LE>(p, s);
}

bool engine_shape(int H, int Dh, int elem_bytes, int &V, int &LE) {
    const int VE = 16 / elem_bytes;
    if (Dh % VE) return false;
    const int DV = Dh / VE;
    if (DV & (DV - 1)) return false;  // lanes per head must be a power of two
    const int64_t nvec = (int64_t)H * DV;
    if (nvec >= 32) {
        if (nvec % 32 || DV > 32) return false;
        V = (int)(nvec / 32);
        if (V != 1 && V != 2 && V != 4) return false;
        LE = 32;
        return true;
    }
    if (nvec < 4 || (nvec & (nvec - 1))) return false;
    V = 1;
    LE = (int)nvec;
    return true;
}

template <typename T>
static gat_status_t launch_fused(EngineParams p, bool vec_ok, cudaStream_t s) {
    int V = 0, LE = 0;
    if (vec_ok && engine_shape(p.H, p.Dh, sizeof(T), V, LE)) {
        if (V == 1 && LE == 4) return launch_fused_fast<T, 1, 4>(p, s);
        if (V == 1 && LE == 8) return launch_fused_fast<T, 1, 8>(p, s);
        if (V == 1 && LE == 16) return launch_fused_fast<T, 1, 16>(p, s);
        if (V == 1 && LE == 32) return launch_fused_fast<T, 1, 32>(p, s);
        if (V == 2) return launch_fused_fast<T, 2, 32>(p, s);
        if (V == 4) return launch_fused_fast<T, 4, 32>(p, s);
    }
    if (p.Dh > 32 * 16)
        return fail(GAT_ERR_UNSUPPORTED, "gat_fused_layer: Dh=%d not supported by the scalar path",
                    (int)p.Dh);
    // the scalar path handles every row whole: no chunks, no workspace
    p.n_chunks = 0;
    p.heavy_threshold = INT_MAX;
    static std::atomic<int64_t> caps[kMaxDevices];
    const int64_t cap = device_blocks(caps, fused_generic_kernel<T>, kEngineThreads, 0);
    const int64_t wpb = kEngineThreads / 32;
    int64_t blocks = (p.n_rows + wpb - 1) / wpb;
    if (blocks > cap) blocks = cap;
    fused_generic_kernel<T><<<(unsigned)blocks, kEngineThreads, 0, s>>>(p);
    return check_launch("gat_fused_layer (scalar)");
}

// The widest head group g (g divides H) whose (g, Dh) the vector engine
// covers; 0 when there is none. Heads are independent in the layer, so a row
// is computed group by group, each group a slice of every q/k/v/out row.
static int engine_group(int H, int Dh, int elem_bytes) {
    int V, LE;
    for (int g = H; g >= 1; --g)
        if (H % g == 0 && engine_shape(g, Dh, elem_bytes, V, LE)) return g;
    return 0;
}

int64_t slot_floats(int H, int Dh) {
    const int64_t f = (int64_t)H * Dh + 2 * (int64_t)H;
    return (f + 3) / 4 * 4;
}

}  // namespace gat

using namespace gat;

extern "C" gat_status_t gat_fused_layer_workspace_size(gat_plan_t plan, int32_t H, int32_t Dh,
                                                       size_t *bytes) {
    if (!bytes || H < 1 || Dh < 1)
        return fail(GAT_ERR_INVALID_ARG, "gat_fused_layer_workspace_size: bad arguments");
    *bytes = plan ? (size_t)plan->n_chunks * (size_t)slot_floats(H, Dh) * sizeof(float) : 0;
    return GAT_OK;
}

extern "C" gat_status_t gat_fused_layer(const int32_t *row_ptr, const int32_t *col_idx,
                                        int64_t n_rows, int64_t n_src, int64_t n_edges, int32_t H,
                                        int32_t Dh, float scale, const void *q, const void *k,
                                        const void *v, gat_dtype_t dtype, void *out,
                                        gat_plan_t plan, void *workspace, size_t workspace_bytes,
                                        void *stream) {
    if (n_rows < 0 || n_src < 0 || n_edges < 0 || H < 1 || Dh < 1)
        return fail(GAT_ERR_INVALID_ARG, "gat_fused_layer: bad sizes");
    if (dtype != GAT_F32 && dtype != GAT_BF16)
        return fail(GAT_ERR_UNSUPPORTED, "gat_fused_layer: unknown dtype %d", (int)dtype);
    if (n_rows == 0) return GAT_OK;
    if (!row_ptr || !q || !out || (n_edges > 0 && (!col_idx || !k || !v)))
        return fail(GAT_ERR_INVALID_ARG, "gat_fused_layer: NULL pointer");
    if (plan && (plan->n_rows != n_rows || plan->n_edges != n_edges))
        return fail(GAT_ERR_PLAN_MISMATCH, "gat_fused_layer: plan is for n_rows=%lld n_edges=%lld",
                    (long long)plan->n_rows, (long long)plan->n_edges);
    EngineParams p{};
    p.row_ptr = row_ptr;
    p.col_idx = col_idx;
    p.q = q;
    p.k = k;
    p.v = v;
    p.out = out;
    p.n_rows = n_rows;
    p.H = H;
    p.Dh = Dh;
    p.row_elems = (int64_t)H * Dh;
    p.qscale = scale * kLog2e;
    p.heavy_threshold = INT_MAX;
    p.chunk_edges = 1;
    p.slot_floats = slot_floats(H, Dh);
    const int eb = dtype == GAT_F32 ? 4 : 2;
    const bool vec_ok = aligned16(q) && aligned16(out) && (n_edges == 0 || (aligned16(k) && aligned16(v)));
    const int Hg = vec_ok ? engine_group(H, Dh, eb) : 0;
    const bool fast = Hg > 0;
    if (plan && fast) {
        p.heavy_threshold = plan->heavy_threshold;
        p.chunk_edges = plan->chunk_edges;
        p.n_chunks = plan->n_chunks;
        p.heavy_rows = plan->heavy_rows;
        p.chunk_start = plan->chunk_start;
        p.chunk_row = plan->chunk_row;
        p.chunk_desc = plan->chunk_desc;
        p.counters = plan->counters;
        if (p.n_chunks > 0) {
            const size_t need = (size_t)p.n_chunks * (size_t)p.slot_floats * sizeof(float);
            if (!workspace || workspace_bytes < need || !aligned16(workspace))
                return fail(GAT_ERR_WORKSPACE,
                            "gat_fused_layer: workspace needs %zu bytes (16-byte aligned), got %zu",
                            need, workspace_bytes);
            p.partials = static_cast<float *>(workspace);
        }
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (fast && Hg < H) {
        // one launch per group of Hg heads over the slices of the rows at
        // head h0 (Dh * elem_bytes is a multiple of 16, so every slice keeps
        // the 16-byte alignment); the chunk states of a launch fit the
        // workspace sized for all H heads, and each launch leaves the plan's
        // arrival counters at zero for the next
        for (int h0 = 0; h0 < H; h0 += Hg) {
            EngineParams pg = p;
            const size_t off = (size_t)h0 * Dh * eb;
            pg.H = Hg;
            pg.q = static_cast<const char *>(q) + off;
            pg.out = static_cast<char *>(out) + off;
            if (n_edges > 0) {
                pg.k = static_cast<const char *>(k) + off;
                pg.v = static_cast<const char *>(v) + off;
            }
            const gat_status_t st = dtype == GAT_F32 ? launch_fused<float>(pg, true, s)
                                                     : launch_fused<__nv_bfloat16>(pg, true, s);
            if (st != GAT_OK) return st;
        }
        return GAT_OK;
    }
    if (dtype == GAT_F32) return launch_fused<float>(p, vec_ok, s);
    return launch_fused<__nv_bfloat16>(p, vec_ok, s);
}

// ---------------------------------------------------------------------------
// softmax of given edge scores + aggregation, one launch
// ---------------------------------------------------------------------------
namespace gat {

template <typename T>
static gat_status_t launch_given(const EngineParams &p, cudaStream_t s) {
    int V = 0, LE = 0;
    if (!engine_shape(p.H, p.Dh, sizeof(T), V, LE))
        return fail(GAT_ERR_UNSUPPORTED, "gat_softmax_aggregate: shape H=%d Dh=%d", (int)p.H,
                    (int)p.Dh);
    if (V == 1 && LE == 4) return launch_fused_engine<T, 1, 4, true>(p, s);
    if (V == 1 && LE == 8) return launch_fused_engine<T, 1, 8, true>(p, s);
    if (V == 1 && LE == 16) return launch_fused_engine<T, 1, 16, true>(p, s);
    if (V == 1 && LE == 32) return launch_fused_engine<T, 1, 32, true>(p, s);
    if (V == 2) return launch_fused_engine<T, 2, 32, true>(p, s);
    return launch_fused_engine<T, 4, 32, true>(p, s);
}

}  // namespace gat

extern "C" gat_status_t gat_softmax_aggregate(const int32_t *row_ptr, const int32_t *col_idx,
                                              int64_t n_rows, int64_t n_src, int64_t n_edges,
                                              int32_t H, int32_t Dh, const float *scores,
                                              const void *feat, gat_dtype_t dtype, void *out,
                                              gat_plan_t plan, void *workspace,
                                              size_t workspace_bytes, void *stream) {
    if (n_rows < 0 || n_src < 0 || n_edges < 0 || H < 1 || Dh < 1)
        return fail(GAT_ERR_INVALID_ARG, "gat_softmax_aggregate: bad sizes");
    if (dtype != GAT_F32 && dtype != GAT_BF16)
        return fail(GAT_ERR_UNSUPPORTED, "gat_softmax_aggregate: unknown dtype %d", (int)dtype);
    if (n_rows == 0) return GAT_OK;
    if (!row_ptr || !out || (n_edges > 0 && (!col_idx || !scores || !feat)))
        return fail(GAT_ERR_INVALID_ARG, "gat_softmax_aggregate: NULL pointer");
    if (plan && (plan->n_rows != n_rows || plan->n_edges != n_edges))
        return fail(GAT_ERR_PLAN_MISMATCH,
                    "gat_softmax_aggregate: plan is for n_rows=%lld n_edges=%lld",
                    (long long)plan->n_rows, (long long)plan->n_edges);
    const int eb = dtype == GAT_F32 ? 4 : 2;
    const bool vec_ok = aligned16(out) && (n_edges == 0 || aligned16(feat));
    const int Hg = vec_ok ? engine_group(H, Dh, eb) : 0;
    if (Hg == 0)
        return fail(GAT_ERR_UNSUPPORTED,
                    "gat_softmax_aggregate: needs 16-byte aligned rows and a vector-engine shape "
                    "(H=%d, Dh=%d); use gat_edge_softmax + gat_spmm_weighted", (int)H, (int)Dh);
    EngineParams p{};
    p.row_ptr = row_ptr;
    p.col_idx = col_idx;
    p.v = feat;
    p.w = scores;
    p.w_stride = H;
    p.out = out;
    p.n_rows = n_rows;
    p.H = Hg;
    p.Dh = Dh;
    p.row_elems = (int64_t)H * Dh;
    p.qscale = kLog2e;
    p.heavy_threshold = INT_MAX;
    p.chunk_edges = 1;
    p.slot_floats = slot_floats(H, Dh);
    if (plan) {
        p.heavy_threshold = plan->heavy_threshold;
        p.chunk_edges = plan->chunk_edges;
        p.n_chunks = plan->n_chunks;
        p.heavy_rows = plan->heavy_rows;
        p.chunk_start = plan->chunk_start;
        p.chunk_row = plan->chunk_row;
        p.chunk_desc = plan->chunk_desc;
        p.counters = plan->counters;
        if (p.n_chunks > 0) {
            const size_t need = (size_t)p.n_chunks * (size_t)p.slot_floats * sizeof(float);
            if (!workspace || workspace_bytes < need || !aligned16(workspace))
                return fail(GAT_ERR_WORKSPACE,
                            "gat_softmax_aggregate: workspace needs %zu bytes (16-byte aligned), "
                            "got %zu", need, workspace_bytes);
            p.partials = static_cast<float *>(workspace);
        }
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // one launch per group of Hg heads (a slice of every feature / out row and
    // the group's columns of the scores)
    for (int h0 = 0; h0 < H; h0 += Hg) {
        EngineParams pg = p;
        const size_t off = (size_t)h0 * Dh * eb;
        pg.out = static_cast<char *>(out) + off;
        if (n_edges > 0) {
            pg.v = static_cast<const char *>(feat) + off;
            pg.w = scores + h0;
        }
        const gat_status_t st = dtype == GAT_F32 ? launch_given<float>(pg, s)
                                                 : launch_given<__nv_bfloat16>(pg, s);
        if (st != GAT_OK) return st;
    }
    return GAT_OK;
}
