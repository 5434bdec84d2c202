// spmm.cu - gat_spmm_weighted: out[i,h,:] = sum_e w[e,h] * feat[col_idx[e],h,:]
// (FW-GLM-5-1 l1_p18, reference model; Kimi-K2.6 l2_p37: a destination with
// no edges stays zero). Light rows: one warp per row (row_engine.cuh);
// heavy rows (with a plan): one block per row, warps summed in warp order.
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

template <typename T, int V, int LE>
static gat_status_t launch_spmm_fast(const EngineParams &p, cudaStream_t s) {
    constexpr int U = 8 / V;
    auto kern = spmm_engine_kernel<T, V, LE, U>;
    static int64_t cap = 0;
    if (cap == 0) cap = persistent_blocks(kern, INT64_MAX);
    const int64_t wpb = kEngineThreads / 32;
    int64_t blocks = (p.n_rows + wpb - 1) / wpb;
    if (blocks > cap) blocks = cap;
    kern<<<(unsigned)blocks, kEngineThreads, 0, s>>>(p);
    gat_status_t st = check_launch("gat_spmm_weighted");
    if (st != GAT_OK || p.n_block_rows == 0) return st;
    auto hk = spmm_heavy_kernel<T, V, LE, U>;
    static int64_t hcap = 0;
    if (hcap == 0) hcap = persistent_blocks(hk, INT64_MAX);
    int64_t hb = p.n_block_rows < hcap ? p.n_block_rows : hcap;
    hk<<<(unsigned)hb, kEngineThreads, 0, s>>>(p);
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
    static int64_t cap = 0;
    if (cap == 0) cap = persistent_blocks(spmm_generic_kernel<T>, INT64_MAX);
    const int64_t wpb = kEngineThreads / 32;
    int64_t blocks = (p.n_rows + wpb - 1) / wpb;
    if (blocks > cap) blocks = cap;
    spmm_generic_kernel<T><<<(unsigned)blocks, kEngineThreads, 0, s>>>(p);
    return check_launch("gat_spmm_weighted (scalar)");
}

}  // namespace gat

using namespace gat;

extern "C" gat_status_t gat_spmm_weighted(const int32_t *row_ptr, const int32_t *col_idx,
                                          int64_t n_rows, int64_t n_src, int64_t n_edges,
                                          int32_t H, int32_t Dh, const float *w, const void *feat,
                                          gat_dtype_t dtype, void *out, gat_plan_t plan,
                                          void *stream) {
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
    p.heavy_threshold = INT_MAX;
    const bool vec_ok = aligned16(out) && (n_edges == 0 || aligned16(feat));
    int V, LE;
    const int eb = dtype == GAT_F32 ? 4 : 2;
    if (plan && vec_ok && engine_shape(H, Dh, eb, V, LE) && plan->n_heavy > 0) {
        p.heavy_threshold = plan->heavy_threshold;
        p.heavy_rows = plan->heavy_rows;
        p.n_block_rows = plan->n_heavy;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (dtype == GAT_F32) return launch_spmm<float>(p, vec_ok, s);
    return launch_spmm<__nv_bfloat16>(p, vec_ok, s);
}
