// edge_softmax.cu - segmented, numerically stable softmax over each CSR
// row's edge range, independently per head (FW-GLM-5-1 l1_p6, reference
// model: softmax of every node's edge scores, max-subtracted).
//
// scores/out are [E, H] with heads contiguous, so a row's scores form one
// contiguous run of deg*H floats. Light rows: one warp per row; when H
// divides 32 lane l only ever sees head l % H, so each lane keeps one
// (max, sum) pair and the per-head reduction is a xor-shuffle over the lanes
// sharing that head. Heavy rows (with a plan): one block per row.
// Three passes over the row (max, sum of exp, write); the first K elements of
// each lane stay in registers, the rest are re-read (L1/L2 resident).
#include <climits>

#include "common.cuh"

namespace gat {

constexpr int kSoftmaxThreads = 256;
constexpr int kSoftmaxCache = 4;  // cached elements per lane

// H divides 32: lane-per-head-residue path
__global__ void __launch_bounds__(kSoftmaxThreads)
softmax_rows_hdiv_kernel(const int32_t *__restrict__ row_ptr, int64_t n_rows, int32_t H,
                         const float *scores, float *out, int32_t heavy_threshold) {
    const int lane = threadIdx.x & 31;
    const int64_t wpb = blockDim.x >> 5;
    const int64_t n_warps = (int64_t)gridDim.x * wpb;
    for (int64_t row = (int64_t)blockIdx.x * wpb + (threadIdx.x >> 5); row < n_rows;
         row += n_warps) {
        const int64_t e0 = row_ptr[row], e1 = row_ptr[row + 1];
        if (e1 - e0 > heavy_threshold || e1 == e0) continue;
        const int64_t x0 = e0 * H, x1 = e1 * H;
        float c[kSoftmaxCache];
        float m = -INFINITY;
#pragma unroll
        for (int k = 0; k < kSoftmaxCache; ++k) {
            const int64_t x = x0 + lane + 32 * k;
            c[k] = x < x1 ? scores[x] : -INFINITY;
            m = fmaxf(m, c[k]);
        }
        for (int64_t x = x0 + lane + 32 * kSoftmaxCache; x < x1; x += 32) m = fmaxf(m, scores[x]);
        for (int o = 16; o >= H; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
        float z = 0.f;
#pragma unroll
        for (int k = 0; k < kSoftmaxCache; ++k)
            if (x0 + lane + 32 * k < x1) z += expf(c[k] - m);
        for (int64_t x = x0 + lane + 32 * kSoftmaxCache; x < x1; x += 32) z += expf(scores[x] - m);
        for (int o = 16; o >= H; o >>= 1) z += __shfl_xor_sync(kFull, z, o);
#pragma unroll
        for (int k = 0; k < kSoftmaxCache; ++k) {
            const int64_t x = x0 + lane + 32 * k;
            if (x < x1) out[x] = expf(c[k] - m) / z;
        }
        for (int64_t x = x0 + lane + 32 * kSoftmaxCache; x < x1; x += 32)
            out[x] = expf(scores[x] - m) / z;
    }
}

// any H: lanes over edges, one head at a time
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

// heavy rows: one block per row, heads one at a time, block reductions
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
    int64_t blocks = (n_rows + wpb - 1) / wpb;
    const int64_t cap = (int64_t)sm_count() * 8;
    if (blocks > cap) blocks = cap;
    if (32 % H == 0)
        softmax_rows_hdiv_kernel<<<(unsigned)blocks, kSoftmaxThreads, 0, s>>>(row_ptr, n_rows, H,
                                                                              scores, out, T);
    else
        softmax_rows_generic_kernel<<<(unsigned)blocks, kSoftmaxThreads, 0, s>>>(
            row_ptr, n_rows, H, scores, out, T);
    gat_status_t st = check_launch("gat_edge_softmax: rows");
    if (st != GAT_OK) return st;
    if (plan && plan->n_heavy > 0) {
        int64_t hb = plan->n_heavy;
        if (hb > cap) hb = cap;
        softmax_heavy_kernel<<<(unsigned)hb, kSoftmaxThreads, 0, s>>>(
            row_ptr, plan->heavy_rows, plan->n_heavy, H, scores, out);
        st = check_launch("gat_edge_softmax: heavy rows");
    }
    return st;
}
