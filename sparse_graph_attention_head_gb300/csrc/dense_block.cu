// dense_block.cu - gat_dense_masked_attention: the scene-graph relation
// attention block of Kimi-K2.6 l2_p4 (reference model: LayerNorm -> Q/K/V
// Linear without bias -> Q K^T / sqrt(head_dim) + relation-MLP bias ->
// mask (< 0.5 -> -inf) -> softmax -> A V -> out_proj -> residual), fp32.
//
// One thread block per graph; everything for the graph stays in shared
// memory (node rows padded to D+1 floats so column walks are bank-conflict
// free). Phases: LayerNorm (warp per node, two-pass mean / biased variance),
// the three projections, the relation MLP per node pair (all heads at once),
// masked softmax attention (warp per (head, query) with lane = key, as the
// page's attention kernel maps it), then out_proj + residual straight to
// global memory.
#include "common.cuh"

namespace gat {

constexpr int kDenseThreads = 256;
constexpr int kDenseMaxH = 8;

struct DenseParams {
    int32_t B, N, D, H, P;
    const float *nodes, *pair, *mask, *ln_w, *ln_b;
    float ln_eps;
    const float *Wq, *Wk, *Wv, *W1, *b1, *W2, *b2, *Wout;
    float *out;
};

__global__ void __launch_bounds__(kDenseThreads)
dense_block_kernel(const DenseParams p) {
    extern __shared__ float sm[];
    const int N = p.N, D = p.D, H = p.H, P = p.P, dh = D / H, DS = D + 1;
    float *xs = sm;               // [N][DS] input rows
    float *xn = xs + N * DS;      // [N][DS] normalised rows
    float *qs = xn + N * DS;      // [N][DS]
    float *ks = qs + N * DS;      // [N][DS]
    float *vs = ks + N * DS;      // [N][DS]
    float *cs = vs + N * DS;      // [N][DS] attention context
    float *rb = cs + N * DS;      // [H][N][N] relation bias
    float *w1 = rb + H * N * N;   // [P][P]
    float *bb1 = w1 + P * P;      // [P]
    float *w2 = bb1 + P;          // [H][P]
    float *bb2 = w2 + H * P;      // [H]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
    const float inv_sqrt_dh = 1.0f / sqrtf((float)dh);

    for (int i = tid; i < P * P; i += blockDim.x) w1[i] = p.W1[i];
    for (int i = tid; i < P; i += blockDim.x) bb1[i] = p.b1[i];
    for (int i = tid; i < H * P; i += blockDim.x) w2[i] = p.W2[i];
    for (int i = tid; i < H; i += blockDim.x) bb2[i] = p.b2[i];

    for (int64_t b = blockIdx.x; b < p.B; b += gridDim.x) {
        const float *x = p.nodes + b * (int64_t)N * D;
        for (int i = tid; i < N * D; i += blockDim.x) xs[(i / D) * DS + i % D] = __ldg(x + i);
        __syncthreads();
        // LayerNorm: warp per node
        for (int n = warp; n < N; n += nw) {
            float s = 0.f;
            for (int d = lane; d < D; d += 32) s += xs[n * DS + d];
            const float mean = warp_sum(s) / (float)D;
            float v2 = 0.f;
            for (int d = lane; d < D; d += 32) {
                const float t = xs[n * DS + d] - mean;
                v2 = fmaf(t, t, v2);
            }
            const float rstd = 1.0f / sqrtf(warp_sum(v2) / (float)D + p.ln_eps);
            for (int d = lane; d < D; d += 32)
                xn[n * DS + d] = (xs[n * DS + d] - mean) * rstd * __ldg(p.ln_w + d) + __ldg(p.ln_b + d);
        }
        __syncthreads();
        // Q, K, V = xn W^T
        for (int i = tid; i < N * 3 * D; i += blockDim.x) {
            const int n = i / (3 * D), oo = i % (3 * D), which = oo / D, o = oo % D;
            const float *W = which == 0 ? p.Wq : (which == 1 ? p.Wk : p.Wv);
            const float4 *wr = reinterpret_cast<const float4 *>(W + (int64_t)o * D);
            const float *xr = xn + n * DS;
            float a = 0.f;
            for (int c = 0; c < D / 4; ++c) {
                const float4 w4 = __ldg(wr + c);
                a = fmaf(w4.x, xr[4 * c], a);
                a = fmaf(w4.y, xr[4 * c + 1], a);
                a = fmaf(w4.z, xr[4 * c + 2], a);
                a = fmaf(w4.w, xr[4 * c + 3], a);
            }
            float *dst = which == 0 ? qs : (which == 1 ? ks : vs);
            dst[n * DS + o] = a;
        }
        // relation MLP bias for every pair (i, j), all heads
        for (int pr = tid; pr < N * N; pr += blockDim.x) {
            const float *pf = p.pair + (b * (int64_t)N * N + pr) * P;
            float r[kDenseMaxH];
#pragma unroll
            for (int h = 0; h < kDenseMaxH; ++h) r[h] = h < H ? bb2[h] : 0.f;
            for (int u = 0; u < P; ++u) {
                float a = bb1[u];
                for (int c = 0; c < P; ++c) a = fmaf(w1[u * P + c], __ldg(pf + c), a);
                const float hid = a / (1.0f + expf(-a));
#pragma unroll
                for (int h = 0; h < kDenseMaxH; ++h)
                    if (h < H) r[h] = fmaf(w2[h * P + u], hid, r[h]);
            }
#pragma unroll
            for (int h = 0; h < kDenseMaxH; ++h)
                if (h < H) rb[h * N * N + pr] = r[h];
        }
        __syncthreads();
        // masked softmax attention: warp per (head, query), lane = key
        const float *mk = p.mask + b * (int64_t)N * N;
        for (int hi = warp; hi < H * N; hi += nw) {
            const int h = hi / N, i = hi % N;
            float logit = -INFINITY;
            if (lane < N) {
                float a = 0.f;
                for (int c = 0; c < dh; ++c) a = fmaf(qs[i * DS + h * dh + c], ks[lane * DS + h * dh + c], a);
                logit = a * inv_sqrt_dh + rb[h * N * N + i * N + lane];
                if (__ldg(mk + i * N + lane) < 0.5f) logit = -INFINITY;
            }
            const float m = warp_max(logit);
            const float e = lane < N ? expf(logit - m) : 0.f;  // all-masked row: NaN, as the reference
            const float z = warp_sum(e);
            const float a = e / z;
            float ctx = 0.f;
            for (int j = 0; j < N; ++j) {
                const float aj = __shfl_sync(kFull, a, j);
                if (lane < dh) ctx = fmaf(aj, vs[j * DS + h * dh + lane], ctx);
            }
            if (lane < dh) cs[i * DS + h * dh + lane] = ctx;
        }
        __syncthreads();
        // out = x + ctx Wout^T
        float *ob = p.out + b * (int64_t)N * D;
        for (int i = tid; i < N * D; i += blockDim.x) {
            const int n = i / D, o = i % D;
            const float4 *wr = reinterpret_cast<const float4 *>(p.Wout + (int64_t)o * D);
            const float *cr = cs + n * DS;
            float a = 0.f;
            for (int c = 0; c < D / 4; ++c) {
                const float4 w4 = __ldg(wr + c);
                a = fmaf(w4.x, cr[4 * c], a);
                a = fmaf(w4.y, cr[4 * c + 1], a);
                a = fmaf(w4.z, cr[4 * c + 2], a);
                a = fmaf(w4.w, cr[4 * c + 3], a);
            }
            ob[i] = xs[n * DS + o] + a;
        }
        __syncthreads();
    }
}

// tensor-core path (dense_block_tc.cu); GAT_ERR_UNSUPPORTED outside its shapes
bool dense_block_tc_shape(int32_t N, int32_t D, int32_t H, int32_t P);
size_t dense_block_tc_workspace();
gat_status_t dense_block_tc(int32_t B, int32_t N, int32_t D, int32_t H, int32_t P,
                            const float *nodes, const float *pair, const float *mask,
                            const float *ln_w, const float *ln_b, float ln_eps, const float *Wq,
                            const float *Wk, const float *Wv, const float *W1, const float *b1,
                            const float *W2, const float *b2, const float *Wout, float *out,
                            void *workspace, size_t workspace_bytes, cudaStream_t s);
gat_status_t dense_block_tc_status(const void *workspace, cudaStream_t s);

}  // namespace gat

using namespace gat;

extern "C" gat_status_t gat_dense_masked_attention(
    int32_t B, int32_t N, int32_t D, int32_t H, int32_t P, const float *nodes,
    const float *pair_feats, const float *edge_mask, const float *ln_w, const float *ln_b,
    float ln_eps, const float *Wq, const float *Wk, const float *Wv, const float *W1,
    const float *b1, const float *W2, const float *b2, const float *Wout, float *out,
    void *workspace, size_t workspace_bytes, void *stream) {
    if (B < 0 || N < 1 || D < 1 || H < 1 || P < 1)
        return fail(GAT_ERR_INVALID_ARG, "gat_dense_masked_attention: bad sizes");
    if (N > 32 || D % H || D / H > 32 || D > 128 || D % 4 || P > 32 || H > kDenseMaxH)
        return fail(GAT_ERR_UNSUPPORTED,
                    "gat_dense_masked_attention: unsupported shape N=%d D=%d H=%d P=%d", N, D, H, P);
    if (B == 0) return GAT_OK;
    const void *ptrs[] = {nodes, pair_feats, edge_mask, ln_w, ln_b, Wq, Wk, Wv,
                          W1,    b1,         W2,        b2,   Wout, out};
    for (const void *q : ptrs)
        if (!q) return fail(GAT_ERR_INVALID_ARG, "gat_dense_masked_attention: NULL pointer");
    if (!aligned16(nodes) || !aligned16(Wq) || !aligned16(Wk) || !aligned16(Wv) ||
        !aligned16(Wout) || !aligned16(out))
        return fail(GAT_ERR_UNSUPPORTED, "gat_dense_masked_attention: pointers must be 16-byte aligned");
    // the module shape of the block page runs its projections on the tensor
    // cores (dense_block_tc.cu); every other shape runs the SIMT kernel below
    if (aligned16(pair_feats) && dense_block_tc_shape(N, D, H, P))
        return dense_block_tc(B, N, D, H, P, nodes, pair_feats, edge_mask, ln_w, ln_b, ln_eps, Wq,
                              Wk, Wv, W1, b1, W2, b2, Wout, out, workspace, workspace_bytes,
                              static_cast<cudaStream_t>(stream));
    DenseParams p{B, N, D, H, P, nodes, pair_feats, edge_mask, ln_w, ln_b, ln_eps,
                  Wq, Wk, Wv, W1, b1, W2, b2, Wout, out};
    const int DS = D + 1;
    const size_t smem = (size_t)(6 * N * DS + H * N * N + P * P + P + H * P + H) * sizeof(float);
    // the attribute is set once per device, to the device's opt-in maximum, so
    // every shape (and concurrent first calls with different shapes) fits it
    static std::atomic<int> smem_set[kMaxDevices];
    int optin = 0;
    cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, current_device());
    if (smem > (size_t)optin)
        return fail(GAT_ERR_UNSUPPORTED, "gat_dense_masked_attention: %zu bytes of shared memory "
                    "needed, %d available", smem, optin);
    cudaError_t e = allow_dynamic_smem(smem_set, dense_block_kernel, optin);
    if (e != cudaSuccess) return cuda_fail(e, "gat_dense_masked_attention: smem attribute");
    int per_sm = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, dense_block_kernel, kDenseThreads, smem);
    if (per_sm < 1) per_sm = 1;
    int64_t blocks = (int64_t)sm_count() * per_sm;
    if (blocks > B) blocks = B;
    dense_block_kernel<<<(unsigned)blocks, kDenseThreads, smem, static_cast<cudaStream_t>(stream)>>>(p);
    return check_launch("gat_dense_masked_attention");
}

extern "C" gat_status_t gat_dense_masked_attention_workspace_size(int32_t N, int32_t D, int32_t H,
                                                                  int32_t P, size_t *bytes) {
    if (!bytes || N < 1 || D < 1 || H < 1 || P < 1)
        return fail(GAT_ERR_INVALID_ARG, "gat_dense_masked_attention_workspace_size: bad arguments");
    *bytes = dense_block_tc_shape(N, D, H, P) ? dense_block_tc_workspace() : 0;
    return GAT_OK;
}

extern "C" gat_status_t gat_dense_masked_attention_status(const void *workspace, void *stream) {
    if (!workspace)
        return fail(GAT_ERR_INVALID_ARG, "gat_dense_masked_attention_status: workspace is NULL");
    return dense_block_tc_status(workspace, static_cast<cudaStream_t>(stream));
}
