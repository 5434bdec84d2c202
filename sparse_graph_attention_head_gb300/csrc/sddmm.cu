// sddmm.cu - gathered per-edge dot products (FW-GLM-5-1 l1_p10, reference
// model: gather the two endpoint feature rows of every edge, multiply
// elementwise, sum over the feature dimension), with heads and a scale.
//
// Work unit: one (edge, head) pair, handled by a group of G lanes; each lane
// loads 16-byte vectors of both rows (coalesced across the group, the
// warp-per-edge idea of the page's drafts narrowed to the head width) and the
// group finishes with a xor-shuffle sum. Consecutive pairs of a warp are
// consecutive heads of the same edge, so a warp reads whole feature rows.
// CSR form, row layouts the vector engine covers (sddmm_rows_kernel): each
// warp takes an equal contiguous span of edges (balanced whatever the degree
// distribution), finds the row of its first edge by one binary search on
// row_ptr and walks the rows of its span; the destination row's features stay
// in registers, spread over the lanes in 16-byte vectors as in the fused
// layer, while U source rows per warp are in flight; a head is G adjacent
// lanes (G-lane xor-shuffle sum) and one store per edge writes all its heads.
// Other CSR layouts find each edge's row by binary search (sddmm_kernel).
#include "row_engine.cuh"

namespace gat {

constexpr int kSddmmThreads = 256;

__device__ __forceinline__ int64_t row_of_edge(const int32_t *__restrict__ row_ptr, int64_t n_rows,
                                               int64_t e) {
    // largest r with row_ptr[r] <= e (rows of degree 0 are skipped over)
    int64_t lo = 0, hi = n_rows;  // invariant: row_ptr[lo] <= e < row_ptr[hi]
    while (hi - lo > 1) {
        const int64_t mid = (lo + hi) >> 1;
        if (__ldg(row_ptr + mid) <= e)
            lo = mid;
        else
            hi = mid;
    }
    return lo;
}

// VEC elements per load (16 bytes, or 1 for the scalar path); G lanes per pair
template <typename T, int VEC>
__global__ void __launch_bounds__(kSddmmThreads)
sddmm_kernel(const int32_t *__restrict__ row_ptr, const int32_t *__restrict__ src_idx,
             const int32_t *__restrict__ dst_idx, int64_t n_rows, int64_t n_edges,
             const T *__restrict__ a, const T *__restrict__ b, int32_t H, int32_t Dh, float scale,
             float *__restrict__ out, int G) {
    const int lane = threadIdx.x & 31;
    const int per_warp = 32 / G;
    const int grp = lane / G, gl = lane % G;
    const int64_t n_pairs = n_edges * H;
    const int64_t wpb = blockDim.x >> 5;
    const int64_t warp0 = (int64_t)blockIdx.x * wpb + (threadIdx.x >> 5);
    const int64_t n_warps = (int64_t)gridDim.x * wpb;
    const int nv = Dh / VEC;  // vectors per head row
    for (int64_t pb = warp0 * per_warp; pb < n_pairs; pb += n_warps * per_warp) {
        const int64_t pr = pb + grp;
        const bool valid = pr < n_pairs;
        float acc = 0.f;
        if (valid) {
            const int64_t e = pr / H;
            const int h = (int)(pr - e * H);
            const int64_t s = __ldg(src_idx + e);
            const int64_t d = row_ptr ? row_of_edge(row_ptr, n_rows, e) : (int64_t)__ldg(dst_idx + e);
            const T *ra = a + (s * H + h) * (int64_t)Dh;
            const T *rb = b + (d * H + h) * (int64_t)Dh;
            for (int t = gl; t < nv; t += G) {
                if constexpr (VEC > 1) {
                    float fa[VEC], fb[VEC];
                    Vec<T>::unpack(ld_stream16(ra + t * VEC), fa);
                    Vec<T>::unpack(ld_stream16(rb + t * VEC), fb);
#pragma unroll
                    for (int i = 0; i < VEC; ++i) acc = fmaf(fa[i], fb[i], acc);
                } else {
                    acc = fmaf(load_elem(ra, t), load_elem(rb, t), acc);
                }
            }
        }
        for (int o = 1; o < G; o <<= 1) acc += __shfl_xor_sync(kFull, acc, o);
        if (valid && gl == 0) out[pr] = scale * acc;
    }
}

// CSR SDDMM over equal edge spans per warp. V 16-byte vectors per lane (the
// row is V * 32 vectors), G = Dh / VE lanes per head (G >= V), U edges in
// flight per warp, MINB resident blocks per SM (the register budget).
constexpr int kSddmmRowsThreads = 256;

template <typename T, int V, int U, int MINB>
__global__ void __launch_bounds__(kSddmmRowsThreads, MINB)
sddmm_rows_kernel(const int32_t *__restrict__ row_ptr, const int32_t *__restrict__ col_idx,
                  int64_t n_rows, int64_t n_edges, const T *__restrict__ a,
                  const T *__restrict__ b, int32_t H, int32_t Dh, float scale,
                  float *__restrict__ out) {
    constexpr int VE = Vec<T>::N;
    const int lane = threadIdx.x & 31;
    const int64_t n_warps = (int64_t)gridDim.x * (kSddmmRowsThreads / 32);
    const int64_t w = (int64_t)blockIdx.x * (kSddmmRowsThreads / 32) + (threadIdx.x >> 5);
    const int64_t e_begin = n_edges * w / n_warps, e_end = n_edges * (w + 1) / n_warps;
    if (e_begin >= e_end) return;
    const int G = Dh / VE;                          // lanes per head
    const int64_t row_bytes = (int64_t)H * Dh * sizeof(T);
    // the lane that stores head (s * 32 + lane) / G of this edge: lane % G == s
    const int my_slot = lane % G;
    const int my_head = my_slot < V ? (my_slot * 32 + lane) / G : 0;
    const char *ab = reinterpret_cast<const char *>(a);
    const char *bb = reinterpret_cast<const char *>(b);
    int64_t r = row_of_edge(row_ptr, n_rows, e_begin);
    int64_t e = e_begin;
    while (e < e_end) {
        int64_t rend = __ldg(row_ptr + r + 1);
        while (rend <= e) {  // rows of degree 0
            ++r;
            rend = __ldg(row_ptr + r + 1);
        }
        // the row's b vectors: as stored for bf16 (the dot on the packed pairs,
        // scaled after the head's sum), else unpacked and scaled
        constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
        float qf[V][VE];
        uint4 qpk[V];
#pragma unroll
        for (int s = 0; s < V; ++s) {
            const uint4 u = ld_stream16(bb + r * row_bytes + (s * 32 + lane) * 16);
            if (kBf16) {
                qpk[s] = u;
            } else {
                Vec<T>::unpack(u, qf[s]);
#pragma unroll
                for (int t = 0; t < VE; ++t) qf[s][t] *= scale;
            }
        }
        const int64_t seg_end = rend < e_end ? rend : e_end;
        for (int64_t base = e; base < seg_end; base += 32) {
            const int n = (int)(seg_end - base < 32 ? seg_end - base : 32);
            const int my_ci = lane < n ? __ldg(col_idx + base + lane) : 0;
            for (int j0 = 0; j0 < n; j0 += U) {
                uint4 kr[U][V];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int64_t src = __shfl_sync(kFull, my_ci, (j0 + u) & 31);
                    if (j0 + u < n) {
#pragma unroll
                        for (int s = 0; s < V; ++s)
                            kr[u][s] = ld_stream16(ab + src * row_bytes + (s * 32 + lane) * 16);
                    }
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    float part[V];
#pragma unroll
                    for (int s = 0; s < V; ++s) {
                        if constexpr (kBf16) {
                            part[s] = dot_bf16x8(qpk[s], kr[u][s]);
                        } else {
                            float kf[VE];
                            Vec<T>::unpack(kr[u][s], kf);
                            float acc = 0.f;
#pragma unroll
                            for (int t = 0; t < VE; ++t) acc = fmaf(qf[s][t], kf[t], acc);
                            part[s] = acc;
                        }
                    }
                    for (int o = 1; o < G; o <<= 1) {
#pragma unroll
                        for (int s = 0; s < V; ++s) part[s] += __shfl_xor_sync(kFull, part[s], o);
                    }
                    if (kBf16)
#pragma unroll
                        for (int s = 0; s < V; ++s) part[s] *= scale;
                    if (j0 + u < n && my_slot < V) {
                        float val = part[0];
#pragma unroll
                        for (int s = 1; s < V; ++s) val = my_slot == s ? part[s] : val;
                        out[(base + j0 + u) * H + my_head] = val;
                    }
                }
            }
        }
        e = seg_end;
    }
}

template <typename T, int V>
static gat_status_t launch_sddmm_rows(const int32_t *row_ptr, const int32_t *ci, int64_t n_rows,
                                      int64_t E, const void *a, const void *b, int32_t H,
                                      int32_t Dh, float scale, float *out, cudaStream_t s) {
    // 2 KB of source rows in flight per warp at 5 blocks of 8 warps per SM:
    // a sweep on the 1e6-row workload (H=8, Dh=64, bf16) over 1-8 edges in
    // flight x 1-8 blocks per SM put this at 2.84 ms, the rest at 2.9-4.5 ms
    constexpr int U = V == 1 ? 4 : (V == 2 ? 2 : 1);
    auto kern = sddmm_rows_kernel<T, V, U, 5>;
    static std::atomic<int64_t> caps[kMaxDevices];
    int64_t blocks = device_blocks(caps, kern, kSddmmRowsThreads, 0);
    // at least ~32 edges per warp
    const int64_t want = (E + 32 * (kSddmmRowsThreads / 32) - 1) / (32 * (kSddmmRowsThreads / 32));
    if (blocks > want) blocks = want < 1 ? 1 : want;
    kern<<<(unsigned)blocks, kSddmmRowsThreads, 0, s>>>(row_ptr, ci, n_rows, E,
                                                       static_cast<const T *>(a),
                                                       static_cast<const T *>(b), H, Dh, scale, out);
    return check_launch("gat_sddmm (CSR rows)");
}

template <typename T>
static gat_status_t launch_sddmm(const int32_t *row_ptr, const int32_t *si, const int32_t *di,
                                 int64_t n_rows, int64_t E, const void *a, const void *b,
                                 int32_t H, int32_t Dh, float scale, float *out, cudaStream_t s) {
    constexpr int VE = Vec<T>::N;
    const bool vec = (Dh % VE == 0) && aligned16(a) && aligned16(b);
    int V = 0, LE = 0;
    if (row_ptr && vec && engine_shape(H, Dh, sizeof(T), V, LE) && LE == 32 && Dh / VE >= V) {
        if (V == 1) return launch_sddmm_rows<T, 1>(row_ptr, si, n_rows, E, a, b, H, Dh, scale, out, s);
        if (V == 2) return launch_sddmm_rows<T, 2>(row_ptr, si, n_rows, E, a, b, H, Dh, scale, out, s);
        if (V == 4) return launch_sddmm_rows<T, 4>(row_ptr, si, n_rows, E, a, b, H, Dh, scale, out, s);
    }
    const int nv = vec ? Dh / VE : Dh;
    int G = 1;
    while (G < 32 && G * 2 <= nv) G *= 2;
    const int64_t pairs = E * H;
    const int64_t per_block = (int64_t)(kSddmmThreads / 32) * (32 / G);
    int64_t blocks = (pairs + per_block - 1) / per_block;
    const int64_t cap = (int64_t)sm_count() * 16;
    if (blocks > cap) blocks = cap;
    if (vec)
        sddmm_kernel<T, VE><<<(unsigned)blocks, kSddmmThreads, 0, s>>>(
            row_ptr, si, di, n_rows, E, static_cast<const T *>(a), static_cast<const T *>(b), H,
            Dh, scale, out, G);
    else
        sddmm_kernel<T, 1><<<(unsigned)blocks, kSddmmThreads, 0, s>>>(
            row_ptr, si, di, n_rows, E, static_cast<const T *>(a), static_cast<const T *>(b), H,
            Dh, scale, out, G);
    return check_launch("gat_sddmm");
}

}  // namespace gat

using namespace gat;

extern "C" gat_status_t gat_sddmm(const int32_t *row_ptr, const int32_t *src_idx,
                                  const int32_t *dst_idx, int64_t n_rows, int64_t n_edges,
                                  const void *src_feat, int64_t n_src, const void *dst_feat,
                                  int64_t n_dst, int32_t H, int32_t Dh, float scale,
                                  gat_dtype_t dtype, float *out, void *stream) {
    if (n_edges < 0 || n_src < 0 || n_dst < 0 || H < 1 || Dh < 1 || (row_ptr && n_rows < 0))
        return fail(GAT_ERR_INVALID_ARG, "gat_sddmm: bad sizes");
    if (dtype != GAT_F32 && dtype != GAT_BF16)
        return fail(GAT_ERR_UNSUPPORTED, "gat_sddmm: unknown dtype %d", (int)dtype);
    if (n_edges == 0) return GAT_OK;
    if (!src_idx || !src_feat || !dst_feat || !out || (!row_ptr && !dst_idx))
        return fail(GAT_ERR_INVALID_ARG, "gat_sddmm: NULL pointer");
    if (row_ptr && (n_rows < 1 || n_dst < n_rows))
        return fail(GAT_ERR_INVALID_ARG, "gat_sddmm: CSR form needs 1 <= n_rows <= n_dst");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (dtype == GAT_F32)
        return launch_sddmm<float>(row_ptr, src_idx, dst_idx, n_rows, n_edges, src_feat, dst_feat,
                                   H, Dh, scale, out, s);
    return launch_sddmm<__nv_bfloat16>(row_ptr, src_idx, dst_idx, n_rows, n_edges, src_feat,
                                       dst_feat, H, Dh, scale, out, s);
}
