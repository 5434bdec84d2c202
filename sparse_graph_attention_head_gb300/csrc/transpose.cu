// transpose.cu - the transposed (source-major) view of a CSR graph, used by
// the backward pass. In the backward, every edge's gradients land on the
// feature rows of its source node, and a source read by several edges
// collects several contributions (FW-GLM-5-1 l1_p10, discussion of the
// backward pass, which adds them with atomics). Here each source's edges are
// listed together, in increasing edge order, so a source's gradient is a
// plain sum in a fixed order: no floating-point atomics, bitwise repeatable.
//
// Build (once per graph, on the device):
//   count edges per source (integer atomics) -> exclusive scan = src_ptr
//   scatter edge ids into their source's group (integer atomics: any order)
//   order every group by edge id: a warp sorts each run of 32 (bitonic, in
//     registers), then log2(max group size / 32) rank-merge passes, in which
//     each element finds its place in the merged pair of runs by a binary
//     search in the partner run (edge ids are distinct, so every place is
//     unique)
//   dst[k] = the row owning edge perm[k]
//   a degree plan over src_ptr for sources with many edges.
#include <climits>

#include "common.cuh"

namespace gat {

constexpr int kTrThreads = 256;
constexpr int kScanItems = 8;  // per thread
constexpr int64_t kScanTile = (int64_t)kTrThreads * kScanItems;

static unsigned grid_for(int64_t n, int threads) {
    int64_t b = (n + threads - 1) / threads;
    const int64_t cap = (int64_t)sm_count() * 16;
    if (b > cap) b = cap;
    return (unsigned)(b < 1 ? 1 : b);
}

__global__ void __launch_bounds__(kTrThreads)
tr_count_kernel(const int32_t *__restrict__ col_idx, int64_t E, int64_t n_src,
                int32_t *__restrict__ cnt, int32_t *__restrict__ bad) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < E; e += stride) {
        const int32_t c = col_idx[e];
        if (c < 0 || c >= n_src) {
            *bad = 1;
            continue;
        }
        atomicAdd(cnt + c, 1);
    }
}

// exclusive scan, pass 1: each block scans one tile and records its total
__global__ void __launch_bounds__(kTrThreads)
tr_scan_tiles_kernel(const int32_t *__restrict__ in, int64_t n, int32_t *__restrict__ out,
                     int64_t *__restrict__ tile_sums) {
    __shared__ int64_t wsum[kTrThreads / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t base = (int64_t)blockIdx.x * kScanTile + (int64_t)threadIdx.x * kScanItems;
    int64_t v[kScanItems], t = 0;
#pragma unroll
    for (int k = 0; k < kScanItems; ++k) {
        v[k] = base + k < n ? in[base + k] : 0;
        t += v[k];
    }
    int64_t inc = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int64_t x = __shfl_up_sync(kFull, inc, o);
        if (lane >= o) inc += x;
    }
    if (lane == 31) wsum[warp] = inc;
    __syncthreads();
    int64_t before = 0;
    for (int w = 0; w < warp; ++w) before += wsum[w];
    int64_t run = before + inc - t;
#pragma unroll
    for (int k = 0; k < kScanItems; ++k) {
        if (base + k < n) out[base + k] = (int32_t)run;
        run += v[k];
    }
    if (threadIdx.x == kTrThreads - 1) tile_sums[blockIdx.x] = before + inc;
}

// pass 2: exclusive scan of the tile totals (one block, tiles in sequence)
__global__ void __launch_bounds__(1024)
tr_scan_sums_kernel(int64_t *__restrict__ sums, int64_t nb) {
    __shared__ int64_t wsum[32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int64_t carry = 0;
    for (int64_t t0 = 0; t0 < nb; t0 += blockDim.x) {
        const int64_t i = t0 + threadIdx.x;
        const int64_t v = i < nb ? sums[i] : 0;
        int64_t inc = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int64_t x = __shfl_up_sync(kFull, inc, o);
            if (lane >= o) inc += x;
        }
        if (lane == 31) wsum[warp] = inc;
        __syncthreads();
        int64_t before = 0;
        for (int w = 0; w < warp; ++w) before += wsum[w];
        int64_t total = 0;
        for (int w = 0; w < nw; ++w) total += wsum[w];
        if (i < nb) sums[i] = carry + before + inc - v;
        carry += total;
        __syncthreads();
    }
}

// pass 3: add each tile's offset
__global__ void __launch_bounds__(kTrThreads)
tr_scan_add_kernel(int32_t *__restrict__ out, int64_t n, const int64_t *__restrict__ sums) {
    const int64_t base = (int64_t)blockIdx.x * kScanTile;
    const int64_t add = sums[blockIdx.x];
    for (int k = threadIdx.x; k < kScanTile; k += kTrThreads)
        if (base + k < n) out[base + k] = (int32_t)(out[base + k] + add);
}

// row_of[e] = the row owning edge e (one warp per row)
__global__ void __launch_bounds__(kTrThreads)
tr_row_of_kernel(const int32_t *__restrict__ row_ptr, int64_t n_rows, int32_t *__restrict__ row_of) {
    const int lane = threadIdx.x & 31;
    const int64_t n_warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < n_rows;
         r += n_warps) {
        const int32_t e1 = row_ptr[r + 1];
        for (int32_t e = row_ptr[r] + lane; e < e1; e += 32) row_of[e] = (int32_t)r;
    }
}

__global__ void __launch_bounds__(kTrThreads)
tr_fill_kernel(const int32_t *__restrict__ col_idx, int64_t E, int32_t *__restrict__ cursor,
               int32_t *__restrict__ perm) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < E; e += stride)
        perm[atomicAdd(cursor + col_idx[e], 1)] = (int32_t)e;
}

// seg[k] = the source owning position k
__global__ void __launch_bounds__(kTrThreads)
tr_seg_kernel(const int32_t *__restrict__ src_ptr, int64_t n_src, int32_t *__restrict__ seg) {
    const int lane = threadIdx.x & 31;
    const int64_t n_warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t j = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); j < n_src;
         j += n_warps) {
        const int32_t k0 = src_ptr[j], k1 = src_ptr[j + 1];
        for (int32_t k = k0 + lane; k < k1; k += 32) seg[k] = (int32_t)j;
    }
}

// largest count into *max_deg
__global__ void __launch_bounds__(kTrThreads)
tr_max_kernel(const int32_t *__restrict__ cnt, int64_t n, int32_t *__restrict__ max_deg) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    int32_t m = 0;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
        m = max(m, cnt[i]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(kFull, m, o));
    if ((threadIdx.x & 31) == 0 && m > 0) atomicMax(max_deg, m);
}

// Every run of 32 positions of a group (from the group's start) sorted
// ascending, one warp per group: a bitonic network over the lanes (lanes past
// the group's end hold INT_MAX, above every edge id).
__global__ void __launch_bounds__(kTrThreads)
tr_sort32_kernel(int32_t *__restrict__ perm, const int32_t *__restrict__ src_ptr, int64_t n_src) {
    const int lane = threadIdx.x & 31;
    const int64_t n_warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t j = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); j < n_src;
         j += n_warps) {
        const int32_t k0 = src_ptr[j], k1 = src_ptr[j + 1];
        if (k1 - k0 < 2) continue;
        for (int32_t r0 = k0; r0 < k1; r0 += 32) {
            const int32_t k = r0 + lane;
            int32_t v = k < k1 ? perm[k] : INT_MAX;
#pragma unroll
            for (int w = 2; w <= 32; w <<= 1)
#pragma unroll
                for (int o = w >> 1; o > 0; o >>= 1) {
                    const int32_t x = __shfl_xor_sync(kFull, v, o);
                    // ascending within blocks of w lanes with (lane & w) == 0, descending
                    // in the others; the lower lane of a pair keeps the block's order
                    const bool up = (lane & w) == 0, lower = (lane & o) == 0;
                    v = (lower == up) ? min(v, x) : max(v, x);
                }
            if (k < k1) perm[k] = v;
        }
    }
}

// One merge pass: runs of length L inside every group are merged pairwise.
__global__ void __launch_bounds__(kTrThreads)
tr_merge_kernel(const int32_t *__restrict__ in, int32_t *__restrict__ out,
                const int32_t *__restrict__ seg, const int32_t *__restrict__ src_ptr, int64_t E,
                int64_t L) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < E; k += stride) {
        const int32_t j = seg[k];
        const int64_t s0 = src_ptr[j], s1 = src_ptr[j + 1];
        const int64_t x = k - s0, r = x / L, o = x - r * L;
        const int64_t ps = s0 + (r >> 1) * 2 * L;  // first position of the pair
        int64_t lo, hi;                            // the partner run
        if (r & 1) {
            lo = ps;
            hi = ps + L;
        } else {
            lo = min(ps + L, s1);
            hi = min(ps + 2 * L, s1);
        }
        const int32_t v = in[k];
        int64_t a = lo, b = hi;  // partner elements below v
        while (a < b) {
            const int64_t m = (a + b) >> 1;
            if (in[m] < v)
                a = m + 1;
            else
                b = m;
        }
        out[ps + o + (a - lo)] = v;
    }
}

__global__ void __launch_bounds__(kTrThreads)
tr_dst_kernel(const int32_t *__restrict__ perm, const int32_t *__restrict__ row_of, int64_t E,
              int32_t *__restrict__ dst) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < E; k += stride)
        dst[k] = row_of[perm[k]];
}

static cudaError_t exclusive_scan(const int32_t *in, int32_t *out, int64_t n, int64_t *sums,
                                  cudaStream_t s) {
    const int64_t nb = (n + kScanTile - 1) / kScanTile;
    tr_scan_tiles_kernel<<<(unsigned)nb, kTrThreads, 0, s>>>(in, n, out, sums);
    tr_scan_sums_kernel<<<1, 1024, 0, s>>>(sums, nb);
    tr_scan_add_kernel<<<(unsigned)nb, kTrThreads, 0, s>>>(out, n, sums);
    return cudaGetLastError();
}

}  // namespace gat

using namespace gat;

extern "C" gat_status_t gat_transpose_destroy(gat_transpose_t t) {
    if (!t) return GAT_OK;
    cudaFree(t->src_ptr);
    cudaFree(t->perm);
    cudaFree(t->dst);
    gat_plan_destroy(t->src_plan);
    delete t;
    return GAT_OK;
}

extern "C" gat_status_t gat_transpose_create(const int32_t *row_ptr, const int32_t *col_idx,
                                             int64_t n_rows, int64_t n_src, int64_t n_edges,
                                             void *stream, gat_transpose_t *out) {
    if (!out) return fail(GAT_ERR_INVALID_ARG, "gat_transpose_create: output pointer is NULL");
    *out = nullptr;
    if (n_rows < 0 || n_src < 0 || n_edges < 0 || n_rows >= INT32_MAX || n_src >= INT32_MAX ||
        n_edges >= INT32_MAX)
        return fail(GAT_ERR_INVALID_ARG, "gat_transpose_create: bad sizes");
    if (!row_ptr || (n_edges > 0 && !col_idx))
        return fail(GAT_ERR_INVALID_ARG, "gat_transpose_create: NULL pointer");
    if (n_edges > 0 && n_src == 0)
        return fail(GAT_ERR_INDEX_OUT_OF_RANGE, "gat_transpose_create: edges but no sources");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t E = n_edges;
    gat_transpose_s *t = new gat_transpose_s();
    t->n_rows = n_rows;
    t->n_src = n_src;
    t->n_edges = E;
    cudaGetDevice(&t->device);
    // one scratch block: counts / cursors [n_src + 1], flags [2] (bad index,
    // largest group), scan tile sums, and for E > 0 row_of, tmp and seg [E]
    const int64_t nb = (n_src + 1 + kScanTile - 1) / kScanTile;
    const size_t o_flags = (size_t)(n_src + 1) * 4;
    const size_t o_sums = (o_flags + 8 + 15) & ~(size_t)15;
    const size_t o_row_of = (o_sums + (size_t)nb * 8 + 15) & ~(size_t)15;
    const size_t o_tmp = o_row_of + (size_t)E * 4;
    const size_t o_seg = o_tmp + (size_t)E * 4;
    const size_t scratch_bytes = o_seg + (size_t)E * 4;
    unsigned char *scratch = nullptr;
    int32_t host_flags[2] = {0, 0};
    gat_status_t st = GAT_OK;
    cudaError_t e = cudaMalloc(&t->src_ptr, (n_src + 1) * sizeof(int32_t));
    if (e == cudaSuccess) e = cudaMalloc(&t->perm, (E > 0 ? E : 1) * sizeof(int32_t));
    if (e == cudaSuccess) e = cudaMalloc(&t->dst, (E > 0 ? E : 1) * sizeof(int32_t));
    if (e == cudaSuccess) e = cudaMalloc(&scratch, scratch_bytes);
    if (e == cudaSuccess) e = cudaMemsetAsync(scratch, 0, o_flags + 8, s);  // counts and flags
    if (e != cudaSuccess) {
        st = cuda_fail(e, "gat_transpose_create: allocation");
        goto done;
    }
    {
        int32_t *cnt = reinterpret_cast<int32_t *>(scratch);
        int32_t *flags = reinterpret_cast<int32_t *>(scratch + o_flags);
        int64_t *sums = reinterpret_cast<int64_t *>(scratch + o_sums);
        int32_t *row_of = reinterpret_cast<int32_t *>(scratch + o_row_of);
        int32_t *tmp = reinterpret_cast<int32_t *>(scratch + o_tmp);
        int32_t *seg = reinterpret_cast<int32_t *>(scratch + o_seg);
        if (E > 0) {
            // counts and the largest group; an out-of-range column index stops
            // the build here
            tr_count_kernel<<<grid_for(E, kTrThreads), kTrThreads, 0, s>>>(col_idx, E, n_src, cnt,
                                                                             flags);
            tr_max_kernel<<<grid_for(n_src, kTrThreads), kTrThreads, 0, s>>>(cnt, n_src, flags + 1);
            if ((st = check_launch("gat_transpose_create: count")) != GAT_OK) goto done;
            e = cudaMemcpyAsync(host_flags, flags, 2 * sizeof(int32_t), cudaMemcpyDeviceToHost, s);
            if (e == cudaSuccess) e = cudaStreamSynchronize(s);
            if (e != cudaSuccess) {
                st = cuda_fail(e, "gat_transpose_create: count");
                goto done;
            }
            if (host_flags[0]) {
                st = fail(GAT_ERR_INDEX_OUT_OF_RANGE,
                          "gat_transpose_create: a column index is outside [0, n_src)");
                goto done;
            }
            t->max_src_degree = host_flags[1];
        }
        e = exclusive_scan(cnt, t->src_ptr, n_src + 1, sums, s);
        if (e != cudaSuccess) {
            st = cuda_fail(e, "gat_transpose_create: scan");
            goto done;
        }
        if (E > 0) {
            e = cudaMemcpyAsync(cnt, t->src_ptr, n_src * sizeof(int32_t), cudaMemcpyDeviceToDevice,
                                s);
            if (e != cudaSuccess) {
                st = cuda_fail(e, "gat_transpose_create: cursor copy");
                goto done;
            }
            const unsigned rw = grid_for(n_rows * 32, kTrThreads);
            tr_row_of_kernel<<<rw, kTrThreads, 0, s>>>(row_ptr, n_rows, row_of);
            tr_fill_kernel<<<grid_for(E, kTrThreads), kTrThreads, 0, s>>>(col_idx, E, cnt, t->perm);
            tr_sort32_kernel<<<grid_for(n_src * 32, kTrThreads), kTrThreads, 0, s>>>(
                t->perm, t->src_ptr, n_src);
            if ((st = check_launch("gat_transpose_create: fill")) != GAT_OK) goto done;
            int32_t *a = t->perm, *b = tmp;
            if (t->max_src_degree > 32) {
                tr_seg_kernel<<<grid_for(n_src * 32, kTrThreads), kTrThreads, 0, s>>>(
                    t->src_ptr, n_src, seg);
                for (int64_t L = 32; L < t->max_src_degree; L <<= 1) {
                    tr_merge_kernel<<<grid_for(E, kTrThreads), kTrThreads, 0, s>>>(
                        a, b, seg, t->src_ptr, E, L);
                    int32_t *c = a;
                    a = b;
                    b = c;
                }
                if ((st = check_launch("gat_transpose_create: merge")) != GAT_OK) goto done;
            }
            if (a != t->perm) {  // the sorted order ended in the scratch buffer
                e = cudaMemcpyAsync(t->perm, a, E * sizeof(int32_t), cudaMemcpyDeviceToDevice, s);
                if (e != cudaSuccess) {
                    st = cuda_fail(e, "gat_transpose_create: order copy");
                    goto done;
                }
            }
            tr_dst_kernel<<<grid_for(E, kTrThreads), kTrThreads, 0, s>>>(t->perm, row_of, E,
                                                                         t->dst);
            if ((st = check_launch("gat_transpose_create: dst")) != GAT_OK) goto done;
        }
    }
    st = gat_plan_create(t->src_ptr, n_src, E, 0, 0, stream, &t->src_plan);
done:
    if (st == GAT_OK) {
        e = cudaStreamSynchronize(s);
        if (e != cudaSuccess) st = cuda_fail(e, "gat_transpose_create");
    } else {
        cudaStreamSynchronize(s);
    }
    cudaFree(scratch);
    if (st != GAT_OK) {
        gat_transpose_destroy(t);
        return st;
    }
    *out = t;
    return GAT_OK;
}

extern "C" gat_status_t gat_transpose_info(gat_transpose_t t, int64_t *n_rows, int64_t *n_src,
                                           int64_t *n_edges, int32_t *max_src_degree,
                                           int64_t *n_heavy_src) {
    if (!t) return fail(GAT_ERR_INVALID_ARG, "gat_transpose_info: NULL transpose");
    if (n_rows) *n_rows = t->n_rows;
    if (n_src) *n_src = t->n_src;
    if (n_edges) *n_edges = t->n_edges;
    if (max_src_degree) *max_src_degree = t->max_src_degree;
    if (n_heavy_src) *n_heavy_src = t->src_plan ? t->src_plan->n_heavy : 0;
    return GAT_OK;
}

extern "C" gat_status_t gat_transpose_export(gat_transpose_t t, int32_t *src_ptr, int32_t *perm,
                                             int32_t *dst, void *stream) {
    if (!t) return fail(GAT_ERR_INVALID_ARG, "gat_transpose_export: NULL transpose");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    if (src_ptr)
        e = cudaMemcpyAsync(src_ptr, t->src_ptr, (t->n_src + 1) * sizeof(int32_t),
                            cudaMemcpyDeviceToDevice, s);
    if (e == cudaSuccess && perm && t->n_edges)
        e = cudaMemcpyAsync(perm, t->perm, t->n_edges * sizeof(int32_t), cudaMemcpyDeviceToDevice, s);
    if (e == cudaSuccess && dst && t->n_edges)
        e = cudaMemcpyAsync(dst, t->dst, t->n_edges * sizeof(int32_t), cudaMemcpyDeviceToDevice, s);
    return e == cudaSuccess ? GAT_OK : cuda_fail(e, "gat_transpose_export");
}
