// plan.cu - degree-bucket plan (light rows / chunked heavy rows), graph
// validation, and the library's status/error plumbing.
//
// The pages give each destination row to one thread, warp or block and pick
// the granularity by hand (Kimi-K2.6 l2_p37, kernel design discussion: block
// per destination vs. warp per destination). On a power-law graph no single
// choice balances, so rows are bucketed once per graph: light rows run one
// warp each, heavy rows are cut into fixed-size edge chunks.
#include <cstdarg>
#include <cstdio>

#include "plan.cuh"

namespace gat {

// ---------------------------------------------------------------------------
// error plumbing
// ---------------------------------------------------------------------------
static thread_local char g_err[512] = "";

gat_status_t fail(gat_status_t st, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return st;
}

gat_status_t cuda_fail(cudaError_t err, const char *what) {
    return fail(GAT_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(err), cudaGetErrorString(err));
}

gat_status_t check_launch(const char *what) {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, what);
    return GAT_OK;
}

// ---------------------------------------------------------------------------
// plan kernels
// ---------------------------------------------------------------------------
__device__ __forceinline__ void row_class(const int32_t *__restrict__ row_ptr, int64_t r,
                                          int64_t n_rows, int32_t T, int32_t C, int &is_heavy,
                                          int &chunks, int &deg) {
    is_heavy = 0;
    chunks = 0;
    deg = 0;
    if (r < n_rows) {
        deg = row_ptr[r + 1] - row_ptr[r];
        if (deg > T) {
            is_heavy = 1;
            chunks = (deg + C - 1) / C;
        }
    }
}

// Block-wide exclusive scan of two int counters in thread order; returns the
// block totals. Uses 2 * 32 ints of shared scratch.
__device__ __forceinline__ void block_scan2(int a, int b, int &pa, int &pb, int &ta, int &tb,
                                            int *sh) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nw = blockDim.x >> 5;
    int ia = a, ib = b;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int xa = __shfl_up_sync(kFull, ia, o), xb = __shfl_up_sync(kFull, ib, o);
        if (lane >= o) {
            ia += xa;
            ib += xb;
        }
    }
    if (lane == 31) {
        sh[warp] = ia;
        sh[32 + warp] = ib;
    }
    __syncthreads();
    if (warp == 0) {
        int wa = lane < nw ? sh[lane] : 0, wb = lane < nw ? sh[32 + lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int xa = __shfl_up_sync(kFull, wa, o), xb = __shfl_up_sync(kFull, wb, o);
            if (lane >= o) {
                wa += xa;
                wb += xb;
            }
        }
        if (lane < nw) {
            sh[lane] = wa;
            sh[32 + lane] = wb;
        }
    }
    __syncthreads();
    const int ba = warp ? sh[warp - 1] : 0, bb = warp ? sh[32 + warp - 1] : 0;
    pa = ba + ia - a;
    pb = bb + ib - b;
    ta = sh[nw - 1];
    tb = sh[32 + nw - 1];
    __syncthreads();
}

__global__ void __launch_bounds__(kPlanThreads)
plan_count_kernel(const int32_t *__restrict__ row_ptr, int64_t n_rows, int32_t T, int32_t C,
                  Counts *__restrict__ block_counts) {
    __shared__ int sh[64];
    const int64_t base = (int64_t)blockIdx.x * kPlanRowsPerBlock;
    long long h = 0, c = 0, e = 0;
    for (int k = 0; k < kPlanRounds; ++k) {
        int is_heavy, chunks, deg;
        row_class(row_ptr, base + k * kPlanThreads + threadIdx.x, n_rows, T, C, is_heavy, chunks,
                  deg);
        h += is_heavy;
        c += chunks;
        e += is_heavy ? deg : 0;
    }
    // block reduction through the scan helper (totals only); edges reduced separately
    int pa, pb, ta, tb;
    block_scan2((int)h, (int)c, pa, pb, ta, tb, sh);
    long long es = e;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) es += __shfl_xor_sync(kFull, es, o);
    __shared__ long long she[kPlanThreads / 32];
    if ((threadIdx.x & 31) == 0) she[threadIdx.x >> 5] = es;
    __syncthreads();
    if (threadIdx.x == 0) {
        long long t = 0;
        for (int w = 0; w < kPlanThreads / 32; ++w) t += she[w];
        block_counts[blockIdx.x] = Counts{ta, tb, t};
    }
}

// Exclusive scan of the per-block counts (one block, sequential tiles).
__global__ void __launch_bounds__(kPlanScanThreads)
plan_scan_kernel(const Counts *__restrict__ block_counts, int64_t nb, Counts *__restrict__ offsets,
                 Counts *__restrict__ totals) {
    __shared__ long long sh[3][32];
    long long carry_h = 0, carry_c = 0, carry_e = 0;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int64_t t0 = 0; t0 < nb; t0 += blockDim.x) {
        const int64_t i = t0 + threadIdx.x;
        Counts v = i < nb ? block_counts[i] : Counts{0, 0, 0};
        long long a = v.heavy, b = v.chunks, c = v.edges;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            long long xa = __shfl_up_sync(kFull, a, o), xb = __shfl_up_sync(kFull, b, o),
                      xc = __shfl_up_sync(kFull, c, o);
            if (lane >= o) {
                a += xa;
                b += xb;
                c += xc;
            }
        }
        if (lane == 31) {
            sh[0][warp] = a;
            sh[1][warp] = b;
            sh[2][warp] = c;
        }
        __syncthreads();
        if (warp == 0) {
            const int nw = blockDim.x >> 5;
            long long wa = lane < nw ? sh[0][lane] : 0, wb = lane < nw ? sh[1][lane] : 0,
                      wc = lane < nw ? sh[2][lane] : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                long long xa = __shfl_up_sync(kFull, wa, o), xb = __shfl_up_sync(kFull, wb, o),
                          xc = __shfl_up_sync(kFull, wc, o);
                if (lane >= o) {
                    wa += xa;
                    wb += xb;
                    wc += xc;
                }
            }
            if (lane < nw) {
                sh[0][lane] = wa;
                sh[1][lane] = wb;
                sh[2][lane] = wc;
            }
        }
        __syncthreads();
        const long long bh = warp ? sh[0][warp - 1] : 0, bc = warp ? sh[1][warp - 1] : 0,
                        be = warp ? sh[2][warp - 1] : 0;
        if (i < nb)
            offsets[i] = Counts{carry_h + bh + a - v.heavy, carry_c + bc + b - v.chunks,
                                carry_e + be + c - v.edges};
        const int last = (blockDim.x >> 5) - 1;
        carry_h += sh[0][last];
        carry_c += sh[1][last];
        carry_e += sh[2][last];
        __syncthreads();
    }
    if (threadIdx.x == 0) *totals = Counts{carry_h, carry_c, carry_e};
}

__global__ void __launch_bounds__(kPlanThreads)
plan_fill_kernel(const int32_t *__restrict__ row_ptr, int64_t n_rows, int32_t T, int32_t C,
                 const Counts *__restrict__ offsets, const Counts *__restrict__ totals,
                 int32_t *__restrict__ heavy_rows, int32_t *__restrict__ chunk_start,
                 int32_t *__restrict__ chunk_row) {
    __shared__ int sh[64];
    const int64_t base = (int64_t)blockIdx.x * kPlanRowsPerBlock;
    long long oh = offsets[blockIdx.x].heavy, oc = offsets[blockIdx.x].chunks;
    for (int k = 0; k < kPlanRounds; ++k) {
        const int64_t r = base + k * kPlanThreads + threadIdx.x;
        int is_heavy, chunks, deg;
        row_class(row_ptr, r, n_rows, T, C, is_heavy, chunks, deg);
        int ph, pc, th, tc;
        block_scan2(is_heavy, chunks, ph, pc, th, tc, sh);
        if (is_heavy) {
            const long long hi = oh + ph, c0 = oc + pc;
            heavy_rows[hi] = (int32_t)r;
            chunk_start[hi] = (int32_t)c0;
            for (int j = 0; j < chunks; ++j) chunk_row[c0 + j] = (int32_t)hi;
        }
        oh += th;
        oc += tc;
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) chunk_start[totals->heavy] = (int32_t)totals->chunks;
}

// One 16-byte descriptor per chunk {row, first edge, end edge, heavy index},
// so a warp learns its chunk's edge range with one load instead of a chain
// chunk_row -> heavy_rows / chunk_start -> row_ptr.
__global__ void __launch_bounds__(kPlanThreads)
plan_desc_kernel(const int32_t *__restrict__ row_ptr, const int32_t *__restrict__ heavy_rows,
                 const int32_t *__restrict__ chunk_start, int64_t n_heavy, int32_t C,
                 int4 *__restrict__ desc) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t hr = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; hr < n_heavy; hr += stride) {
        const int32_t row = heavy_rows[hr];
        const int32_t rs = row_ptr[row], re = row_ptr[row + 1];
        const int32_t c0 = chunk_start[hr], c1 = chunk_start[hr + 1];
        for (int32_t c = c0; c < c1; ++c) {
            const int32_t e0 = rs + (c - c0) * C;
            desc[c] = make_int4(row, e0, min(e0 + C, re), (int32_t)hr);
        }
    }
}

// ---------------------------------------------------------------------------
// graph validation
// ---------------------------------------------------------------------------
__global__ void validate_kernel(const int32_t *__restrict__ row_ptr,
                                const int32_t *__restrict__ col_idx, int64_t n_rows, int64_t n_src,
                                int64_t n_edges, int32_t *flag) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t t0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    int bad = 0;
    if (t0 == 0 && (row_ptr[0] != 0 || (int64_t)row_ptr[n_rows] != n_edges)) bad = 1;
    for (int64_t i = t0; i < n_rows; i += stride)
        if (row_ptr[i + 1] < row_ptr[i]) bad = 1;
    if (col_idx)
        for (int64_t e = t0; e < n_edges; e += stride) {
            const int32_t c = col_idx[e];
            if (c < 0 || (int64_t)c >= n_src) bad = 1;
        }
    if (__any_sync(kFull, bad) && (threadIdx.x & 31) == 0) atomicOr(flag, 1);
}

// ---------------------------------------------------------------------------
// row shards: a contiguous row range as a graph of its own
// ---------------------------------------------------------------------------
__global__ void rebase_row_ptr_kernel(const int32_t *__restrict__ row_ptr, int64_t r0, int64_t n,
                                      int32_t *__restrict__ out) {
    const int32_t base = __ldg(row_ptr + r0);
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i <= n; i += stride)
        out[i] = __ldg(row_ptr + r0 + i) - base;
}

}  // namespace gat

using namespace gat;

// ---------------------------------------------------------------------------
// C ABI: row partition (host) and shard row pointers (device)
// ---------------------------------------------------------------------------
extern "C" gat_status_t gat_partition_rows(const int32_t *row_ptr, int64_t n_rows,
                                           int32_t parts, int64_t *row_begin) {
    if (!row_ptr || !row_begin || n_rows < 0 || parts < 1)
        return fail(GAT_ERR_INVALID_ARG, "gat_partition_rows: bad arguments");
    for (int64_t i = 0; i < n_rows; ++i)
        if (row_ptr[i + 1] < row_ptr[i])
            return fail(GAT_ERR_INDEX_OUT_OF_RANGE, "gat_partition_rows: row_ptr decreases at %lld",
                        (long long)i);
    // weight of rows [0, r): r + row_ptr[r] - row_ptr[0] (a row's q and out rows plus
    // one gathered source row per edge), non-decreasing in r; boundary p is the
    // first r whose prefix weight reaches p / parts of the total
    const int64_t total = n_rows + (int64_t)row_ptr[n_rows] - row_ptr[0];
    row_begin[0] = 0;
    for (int32_t q = 1; q < parts; ++q) {
        const int64_t target = (total * q + parts - 1) / parts;
        int64_t lo = row_begin[q - 1], hi = n_rows;  // first r in [lo, hi] with weight >= target
        while (lo < hi) {
            const int64_t mid = lo + (hi - lo) / 2;
            if (mid + (int64_t)row_ptr[mid] - row_ptr[0] >= target)
                hi = mid;
            else
                lo = mid + 1;
        }
        row_begin[q] = lo;
    }
    row_begin[parts] = n_rows;
    return GAT_OK;
}

extern "C" gat_status_t gat_rebase_row_ptr(const int32_t *row_ptr, int64_t r0, int64_t r1,
                                           int32_t *out, void *stream) {
    if (!row_ptr || !out || r0 < 0 || r1 < r0)
        return fail(GAT_ERR_INVALID_ARG, "gat_rebase_row_ptr: bad arguments");
    const int64_t n = r1 - r0;
    int64_t blocks = (n + 1 + 255) / 256;
    const int64_t cap = (int64_t)sm_count() * 8;
    if (blocks > cap) blocks = cap;
    rebase_row_ptr_kernel<<<(unsigned)blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(
        row_ptr, r0, n, out);
    return check_launch("gat_rebase_row_ptr");
}

// ---------------------------------------------------------------------------
// C ABI: status / version
// ---------------------------------------------------------------------------
extern "C" const char *gat_status_string(gat_status_t s) {
    switch (s) {
        case GAT_OK: return "GAT_OK";
        case GAT_ERR_INVALID_ARG: return "GAT_ERR_INVALID_ARG";
        case GAT_ERR_UNSUPPORTED: return "GAT_ERR_UNSUPPORTED";
        case GAT_ERR_CUDA: return "GAT_ERR_CUDA";
        case GAT_ERR_WORKSPACE: return "GAT_ERR_WORKSPACE";
        case GAT_ERR_INDEX_OUT_OF_RANGE: return "GAT_ERR_INDEX_OUT_OF_RANGE";
        case GAT_ERR_PLAN_MISMATCH: return "GAT_ERR_PLAN_MISMATCH";
    }
    return "GAT_ERR_UNKNOWN";
}

extern "C" const char *gat_last_error(void) { return g_err; }

extern "C" int32_t gat_version(void) { return 10000 * 0 + 100 * 1 + 0; }

// ---------------------------------------------------------------------------
// C ABI: plan
// ---------------------------------------------------------------------------
extern "C" gat_status_t gat_plan_destroy(gat_plan_t p) {
    if (!p) return GAT_OK;
    cudaFree(p->heavy_rows);
    cudaFree(p->chunk_start);
    cudaFree(p->chunk_row);
    cudaFree(p->counters);
    cudaFree(p->chunk_desc);
    cudaFree(p->sched);
    delete p;
    return GAT_OK;
}

extern "C" gat_status_t gat_plan_create(const int32_t *row_ptr, int64_t n_rows, int64_t n_edges,
                                        int32_t heavy_threshold, int32_t chunk_edges,
                                        void *stream, gat_plan_t *out) {
    if (!out) return fail(GAT_ERR_INVALID_ARG, "gat_plan_create: plan output pointer is NULL");
    *out = nullptr;
    if (!row_ptr) return fail(GAT_ERR_INVALID_ARG, "gat_plan_create: row_ptr is NULL");
    if (n_rows < 0 || n_edges < 0 || n_rows >= INT32_MAX || n_edges >= INT32_MAX)
        return fail(GAT_ERR_INVALID_ARG, "gat_plan_create: bad sizes n_rows=%lld n_edges=%lld",
                    (long long)n_rows, (long long)n_edges);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    gat_plan_s *p = new gat_plan_s();
    p->n_rows = n_rows;
    p->n_edges = n_edges;
    p->heavy_threshold = heavy_threshold > 0 ? heavy_threshold : 128;
    p->chunk_edges = chunk_edges > 0 ? chunk_edges : 256;
    cudaGetDevice(&p->device);
    if (n_rows == 0) {
        cudaError_t e = cudaMalloc(&p->chunk_start, sizeof(int32_t));
        if (e == cudaSuccess) e = cudaMemsetAsync(p->chunk_start, 0, sizeof(int32_t), s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
        if (e != cudaSuccess) {
            gat_plan_destroy(p);
            return cuda_fail(e, "gat_plan_create");
        }
        *out = p;
        return GAT_OK;
    }
    const int64_t nb = plan_blocks(n_rows);
    Counts *scratch = nullptr;  // [nb] counts, [nb] offsets, [1] totals
    cudaError_t e = cudaMalloc(&scratch, (2 * nb + 1) * sizeof(Counts));
    Counts host_tot{0, 0, 0};
    gat_status_t st = GAT_OK;
    if (e != cudaSuccess) {
        st = cuda_fail(e, "gat_plan_create: scratch allocation");
        goto out_fail;
    }
    plan_count_kernel<<<(unsigned)nb, kPlanThreads, 0, s>>>(row_ptr, n_rows, p->heavy_threshold,
                                                            p->chunk_edges, scratch);
    plan_scan_kernel<<<1, kPlanScanThreads, 0, s>>>(scratch, nb, scratch + nb, scratch + 2 * nb);
    if ((st = check_launch("gat_plan_create: count/scan")) != GAT_OK) goto out_fail;
    e = cudaMemcpyAsync(&host_tot, scratch + 2 * nb, sizeof(Counts), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) {
        st = cuda_fail(e, "gat_plan_create: reading class sizes");
        goto out_fail;
    }
    p->n_heavy = host_tot.heavy;
    p->n_chunks = host_tot.chunks;
    p->heavy_edges = host_tot.edges;
    if (p->n_chunks >= INT32_MAX) {
        st = fail(GAT_ERR_UNSUPPORTED, "gat_plan_create: too many chunks");
        goto out_fail;
    }
    e = cudaMalloc(&p->chunk_start, (p->n_heavy + 1) * sizeof(int32_t));
    if (e == cudaSuccess && p->n_heavy) e = cudaMalloc(&p->heavy_rows, p->n_heavy * sizeof(int32_t));
    if (e == cudaSuccess && p->n_heavy) e = cudaMalloc(&p->counters, p->n_heavy * sizeof(int32_t));
    if (e == cudaSuccess && p->n_chunks) e = cudaMalloc(&p->chunk_row, p->n_chunks * sizeof(int32_t));
    if (e == cudaSuccess && p->n_chunks) e = cudaMalloc(&p->chunk_desc, p->n_chunks * sizeof(int4));
    if (e == cudaSuccess) e = cudaMalloc(&p->sched, 4 * sizeof(int32_t));
    if (e == cudaSuccess) e = cudaMemsetAsync(p->sched, 0, 4 * sizeof(int32_t), s);
    if (e == cudaSuccess && p->n_heavy)
        e = cudaMemsetAsync(p->counters, 0, p->n_heavy * sizeof(int32_t), s);
    if (e != cudaSuccess) {
        st = cuda_fail(e, "gat_plan_create: plan allocation");
        goto out_fail;
    }
    plan_fill_kernel<<<(unsigned)nb, kPlanThreads, 0, s>>>(
        row_ptr, n_rows, p->heavy_threshold, p->chunk_edges, scratch + nb, scratch + 2 * nb,
        p->heavy_rows, p->chunk_start, p->chunk_row);
    if ((st = check_launch("gat_plan_create: fill")) != GAT_OK) goto out_fail;
    if (p->n_heavy > 0) {
        int64_t db = (p->n_heavy + kPlanThreads - 1) / kPlanThreads;
        if (db > 4096) db = 4096;
        plan_desc_kernel<<<(unsigned)db, kPlanThreads, 0, s>>>(row_ptr, p->heavy_rows, p->chunk_start,
                                                              p->n_heavy, p->chunk_edges,
                                                              p->chunk_desc);
        if ((st = check_launch("gat_plan_create: descriptors")) != GAT_OK) goto out_fail;
    }
    e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) {
        st = cuda_fail(e, "gat_plan_create: fill");
        goto out_fail;
    }
    cudaFree(scratch);
    *out = p;
    return GAT_OK;
out_fail:
    cudaFree(scratch);
    gat_plan_destroy(p);
    return st;
}

extern "C" gat_status_t gat_plan_info(gat_plan_t p, int64_t *n_rows, int64_t *n_edges,
                                      int32_t *heavy_threshold, int32_t *chunk_edges,
                                      int64_t *n_heavy, int64_t *n_chunks) {
    if (!p) return fail(GAT_ERR_INVALID_ARG, "gat_plan_info: plan is NULL");
    if (n_rows) *n_rows = p->n_rows;
    if (n_edges) *n_edges = p->n_edges;
    if (heavy_threshold) *heavy_threshold = p->heavy_threshold;
    if (chunk_edges) *chunk_edges = p->chunk_edges;
    if (n_heavy) *n_heavy = p->n_heavy;
    if (n_chunks) *n_chunks = p->n_chunks;
    return GAT_OK;
}

extern "C" gat_status_t gat_plan_export(gat_plan_t p, int32_t *heavy_rows, int32_t *chunk_start,
                                        int32_t *chunk_row, void *stream) {
    if (!p) return fail(GAT_ERR_INVALID_ARG, "gat_plan_export: plan is NULL");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    if (heavy_rows && p->n_heavy)
        e = cudaMemcpyAsync(heavy_rows, p->heavy_rows, p->n_heavy * sizeof(int32_t),
                            cudaMemcpyDeviceToDevice, s);
    if (e == cudaSuccess && chunk_start)
        e = cudaMemcpyAsync(chunk_start, p->chunk_start, (p->n_heavy + 1) * sizeof(int32_t),
                            cudaMemcpyDeviceToDevice, s);
    if (e == cudaSuccess && chunk_row && p->n_chunks)
        e = cudaMemcpyAsync(chunk_row, p->chunk_row, p->n_chunks * sizeof(int32_t),
                            cudaMemcpyDeviceToDevice, s);
    if (e != cudaSuccess) return cuda_fail(e, "gat_plan_export");
    return GAT_OK;
}

extern "C" gat_status_t gat_validate_graph(const int32_t *row_ptr, const int32_t *col_idx,
                                           int64_t n_rows, int64_t n_src, int64_t n_edges,
                                           int32_t *flag, void *stream) {
    if (!row_ptr || !flag || n_rows < 0 || n_src < 0 || n_edges < 0)
        return fail(GAT_ERR_INVALID_ARG, "gat_validate_graph: bad arguments");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemsetAsync(flag, 0, sizeof(int32_t), s);
    if (e != cudaSuccess) return cuda_fail(e, "gat_validate_graph");
    const int64_t work = n_rows > n_edges ? n_rows : n_edges;
    int64_t blocks = (work + 255) / 256;
    const int64_t cap = (int64_t)sm_count() * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    validate_kernel<<<(unsigned)blocks, 256, 0, s>>>(row_ptr, col_idx, n_rows, n_src, n_edges,
                                                     flag);
    gat_status_t st = check_launch("gat_validate_graph");
    if (st != GAT_OK) return st;
    int32_t h = 0;
    e = cudaMemcpyAsync(&h, flag, sizeof(int32_t), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "gat_validate_graph");
    if (h) return fail(GAT_ERR_INDEX_OUT_OF_RANGE, "gat_validate_graph: malformed row_ptr/col_idx");
    return GAT_OK;
}
