// no_alloc.cu - gat_fused_layer_no_alloc: the fused graph-attention layer
// with heavy-row splitting, for callers that cannot allocate device memory.
//
// Who needs it: code that runs where cudaMalloc is off limits - inside a
// framework that owns every byte of device memory through its own pool,
// inside an allocator or memory-pressure callback, in a process whose
// allocation budget is already spent, or in an embedding that only hands out
// the input and output buffers. gat_plan_create allocates its plan arrays and
// gat_fused_layer wants a caller workspace; this entry point needs neither.
//
// How: the degree-bucket plan, its scan scratch, the per-row arrival counters
// and the chunk softmax states all live in one file-scope device array
// (kNoAllocScratchBytes, 32 MiB). Every GPU that loads the library holds that
// array until the process exits. Its device address is looked up once per
// device (cudaGetSymbolAddress, with that device current) on the first call
// made on the device. The kernels are the library's own plan and fused-layer
// kernels, unchanged.
//
// The array is shared by every call and keeps the previous call's contents:
// each call clears the arrival counters it needs. Calls whose work overlaps
// on the GPU (other streams, other host threads) race on the array; serialise
// them. Every call copies the plan's size back into host memory and
// synchronises `stream` to read it, so no call of this entry point can be
// recorded by stream capture into a CUDA graph (the first call's address
// lookup is a further reason); call it on an uncaptured stream.
#include <mutex>

#include "plan.cuh"
#include "row_engine.cuh"

namespace gat {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;
constexpr int32_t kNoAllocThreshold = 64;  // heavy rows: degree > 64
constexpr int32_t kNoAllocChunk = 64;      // edges per chunk
constexpr float kLog2eNA = 1.4426950408889634f;

static __device__ __align__(256) unsigned char g_no_alloc_scratch[kNoAllocScratchBytes];

static std::mutex g_scratch_mu;
static void *g_scratch_addr[64] = {nullptr};

// Device address of the scratch array on the current device (looked up once).
static gat_status_t scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "gat_fused_layer_no_alloc: cudaGetDevice");
    if (dev < 0 || dev >= 64)
        return fail(GAT_ERR_UNSUPPORTED, "gat_fused_layer_no_alloc: device ordinal %d", dev);
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_no_alloc_scratch);
        if (e != cudaSuccess)
            return cuda_fail(e, "gat_fused_layer_no_alloc: cudaGetSymbolAddress");
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return GAT_OK;
}

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

template <typename T, int V, int LE>
static gat_status_t launch_no_alloc(const EngineParams &p, cudaStream_t s) {
    return launch_fused_engine<T, V, LE>(p, s);
}

template <typename T>
static gat_status_t dispatch_no_alloc(const EngineParams &p, int V, int LE, cudaStream_t s) {
    if (V == 1 && LE == 4) return launch_no_alloc<T, 1, 4>(p, s);
    if (V == 1 && LE == 8) return launch_no_alloc<T, 1, 8>(p, s);
    if (V == 1 && LE == 16) return launch_no_alloc<T, 1, 16>(p, s);
    if (V == 1 && LE == 32) return launch_no_alloc<T, 1, 32>(p, s);
    if (V == 2) return launch_no_alloc<T, 2, 32>(p, s);
    return launch_no_alloc<T, 4, 32>(p, s);
}

}  // namespace gat

using namespace gat;

extern "C" gat_status_t gat_fused_layer_no_alloc(const int32_t *row_ptr, const int32_t *col_idx,
                                                 int64_t n_rows, int64_t n_src, int64_t n_edges,
                                                 int32_t H, int32_t Dh, float scale,
                                                 const void *q, const void *k, const void *v,
                                                 gat_dtype_t dtype, void *out, void *stream) {
    if (n_rows < 0 || n_src < 0 || n_edges < 0 || H < 1 || Dh < 1 || n_rows >= INT32_MAX ||
        n_edges >= INT32_MAX)
        return fail(GAT_ERR_INVALID_ARG, "gat_fused_layer_no_alloc: bad sizes");
    if (dtype != GAT_F32 && dtype != GAT_BF16)
        return fail(GAT_ERR_UNSUPPORTED, "gat_fused_layer_no_alloc: unknown dtype %d", (int)dtype);
    if (n_rows == 0) return GAT_OK;
    if (!row_ptr || !q || !out || (n_edges > 0 && (!col_idx || !k || !v)))
        return fail(GAT_ERR_INVALID_ARG, "gat_fused_layer_no_alloc: NULL pointer");
    const int eb = dtype == GAT_F32 ? 4 : 2;
    int V = 0, LE = 0;
    const bool vec_ok =
        aligned16(q) && aligned16(out) && (n_edges == 0 || (aligned16(k) && aligned16(v)));
    if (!vec_ok || !engine_shape(H, Dh, eb, V, LE))
        return fail(GAT_ERR_UNSUPPORTED,
                    "gat_fused_layer_no_alloc: needs 16-byte aligned rows and a vector-engine "
                    "shape (H=%d, Dh=%d)", (int)H, (int)Dh);

    // the scan records must fit before anything is launched
    const int64_t nb = plan_blocks(n_rows);
    const size_t counts_bytes = align256((size_t)(2 * nb + 1) * sizeof(Counts));
    if (counts_bytes > kNoAllocScratchBytes)
        return fail(GAT_ERR_WORKSPACE,
                    "gat_fused_layer_no_alloc: %lld rows exceed the %zu-byte static scratch",
                    (long long)n_rows, kNoAllocScratchBytes);
    void *base = nullptr;
    gat_status_t st = scratch_address(&base);
    if (st != GAT_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char *sc = static_cast<char *>(base);
    Counts *counts = reinterpret_cast<Counts *>(sc);

    // plan sizes (one read-back)
    plan_count_kernel<<<(unsigned)nb, kPlanThreads, 0, s>>>(row_ptr, n_rows, kNoAllocThreshold,
                                                  kNoAllocChunk, counts);
    plan_scan_kernel<<<1, kPlanScanThreads, 0, s>>>(counts, nb, counts + nb, counts + 2 * nb);
    if ((st = check_launch("gat_fused_layer_no_alloc: plan count")) != GAT_OK) return st;
    Counts tot{0, 0, 0};
    cudaError_t e =
        cudaMemcpyAsync(&tot, counts + 2 * nb, sizeof(Counts), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "gat_fused_layer_no_alloc: reading plan size");

    // carve the rest of the scratch: plan arrays, counters, chunk states
    const int64_t sf = slot_floats(H, Dh);
    size_t off = counts_bytes;
    const size_t o_rows = off;
    off += align256((size_t)tot.heavy * 4);
    const size_t o_start = off;
    off += align256((size_t)(tot.heavy + 1) * 4);
    const size_t o_crow = off;
    off += align256((size_t)tot.chunks * 4);
    const size_t o_cnt = off;
    off += align256((size_t)tot.heavy * 4);
    const size_t o_desc = off;
    off += align256((size_t)tot.chunks * sizeof(int4));
    const size_t o_part = off;
    off += align256((size_t)tot.chunks * (size_t)sf * sizeof(float));
    if (off > kNoAllocScratchBytes)
        return fail(GAT_ERR_WORKSPACE,
                    "gat_fused_layer_no_alloc: this graph's %lld heavy-row chunks need %zu bytes "
                    "of scratch; the static scratch holds %zu (use gat_fused_layer with a plan)",
                    (long long)tot.chunks, off, kNoAllocScratchBytes);

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
    p.qscale = scale * kLog2eNA;
    p.heavy_threshold = kNoAllocThreshold;
    p.chunk_edges = kNoAllocChunk;
    p.n_chunks = tot.chunks;
    p.heavy_rows = reinterpret_cast<int32_t *>(sc + o_rows);
    p.chunk_start = reinterpret_cast<int32_t *>(sc + o_start);
    p.chunk_row = reinterpret_cast<int32_t *>(sc + o_crow);
    p.counters = reinterpret_cast<int32_t *>(sc + o_cnt);
    p.chunk_desc = reinterpret_cast<int4 *>(sc + o_desc);
    p.partials = reinterpret_cast<float *>(sc + o_part);
    p.slot_floats = sf;
    if (tot.heavy > 0) {  // arrival counters start at zero in every call
        e = cudaMemsetAsync(p.counters, 0, (size_t)tot.heavy * 4, s);
        if (e != cudaSuccess) return cuda_fail(e, "gat_fused_layer_no_alloc: clearing counters");
    }
    plan_fill_kernel<<<(unsigned)nb, kPlanThreads, 0, s>>>(row_ptr, n_rows, kNoAllocThreshold, kNoAllocChunk,
                                                 counts + nb, counts + 2 * nb,
                                                 const_cast<int32_t *>(p.heavy_rows),
                                                 const_cast<int32_t *>(p.chunk_start),
                                                 const_cast<int32_t *>(p.chunk_row));
    if ((st = check_launch("gat_fused_layer_no_alloc: plan fill")) != GAT_OK) return st;
    if (tot.heavy > 0) {
        int64_t db = (tot.heavy + kPlanThreads - 1) / kPlanThreads;
        if (db > 4096) db = 4096;
        plan_desc_kernel<<<(unsigned)db, kPlanThreads, 0, s>>>(row_ptr, p.heavy_rows, p.chunk_start,
                                                     tot.heavy, kNoAllocChunk,
                                                     const_cast<int4 *>(p.chunk_desc));
        if ((st = check_launch("gat_fused_layer_no_alloc: chunk descriptors")) != GAT_OK) return st;
    }
    if (dtype == GAT_F32) return dispatch_no_alloc<float>(p, V, LE, s);
    return dispatch_no_alloc<__nv_bfloat16>(p, V, LE, s);
}
