/*
 * gat.h - C ABI of libgat, multi-head graph attention over CSR graphs on
 * NVIDIA GB300 (sm_103a).
 *
 * The operations follow the problem statements of five POPCORNBENCH
 * transcripts, each about replacing a small PyTorch reference model:
 *   [softmax page]   FW-GLM-5-1 l1_p6  - multi-head row-wise softmax over CSR edge scores
 *   [aggregate page] Kimi-K2.6 l2_p37  - CSR softmax + neighbourhood aggregation
 *   [spmm page]      FW-GLM-5-1 l1_p18 - multi-head weighted sparse aggregation
 *   [block page]     Kimi-K2.6 l2_p4   - scene-graph relation attention block
 *   [sddmm page]     FW-GLM-5-1 l1_p10 - edge-only SDDMM (gathered dot product)
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Graphs: row_ptr is int32 [n_rows + 1], non-decreasing, row_ptr[0] = 0,
 *   row_ptr[n_rows] = n_edges; row i owns edges [row_ptr[i], row_ptr[i+1]).
 *   col_idx is int32 [n_edges] with 0 <= col_idx[e] < n_src. Row i is the
 *   destination, col_idx[e] the source of edge e. Duplicate edges are allowed
 *   and count separately; col_idx need not be sorted.
 * - Per-edge tensors are [n_edges, H] row-major (heads contiguous per edge).
 *   Node tensors are [n, H, Dh] row-major. Offsets are computed in 64 bits.
 * - Every data pointer is DEVICE memory owned by the caller, aligned to at
 *   least its element size. 16-byte aligned pointers with 16-byte rows per
 *   head (Dh * element size a multiple of 16) take the vectorised kernels;
 *   other layouts take a scalar kernel with the same semantics.
 * - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *   stream). Every call only enqueues work on it and returns; results are
 *   ready when the stream reaches that point. Calls never synchronise the
 *   device, except gat_plan_create, which does (see there).
 * - No entry point allocates device memory except gat_plan_create.
 * - Errors: arguments the host can check (NULL pointers, negative sizes,
 *   unsupported shapes, a plan built for another graph shape, a too-small
 *   workspace) return an error code before anything is launched. A failed
 *   launch returns GAT_ERR_CUDA; gat_last_error() then describes it. Device
 *   contents of row_ptr/col_idx are NOT checked by the compute calls: an index
 *   out of range is undefined behaviour there; call gat_validate_graph first
 *   when the graph is untrusted.
 * - Results are deterministic: no floating-point atomics; every reduction
 *   runs in a fixed order, so repeated calls give bitwise-identical outputs.
 * - Thread safety: calls on different streams may run concurrently, except
 *   that one plan must not be used by two calls whose work overlaps on the
 *   GPU: it holds per-row arrival counters and a work counter that the calls
 *   taking a plan update and reset (order such calls on one stream, or give
 *   each stream its own plan).
 */
#ifndef GAT_H
#define GAT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GAT_OK = 0,
    GAT_ERR_INVALID_ARG = 1,        /* NULL pointer, negative size, inconsistent sizes */
    GAT_ERR_UNSUPPORTED = 2,        /* shape or dtype this build does not implement */
    GAT_ERR_CUDA = 3,               /* a CUDA runtime call or kernel launch failed */
    GAT_ERR_WORKSPACE = 4,          /* workspace missing or too small */
    GAT_ERR_INDEX_OUT_OF_RANGE = 5, /* gat_validate_graph found a bad row_ptr/col_idx */
    GAT_ERR_PLAN_MISMATCH = 6       /* plan built for a different n_rows / n_edges */
} gat_status_t;

typedef enum {
    GAT_F32 = 0, /* IEEE binary32 */
    GAT_BF16 = 1 /* bfloat16; arithmetic is fp32, results rounded to nearest even */
} gat_dtype_t;

/* Opaque degree-bucket plan; owns a few device arrays (see gat_plan_create). */
typedef struct gat_plan_s *gat_plan_t;

/* Human-readable name of a status code (static storage). */
const char *gat_status_string(gat_status_t status);

/* Detail of the last error returned on the calling host thread (thread-local
 * storage, valid until the next call on that thread). */
const char *gat_last_error(void);

/* Library version as 10000*major + 100*minor + patch. */
int32_t gat_version(void);

/* ------------------------------------------------------------------------
 * Degree-bucket plan
 *
 * The pages assign one thread, warp or block to a destination row; that
 * choice is a load-balance question on a power-law graph. The plan sorts rows
 * into two classes once per graph and is reused by every call on that graph:
 *   light rows  deg <= heavy_threshold: one warp per row
 *   heavy rows  deg >  heavy_threshold: cut into chunks of chunk_edges edges;
 *               gat_fused_layer runs one warp per chunk and merges the chunks'
 *               softmax states; gat_spmm_weighted does the same with
 *               partial sums when given a workspace (else one thread block
 *               per heavy row); gat_edge_softmax runs one thread block per
 *               heavy row.
 * Plan arrays (device, int32):
 *   heavy_rows  [n_heavy]     ascending row ids with deg > heavy_threshold
 *   chunk_start [n_heavy + 1] exclusive prefix sum of ceil(deg / chunk_edges)
 *   chunk_row   [n_chunks]    index into heavy_rows of each chunk's row
 * Chunk c of heavy_rows[r] covers edges [row_ptr[row] + j*chunk_edges,
 * min(row_ptr[row] + (j+1)*chunk_edges, row_ptr[row+1])), j = c - chunk_start[r].
 * ---------------------------------------------------------------------- */

/* Build a plan for the graph `row_ptr` (device, [n_rows+1]).
 * heavy_threshold <= 0 and chunk_edges <= 0 select the defaults (128, 256).
 * Allocates the plan's device arrays (cudaMalloc), runs four small kernels on
 * `stream` and synchronises `stream` once to read the class sizes back.
 * Errors: GAT_ERR_INVALID_ARG (NULL row_ptr/plan, n_rows < 0, n_edges < 0),
 * GAT_ERR_CUDA (allocation or launch failure; *plan is then NULL). */
gat_status_t gat_plan_create(const int32_t *row_ptr, int64_t n_rows, int64_t n_edges,
                             int32_t heavy_threshold, int32_t chunk_edges, void *stream,
                             gat_plan_t *plan);

/* Free a plan and its device arrays (NULL is accepted). The caller must make
 * sure no enqueued work still uses it. */
gat_status_t gat_plan_destroy(gat_plan_t plan);

/* Sizes and parameters of a plan; any output pointer may be NULL. */
gat_status_t gat_plan_info(gat_plan_t plan, int64_t *n_rows, int64_t *n_edges,
                           int32_t *heavy_threshold, int32_t *chunk_edges,
                           int64_t *n_heavy, int64_t *n_chunks);

/* Copy the plan arrays into caller device buffers of sizes n_heavy,
 * n_heavy + 1 and n_chunks (any pointer may be NULL to skip that array).
 * Enqueued on `stream`. */
gat_status_t gat_plan_export(gat_plan_t plan, int32_t *heavy_rows, int32_t *chunk_start,
                             int32_t *chunk_row, void *stream);

/* ------------------------------------------------------------------------
 * Graph validation (optional, for untrusted graphs)
 *
 * Checks on the device that row_ptr[0] == 0, row_ptr is non-decreasing,
 * row_ptr[n_rows] == n_edges and 0 <= col_idx[e] < n_src (col_idx may be NULL
 * to skip that check). Synchronises `stream`. Returns GAT_OK or
 * GAT_ERR_INDEX_OUT_OF_RANGE; never traps. `flag` is caller device scratch of
 * one int32 (its content is overwritten).
 * ---------------------------------------------------------------------- */
gat_status_t gat_validate_graph(const int32_t *row_ptr, const int32_t *col_idx,
                                int64_t n_rows, int64_t n_src, int64_t n_edges,
                                int32_t *flag, void *stream);

/* ------------------------------------------------------------------------
 * Row shards (one process per GPU). Rows are independent in every operation
 * here [softmax page, reference model: a softmax per node's own edge range;
 * spmm page: one output row per destination], so a graph splits into
 * contiguous row ranges that different GPUs compute alone, each needing the
 * source rows its edges read (all of k / v for uniform sources).
 *
 * gat_partition_rows: HOST function (no GPU work, row_ptr in host memory):
 * cuts rows [0, n_rows) into `parts` contiguous ranges
 * [row_begin[p], row_begin[p+1]) of about equal weight, the weight of a row
 * being 1 + its degree (its q and out rows and one gathered source row per
 * edge: the fused layer's traffic). row_begin has parts + 1 entries,
 * row_begin[0] = 0, row_begin[parts] = n_rows, non-decreasing (a part may be
 * empty). Deterministic. Errors: GAT_ERR_INVALID_ARG, and
 * GAT_ERR_INDEX_OUT_OF_RANGE for a decreasing row_ptr.
 *
 * gat_rebase_row_ptr: out[i] = row_ptr[r0 + i] - row_ptr[r0] for
 * i in [0, r1 - r0] (device arrays, enqueued on `stream`): the row pointer of
 * rows [r0, r1) as a graph of its own, whose edges are col_idx + row_ptr[r0],
 * queries q + r0 * H * Dh and outputs out + r0 * H * Dh. Errors:
 * GAT_ERR_INVALID_ARG, GAT_ERR_CUDA.
 * ---------------------------------------------------------------------- */
gat_status_t gat_partition_rows(const int32_t *row_ptr, int64_t n_rows, int32_t parts,
                                int64_t *row_begin);

gat_status_t gat_rebase_row_ptr(const int32_t *row_ptr, int64_t r0, int64_t r1, int32_t *out,
                                void *stream);

/* ------------------------------------------------------------------------
 * SDDMM [sddmm page, reference model: gather both endpoint feature rows of
 * every edge, multiply elementwise, sum over the feature dimension],
 * generalised to heads and a scale:
 *     out[e,h] = scale * sum_{d<Dh} src_feat[src(e),h,d] * dst_feat[dst(e),h,d]
 * COO form (row_ptr == NULL): src(e) = src_idx[e], dst(e) = dst_idx[e],
 *   n_rows is ignored.
 * CSR form (row_ptr != NULL): dst(e) = the row that owns e, src(e) = src_idx[e]
 *   (the column index); dst_idx is ignored and n_dst must be >= n_rows.
 * src_feat [n_src,H,Dh] and dst_feat [n_dst,H,Dh] share `dtype`; out is fp32
 * [n_edges,H]. n_edges == 0 is a no-op.
 * Errors: GAT_ERR_INVALID_ARG for NULL pointers (with n_edges > 0), negative
 * sizes, H < 1 or Dh < 1; GAT_ERR_UNSUPPORTED for an unknown dtype.
 * ---------------------------------------------------------------------- */
gat_status_t gat_sddmm(const int32_t *row_ptr, const int32_t *src_idx, const int32_t *dst_idx,
                       int64_t n_rows, int64_t n_edges, const void *src_feat, int64_t n_src,
                       const void *dst_feat, int64_t n_dst, int32_t H, int32_t Dh, float scale,
                       gat_dtype_t dtype, float *out, void *stream);

/* ------------------------------------------------------------------------
 * Segmented edge softmax [softmax page, reference model: for every node,
 * softmax over that node's CSR edge range, independently per head]:
 *     out[e,h] = exp(s[e,h] - m) / sum_{e' in row} exp(s[e',h] - m),
 *     m = max_{e' in row} s[e',h]
 * scores/out are fp32 [n_edges,H]; out may alias scores (in place). Rows of
 * degree 0 own no entries and write nothing. A row whose scores are all -inf
 * yields NaN, as the reference softmax does. `plan` may be NULL (every row is
 * handled by one warp) or a plan of this graph (heavy rows get a thread block,
 * and warps fetch batches of rows from the plan's work counter, so the plan
 * must not be in use by another call at the same time).
 * Errors: GAT_ERR_INVALID_ARG, GAT_ERR_PLAN_MISMATCH.
 * ---------------------------------------------------------------------- */
gat_status_t gat_edge_softmax(const int32_t *row_ptr, int64_t n_rows, int64_t n_edges, int32_t H,
                              const float *scores, float *out, gat_plan_t plan, void *stream);

/* ------------------------------------------------------------------------
 * Weighted SpMM [spmm page, reference model: each destination sums the
 * per-edge, per-head weight times the source node's feature row;
 * aggregate page: a zero-degree destination stays zero]:
 *     out[i,h,d] = sum_{e in row i} w[e,h] * feat[col_idx[e],h,d]
 * w is fp32 [n_edges,H]; feat [n_src,H,Dh] and out [n_rows,H,Dh] share
 * `dtype` (fp32 accumulation). Zero-degree rows are written as zeros.
 * The aggregate page's operation (softmax of per-edge scores, then this sum)
 * is gat_edge_softmax followed by gat_spmm_weighted with H = 1.
 * plan: NULL (every row by one warp) or a plan of this graph. With a plan,
 * heavy rows are cut into chunks whose partial sums go to `workspace` (at
 * least gat_spmm_weighted_workspace_size bytes, 16-byte aligned) and are
 * added in chunk order by the chunk that finishes last, all in one launch;
 * with workspace NULL each heavy row takes one thread block in a second
 * launch instead. The plan's arrival counters are used in the first form
 * (one plan must not serve two such calls whose work overlaps on the GPU).
 * Errors: GAT_ERR_INVALID_ARG, GAT_ERR_UNSUPPORTED, GAT_ERR_PLAN_MISMATCH,
 * GAT_ERR_WORKSPACE (a workspace given but too small or misaligned).
 * ---------------------------------------------------------------------- */
gat_status_t gat_spmm_weighted_workspace_size(gat_plan_t plan, int32_t H, int32_t Dh,
                                              size_t *bytes);

gat_status_t gat_spmm_weighted(const int32_t *row_ptr, const int32_t *col_idx, int64_t n_rows,
                               int64_t n_src, int64_t n_edges, int32_t H, int32_t Dh,
                               const float *w, const void *feat, gat_dtype_t dtype, void *out,
                               gat_plan_t plan, void *workspace, size_t workspace_bytes,
                               void *stream);

/* ------------------------------------------------------------------------
 * Softmax + neighbourhood aggregation in one pass [aggregate page, reference
 * model: a softmax over each destination's edge scores, then the
 * softmax-weighted sum of the source rows; a zero-degree destination stays
 * zero]:
 *     out[i,h,:] = sum_{e in row i} softmax_e(scores[.,h])[e] * feat[col_idx[e],h,:]
 * scores fp32 [n_edges,H] (given, not computed); feat [n_src,H,Dh] and out
 * [n_rows,H,Dh] share `dtype` (fp32 arithmetic). One launch (per group of
 * heads the vector engine takes) with an online softmax: no weight reaches
 * memory. Same plan / workspace rules as gat_fused_layer (size from
 * gat_fused_layer_workspace_size). Needs 16-byte aligned feat / out and a
 * vector-engine shape (Dh * element size a multiple of 16 with Dh / (16 /
 * element size) a power of two); else GAT_ERR_UNSUPPORTED (compose
 * gat_edge_softmax and gat_spmm_weighted instead). A non-empty row whose
 * scores are all -inf for a head gives NaN for that head, as the softmax of
 * the composition does; a zero-degree row gives zeros.
 * Errors: GAT_ERR_INVALID_ARG, GAT_ERR_UNSUPPORTED, GAT_ERR_PLAN_MISMATCH,
 * GAT_ERR_WORKSPACE.
 * ---------------------------------------------------------------------- */
gat_status_t gat_softmax_aggregate(const int32_t *row_ptr, const int32_t *col_idx,
                                   int64_t n_rows, int64_t n_src, int64_t n_edges, int32_t H,
                                   int32_t Dh, const float *scores, const void *feat,
                                   gat_dtype_t dtype, void *out, gat_plan_t plan, void *workspace,
                                   size_t workspace_bytes, void *stream);

/* ------------------------------------------------------------------------
 * Fused multi-head graph-attention layer: SDDMM -> segmented softmax ->
 * weighted SpMM in one pass (the composition of the sddmm, softmax and spmm
 * pages' operations), with the softmax kept online so no score or weight
 * ever reaches memory:
 *     s[e,h]     = scale * sum_d q[i,h,d] * k[col_idx[e],h,d]
 *     out[i,h,:] = sum_e softmax_e(s[.,h])[e] * v[col_idx[e],h,:]
 *     out[i,:,:] = 0 for a zero-degree row i
 * q/out are [n_rows,H,Dh], k/v are [n_src,H,Dh], all in `dtype` (fp32
 * arithmetic, bf16 results rounded to nearest even). Shapes the vector
 * kernel does not take whole run as groups of heads it takes (one launch
 * per group); shapes with no such group take a scalar kernel (no chunks).
 * plan: NULL (every row by one warp; workspace unused) or a plan of this
 * graph (heavy rows split into chunks whose partial softmax states go to
 * `workspace` and are merged by the last chunk to finish).
 * workspace: caller device memory, 16-byte aligned, at least the size
 * reported by gat_fused_layer_workspace_size (may be NULL when that is 0).
 * Errors: GAT_ERR_INVALID_ARG, GAT_ERR_UNSUPPORTED, GAT_ERR_PLAN_MISMATCH,
 * GAT_ERR_WORKSPACE.
 * ---------------------------------------------------------------------- */
gat_status_t gat_fused_layer_workspace_size(gat_plan_t plan, int32_t H, int32_t Dh,
                                            size_t *bytes);

gat_status_t gat_fused_layer(const int32_t *row_ptr, const int32_t *col_idx, int64_t n_rows,
                             int64_t n_src, int64_t n_edges, int32_t H, int32_t Dh, float scale,
                             const void *q, const void *k, const void *v, gat_dtype_t dtype,
                             void *out, gat_plan_t plan, void *workspace, size_t workspace_bytes,
                             void *stream);

/* ------------------------------------------------------------------------
 * fp8 feature tables. In gat_fused_layer the gathers of the k and v rows are
 * nearly all of the bytes [softmax, sddmm and spmm pages, reference models:
 * every edge reads its source's rows]; stored as E4M3 with one fp32 scale per
 * (node, head), a bf16 row of H*Dh elements shrinks from 2*H*Dh to
 * H*Dh + 4*H bytes.
 *
 * gat_quantize_fp8: x [n,H,Dh] (dtype) -> codes [n,H,Dh] (uint8, E4M3: 1 sign,
 * 4 exponent bits with bias 7, 3 mantissa bits, largest finite 448) and
 * scales [n,H] (fp32): scale = max_d |x[i,h,d]| / 448 (1 for an all-zero
 * head), code = E4M3(x / scale) rounded to nearest even and saturating at
 * +-448 (both divisions in fp32). Errors: GAT_ERR_INVALID_ARG, _UNSUPPORTED.
 *
 * gat_fused_layer_fp8: gat_fused_layer with
 *     k[j,h,:] = E4M3(k8[j,h,:]) * k_scale[j,h],  v likewise,
 * q and out [n_rows,H,Dh] in `dtype`, fp32 arithmetic. Same plan and
 * workspace rules as gat_fused_layer (size from
 * gat_fused_layer_workspace_size). The vector kernel takes H*Dh of 512 or
 * 1024 with Dh a power-of-two multiple of 16 and 16-byte aligned pointers,
 * wider rows as groups of heads of that size (one launch per group); other
 * shapes (Dh <= 256) take a scalar kernel (no chunks, workspace unused). Errors: as gat_fused_layer; GAT_ERR_UNSUPPORTED for Dh > 256.
 * ---------------------------------------------------------------------- */
gat_status_t gat_quantize_fp8(const void *x, gat_dtype_t dtype, int64_t n, int32_t H, int32_t Dh,
                              uint8_t *codes, float *scales, void *stream);

gat_status_t gat_fused_layer_fp8(const int32_t *row_ptr, const int32_t *col_idx, int64_t n_rows,
                                 int64_t n_src, int64_t n_edges, int32_t H, int32_t Dh,
                                 float scale, const void *q, gat_dtype_t dtype, const uint8_t *k8,
                                 const float *k_scale, const uint8_t *v8, const float *v_scale,
                                 void *out, gat_plan_t plan, void *workspace,
                                 size_t workspace_bytes, void *stream);

/* ------------------------------------------------------------------------
 * Transposed (source-major) view of a graph, for the backward pass
 * [sddmm page, discussion of the backward pass: an edge's gradients land on
 * the feature rows of its endpoints, and a row shared by several edges
 * collects several contributions; the page adds them with atomics].
 * gat_transpose_create lists, for every source node j, the edges that read j
 * (col_idx[e] == j) in increasing edge order, so per-source sums run in a
 * fixed order without floating-point atomics:
 *   src_ptr [n_src + 1]  group offsets (exclusive prefix sum of the number
 *                        of edges reading each source)
 *   perm    [n_edges]    edge ids, group after group
 *   dst     [n_edges]    the row that owns edge perm[k]
 * plus a degree plan over src_ptr (sources read by more than 128 edges are
 * summed by one thread block each).
 * Allocates its device arrays and temporary scratch (cudaMalloc), runs a few
 * kernels on `stream` and synchronises it (three times). row_ptr must be a
 * valid row pointer array (see gat_validate_graph).
 * Errors: GAT_ERR_INVALID_ARG (NULL output / pointers, negative or too large
 * sizes), GAT_ERR_INDEX_OUT_OF_RANGE (a col_idx entry outside [0, n_src);
 * nothing is built), GAT_ERR_CUDA.
 * ---------------------------------------------------------------------- */
typedef struct gat_transpose_s *gat_transpose_t;

gat_status_t gat_transpose_create(const int32_t *row_ptr, const int32_t *col_idx,
                                  int64_t n_rows, int64_t n_src, int64_t n_edges, void *stream,
                                  gat_transpose_t *transpose);

/* Free a transpose (NULL is accepted); no enqueued work may still use it. */
gat_status_t gat_transpose_destroy(gat_transpose_t transpose);

/* Sizes of a transpose; any output pointer may be NULL. max_src_degree is
 * the largest number of edges reading one source; n_heavy_src the number of
 * sources its degree plan treats as heavy. */
gat_status_t gat_transpose_info(gat_transpose_t transpose, int64_t *n_rows, int64_t *n_src,
                                int64_t *n_edges, int32_t *max_src_degree, int64_t *n_heavy_src);

/* Copy src_ptr [n_src+1], perm [n_edges] and dst [n_edges] into caller device
 * buffers (any pointer may be NULL to skip that array); enqueued on `stream`. */
gat_status_t gat_transpose_export(gat_transpose_t transpose, int32_t *src_ptr, int32_t *perm,
                                  int32_t *dst, void *stream);

/* ------------------------------------------------------------------------
 * Backward of gat_fused_layer: the chain rule through its score, softmax and
 * aggregation. With a[e] the softmax weights of the forward and dout
 * [n_rows,H,Dh] the gradient of the loss with respect to out, for every row
 * i, head h and edge e of the row (source j = col_idx[e]):
 *     da[e]   = <dout[i,h,:], v[j,h,:]>
 *     Delta   = sum_e a[e] da[e]                (over the row's edges)
 *     ds[e]   = a[e] (da[e] - Delta)
 *     dq[i,h] = scale * sum_e ds[e] k[j,h,:]                    [n_rows,H,Dh]
 *     dk[j,h] = scale * sum over edges e reading j of ds[e] q[i(e),h,:]
 *     dv[j,h] = sum over edges e reading j of a[e] dout[i(e),h,:]  [n_src,H,Dh]
 * A zero-degree row gets dq = 0; a source no edge reads gets dk = dv = 0.
 * q, k, v, dout, dq, dk, dv share `dtype` (fp32 arithmetic, bf16 results
 * rounded to nearest even); the forward's output is not needed (the scores
 * and weights are recomputed).
 * Two passes: over the rows (CSR; recomputes each edge's score and da, writes
 * them and each row's log-sum-exp and Delta into the workspace, and dq) and
 * over the sources of `transpose` (sums dk, dv per source in edge order).
 * Results are bitwise repeatable.
 * plan: NULL or the forward plan of this graph (its heavy rows are cut into
 * chunks whose partial states go to the workspace and are merged by the last
 * chunk to finish; the plan's arrival counters are used, so one plan must not
 * serve two calls whose work overlaps on the GPU). transpose: required, from
 * gat_transpose_create on the same graph.
 * workspace: caller device memory, 16-byte aligned, at least the size that
 * gat_fused_layer_backward_workspace_size reports for the same plan and
 * shape (8 * n_edges * H + 8 * n_rows * H bytes plus the chunk states, each
 * part rounded up to 256 bytes); contents on entry are ignored.
 * Errors: GAT_ERR_INVALID_ARG (NULL pointers, bad sizes, no transpose),
 * GAT_ERR_UNSUPPORTED (dtype), GAT_ERR_PLAN_MISMATCH (plan or transpose of
 * another graph shape), GAT_ERR_WORKSPACE.
 * ---------------------------------------------------------------------- */
gat_status_t gat_fused_layer_backward_workspace_size(gat_plan_t plan, int64_t n_rows,
                                                     int64_t n_edges, int32_t H, int32_t Dh,
                                                     size_t *bytes);

gat_status_t gat_fused_layer_backward(const int32_t *row_ptr, const int32_t *col_idx,
                                      int64_t n_rows, int64_t n_src, int64_t n_edges, int32_t H,
                                      int32_t Dh, float scale, const void *q, const void *k,
                                      const void *v, const void *dout, gat_dtype_t dtype,
                                      void *dq, void *dk, void *dv, gat_plan_t plan,
                                      gat_transpose_t transpose, void *workspace,
                                      size_t workspace_bytes, void *stream);

/* ------------------------------------------------------------------------
 * Fused layer without any device allocation. The source pages have no
 * counterpart: this is a deployment variant of gat_fused_layer for callers
 * that cannot call cudaMalloc (a framework that owns all device memory
 * through its own pool, an allocator or memory-pressure callback, a process
 * whose allocation budget is spent, an embedding that only hands over the
 * input and output buffers). Same operation, arguments and results as
 * gat_fused_layer with a default plan (heavy rows: degree > 64, chunks of 64
 * edges); q, k, v, out must be 16-byte aligned and (H, Dh) a shape of the
 * vector engine (else GAT_ERR_UNSUPPORTED).
 * Scratch: the plan, the arrival counters and the chunk softmax states live
 * in one static 32 MiB device array inside the library, which every GPU that
 * loads the library holds until the process exits. A graph whose plan and
 * chunk states do not fit returns GAT_ERR_WORKSPACE before any layer work is
 * enqueued (use gat_fused_layer with a plan and a workspace instead).
 * The array is shared by all calls and keeps the previous call's contents
 * (each call clears what must start at zero); calls whose work overlaps on
 * the GPU race on it and must be serialised by the caller.
 * The first call on a device looks up the array's device address (once per
 * device, with that device current). Every call copies the plan's size back
 * to the host and synchronises `stream` to read it, so this entry point
 * cannot be used inside stream capture at all (not even after a first
 * uncaptured call); call it on an uncaptured stream.
 * ---------------------------------------------------------------------- */
gat_status_t gat_fused_layer_no_alloc(const int32_t *row_ptr, const int32_t *col_idx,
                                      int64_t n_rows, int64_t n_src, int64_t n_edges, int32_t H,
                                      int32_t Dh, float scale, const void *q, const void *k,
                                      const void *v, gat_dtype_t dtype, void *out, void *stream);

/* ------------------------------------------------------------------------
 * Dense-masked small-graph attention block [block page, reference model],
 * all fp32, per graph b of B:
 *     xn    = LayerNorm(x; ln_w, ln_b, ln_eps)      biased variance, per node
 *     Q,K,V = xn Wq^T, xn Wk^T, xn Wv^T             Wq/Wk/Wv [D,D] (out x in), no bias
 *     r     = W2 SiLU(W1 pair[i,j] + b1) + b2       W1 [P,P], b1 [P], W2 [H,P], b2 [H]
 *     logit = Q_i^h . K_j^h / sqrt(D/H) + r[h];  -inf where edge_mask[i,j] < 0.5
 *     ctx   = softmax_j(logit) V^h                  (an all -inf row gives NaN)
 *     out   = x + ctx Wout^T                        Wout [D,D], no bias
 * nodes/out [B,N,D], pair_feats [B,N,N,P], edge_mask [B,N,N] (float 0/1).
 * Head h owns feature dims [h*D/H, (h+1)*D/H). out must not alias nodes.
 * Supported: 1 <= N <= 32, D % H == 0, D/H <= 32, D <= 128, D % 4 == 0,
 * 1 <= P <= 32, 16-byte aligned nodes, out and weight matrices; else
 * GAT_ERR_UNSUPPORTED.
 * The block page's module shape (P = 16, H = 4, D = 96, N <= 24, 16-byte
 * aligned pair_feats) runs on the tensor cores: its weights are first split
 * into scaled fp16 halves in `workspace` (caller device memory, 16-byte
 * aligned, at least gat_dense_masked_attention_workspace_size bytes; its
 * contents on entry are ignored), then one kernel computes the block (fp32
 * accuracy from three fp16 products per product, see the kernel). That
 * kernel evaluates the relation MLP for unmasked pairs only: the features
 * of a pair whose edge_mask is < 0.5 are never read (its logit is -inf
 * whatever they hold, NaN included). Other shapes run a SIMT kernel and
 * take no workspace (NULL allowed).
 * The tensor-core kernel never traps: a wait on its pipeline that gives up
 * (never expected) sets a flag in the workspace and the affected outputs are
 * NaN; gat_dense_masked_attention_status turns that flag into a status.
 * Concurrent calls must use different workspaces.
 * Errors: GAT_ERR_INVALID_ARG, GAT_ERR_UNSUPPORTED, GAT_ERR_WORKSPACE (the
 * tensor-core shape with a missing, small or misaligned workspace).
 * ---------------------------------------------------------------------- */
gat_status_t gat_dense_masked_attention_workspace_size(int32_t N, int32_t D, int32_t H,
                                                       int32_t P, size_t *bytes);

gat_status_t gat_dense_masked_attention(int32_t B, int32_t N, int32_t D, int32_t H, int32_t P,
                                        const float *nodes, const float *pair_feats,
                                        const float *edge_mask, const float *ln_w,
                                        const float *ln_b, float ln_eps, const float *Wq,
                                        const float *Wk, const float *Wv, const float *W1,
                                        const float *b1, const float *W2, const float *b2,
                                        const float *Wout, float *out, void *workspace,
                                        size_t workspace_bytes, void *stream);

/* Synchronise `stream` and report whether the last tensor-core call that used
 * `workspace` completed its pipeline: GAT_OK, or GAT_ERR_CUDA when one of its
 * bounded waits gave up (its outputs were then written as NaN). */
gat_status_t gat_dense_masked_attention_status(const void *workspace, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* GAT_H */
