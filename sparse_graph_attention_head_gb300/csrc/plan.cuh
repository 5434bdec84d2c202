// plan.cuh - the plan kernels' tiling, scan record and declarations, shared by
// every translation unit that launches them (gat_plan_create in plan.cu, the
// allocation-free fused layer in no_alloc.cu), so the count, scan and fill
// grids always agree with the kernels' own row tiling and record layout.
#pragma once

#include "common.cuh"

namespace gat {

constexpr int kPlanThreads = 256;  // threads per count / fill block
constexpr int kPlanRounds = 8;     // rows per thread of a count / fill block
constexpr int64_t kPlanRowsPerBlock = (int64_t)kPlanThreads * kPlanRounds;
constexpr int kPlanScanThreads = 1024;  // the single scan block

// Per-block class sizes (count kernel), their exclusive prefix (scan kernel)
// and the grand totals: heavy rows, heavy-row chunks, edges of heavy rows.
struct Counts {
    long long heavy, chunks, edges;
};

// Blocks of the count and fill kernels for n_rows rows.
inline int64_t plan_blocks(int64_t n_rows) {
    return (n_rows + kPlanRowsPerBlock - 1) / kPlanRowsPerBlock;
}

// Launch with plan_blocks(n_rows) blocks of kPlanThreads threads.
__global__ void plan_count_kernel(const int32_t *row_ptr, int64_t n_rows, int32_t T, int32_t C,
                                  Counts *block_counts);
// Launch with one block of kPlanScanThreads threads.
__global__ void plan_scan_kernel(const Counts *block_counts, int64_t nb, Counts *offsets,
                                 Counts *totals);
// Launch with plan_blocks(n_rows) blocks of kPlanThreads threads.
__global__ void plan_fill_kernel(const int32_t *row_ptr, int64_t n_rows, int32_t T, int32_t C,
                                 const Counts *offsets, const Counts *totals,
                                 int32_t *heavy_rows, int32_t *chunk_start, int32_t *chunk_row);
// Grid-stride over heavy rows; any grid of kPlanThreads-thread blocks.
__global__ void plan_desc_kernel(const int32_t *row_ptr, const int32_t *heavy_rows,
                                 const int32_t *chunk_start, int64_t n_heavy, int32_t C,
                                 int4 *desc);

}  // namespace gat
