// Page-major gather plan: the block-table entries of a batch, ordered by the
// page they name.
//
// Many sequences often share pages (common prefixes; in the decode workload
// every page is named by ~16 sequences). A gather that walks the table
// sequence by sequence reads a shared page at ~16 unrelated moments, so L2
// rarely still holds it. Walking the entries page by page instead brings all
// readers of a page together in time: L2 merges their reads and DRAM delivers
// each page about once. The order depends only on the block table, which all
// layers share, so one plan serves every layer's gather of a step.
//
// The plan is a counting sort of the entries by page, in a caller-provided
// buffer (int32 words):
//   [0] number of entries in the plan   [1] n_seqs   [2] max_pages
//   [3] flags: bit 0 (kPlanPageMajor) when the page-major order pays
//       (entries >= 1.5 x distinct pages), clear when pages are hardly shared
//       and the table's own order is better (the output writes stay
//       sequential), and the planned gather follows it; bit 1
//       (kPlanKernelFacing) when the table holds kernel-facing entries
//   [4 .. 4+P]            per-page counts, then start offsets (P + 1 words)
//   [5+P .. 5+P+S*maxp)   entry indices s*max_pages + k, grouped by page
// Only entries whose tokens overlap the sequence's window [start, len) enter
// the plan. A tombstoned entry (negative page) reads the sink on page 0 and
// is grouped with page 0; a page >= P raises KV_DEV_ERR_ROW and is left out.
#include "kv_launch.h"
#include "kv_plan.cuh"

namespace gtkv {

namespace {

__global__ void __launch_bounds__(kBlock) k_plan_count(DevPool p, const int32_t* __restrict__ bt, int64_t n_entries,
                                                       int32_t max_pages, const int32_t* __restrict__ seq_start,
                                                       const int32_t* __restrict__ seq_len, int32_t bt_div,
                                                       int32_t* __restrict__ plan) {
  int32_t* counts = plan + kPlanHeaderWords;
  int bits = 0;
  const int64_t step = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < n_entries; e += step) {
    const int64_t b = plan_bucket(p, e, bt, max_pages, seq_start, seq_len, bt_div, bits);
    if (b >= 0) atomicAdd(counts + b, 1);
  }
  if (bits) atomicOr(p.err, bits);
}

// Counts -> start offsets (in place) and the plan header.
__global__ void __launch_bounds__(kScanThreads) k_plan_scan(int64_t n_buckets, int32_t n_seqs, int32_t max_pages,
                                                            int32_t form_flag, int32_t* __restrict__ plan) {
  scan_plan_counts(plan + kPlanHeaderWords, n_buckets, n_seqs, max_pages, form_flag, plan);
}

__global__ void __launch_bounds__(kBlock) k_plan_scatter(DevPool p, const int32_t* __restrict__ bt,
                                                         int64_t n_entries, int32_t max_pages,
                                                         const int32_t* __restrict__ seq_start,
                                                         const int32_t* __restrict__ seq_len, int32_t bt_div,
                                                         int32_t* __restrict__ plan) {
  int32_t* offs = plan + kPlanHeaderWords;
  int32_t* entries = offs + p.num_pages + 1;
  int bits = 0;
  const int64_t step = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < n_entries; e += step) {
    const int64_t b = plan_bucket(p, e, bt, max_pages, seq_start, seq_len, bt_div, bits);
    if (b >= 0) plan_place(entries, offs + b, n_entries, e, bits);
  }
  // page >= P and off-grid entries were already reported by the count pass;
  // a position past the plan means the table changed under the build
  if (bits & KV_DEV_ERR_TABLE) atomicOr(p.err, KV_DEV_ERR_TABLE);
}

}  // namespace

int64_t plan_words(const DevPool& p, int32_t n_seqs, int32_t max_pages) {
  return kPlanHeaderWords + p.num_pages + 1 + static_cast<int64_t>(n_seqs) * max_pages;
}

cudaError_t launch_gather_plan(const DevPool& p, const int32_t* bt, int32_t n_seqs, int32_t max_pages,
                               const int32_t* seq_start, const int32_t* seq_len, int32_t* plan, bool kernel_facing,
                               int sm_count, cudaStream_t s) {
  const int64_t n_entries = static_cast<int64_t>(n_seqs) * max_pages;
  const int32_t bt_div = kernel_facing ? p.blocks : 1;
  cudaError_t e = cudaMemsetAsync(plan, 0, sizeof(int32_t) * (kPlanHeaderWords + p.num_pages + 1), s);
  if (e != cudaSuccess) return e;
  const unsigned grid = grid_for(k_plan_count, (n_entries + 31) / 32, sm_count);
  k_plan_count<<<grid, kBlock, 0, s>>>(p, bt, n_entries, max_pages, seq_start, seq_len, bt_div, plan);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  k_plan_scan<<<1, kScanThreads, 0, s>>>(p.num_pages, n_seqs, max_pages, kernel_facing ? kPlanKernelFacing : 0,
                                         plan);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  k_plan_scatter<<<grid, kBlock, 0, s>>>(p, bt, n_entries, max_pages, seq_start, seq_len, bt_div, plan);
  return cudaGetLastError();
}

}  // namespace gtkv
