// Device pieces of the page-major gather plan shared by kv_gather_plan
// (kv_plan.cu, counters in the caller's plan buffer) and
// kv_gather_plan_noalloc (kv_plan_static.cu, counters in a fixed array).
#pragma once

#include "kv_common.cuh"

namespace gtkv {

constexpr int kPlanHeaderWords = 4;  // entries, n_seqs, max_pages, flags
// Bits of the plan's flags word [3].
constexpr int32_t kPlanPageMajor = 1;      // the page-major order pays: walk the plan, not the table
constexpr int32_t kPlanKernelFacing = 2;   // built from a table of kernel-facing entries (phys * 2L)

// Page bucket of block-table entry e = s * max_pages + k, or -1 when the entry
// holds no token of the sequence's window [start_s, len_s). A tombstone
// (negative page) reads the page-0 sink and joins page 0; a page >= P sets
// KV_DEV_ERR_ROW in `bits` and is left out. bt_div > 1: the table holds
// kernel-facing entries phys * bt_div (bt_div = the row-blocks per page);
// one off that grid sets KV_DEV_ERR_FORM and is left out.
__device__ __forceinline__ int64_t plan_bucket(const DevPool& p, int64_t e, const int32_t* __restrict__ bt,
                                               int32_t max_pages, const int32_t* __restrict__ seq_start,
                                               const int32_t* __restrict__ seq_len, int32_t bt_div, int& bits) {
  const int64_t s = e / max_pages;
  const int64_t k = e - s * max_pages;
  int64_t lo = seq_start ? __ldg(seq_start + s) : 0;
  if (lo < 0) lo = 0;
  const int64_t hi = __ldg(seq_len + s);
  if (k * p.ps >= hi || (k + 1) * p.ps <= lo) return -1;
  int64_t page = __ldg(bt + e);
  if (page >= p.num_pages * bt_div) {
    bits |= KV_DEV_ERR_ROW;
    return -1;
  }
  if (page <= 0) return 0;
  if (bt_div != 1) {
    const int64_t phys = page / bt_div;
    if (phys * bt_div != page) {
      bits |= KV_DEV_ERR_FORM;
      return -1;
    }
    page = phys;
  }
  return page;
}

// Scatter step of the counting sort: entry e takes the next position of its
// page's run. The positions come from the count pass over the same table, so
// they stay below n_entries; if the table changed between the passes (a race
// in the caller) a run could overflow, and such a position is dropped with
// KV_DEV_ERR_TABLE instead of being written past the plan.
__device__ __forceinline__ void plan_place(int32_t* __restrict__ entries, int32_t* next, int64_t n_entries, int64_t e,
                                           int& bits) {
  const int32_t pos = atomicAdd(next, 1);
  if (pos >= 0 && pos < n_entries) {
    entries[pos] = static_cast<int32_t>(e);
  } else {
    bits |= KV_DEV_ERR_TABLE;
  }
}

constexpr int kScanThreads = 1024;
constexpr int kScanPer = 4;                              // counters per thread per tile
constexpr int kScanTile = kScanThreads * kScanPer;      // 4096 counters
constexpr int kScanAhead = 4;                            // tiles whose loads are in flight at once

// Exclusive scan of n_pages counters in place, by one block of kScanThreads
// threads: tile after tile of 4096 counters (thread t owns 4 consecutive
// ones), kScanAhead tiles loaded before any is scanned, a running carry
// between tiles. Then counts[n_pages] = total and the plan header: [0] total
// entries, [1] n_seqs, [2] max_pages, [3] flags: kPlanPageMajor when entries
// >= 1.5 x distinct pages (the page-major order pays), plus `form_flag`
// (kPlanKernelFacing or 0).
__device__ __forceinline__ void scan_plan_counts(int32_t* counts, int64_t n_pages, int32_t n_seqs,
                                                 int32_t max_pages, int32_t form_flag, int32_t* __restrict__ plan) {
  __shared__ int32_t warp_sum[kScanThreads / 32];
  __shared__ int32_t pages_used;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  if (t == 0) pages_used = 0;
  __syncthreads();
  int32_t carry = 0, used = 0;
  for (int64_t base = 0; base < n_pages; base += static_cast<int64_t>(kScanTile) * kScanAhead) {
    int32_t v[kScanAhead][kScanPer];
#pragma unroll
    for (int a = 0; a < kScanAhead; ++a)
#pragma unroll
      for (int e = 0; e < kScanPer; ++e) {
        const int64_t i = base + static_cast<int64_t>(a) * kScanTile + t * kScanPer + e;
        v[a][e] = i < n_pages ? counts[i] : 0;
      }
#pragma unroll
    for (int a = 0; a < kScanAhead; ++a) {
      int32_t mine = 0;
#pragma unroll
      for (int e = 0; e < kScanPer; ++e) {
        mine += v[a][e];
        used += v[a][e] > 0;
      }
      int32_t incl = mine;  // inclusive prefix within the warp
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int32_t x = __shfl_up_sync(kFull, incl, d);
        if (lane >= d) incl += x;
      }
      if (lane == 31) warp_sum[warp] = incl;
      __syncthreads();
      if (warp == 0) {
        int32_t w = warp_sum[lane];  // kScanThreads / 32 == 32 warps
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
          const int32_t x = __shfl_up_sync(kFull, w, d);
          if (lane >= d) w += x;
        }
        warp_sum[lane] = w;  // inclusive prefix over warps
      }
      __syncthreads();
      int32_t run = carry + incl - mine + (warp > 0 ? warp_sum[warp - 1] : 0);
      carry += warp_sum[31];
      __syncthreads();  // warp_sum is rewritten by the next tile
#pragma unroll
      for (int e = 0; e < kScanPer; ++e) {
        const int64_t i = base + static_cast<int64_t>(a) * kScanTile + t * kScanPer + e;
        if (i < n_pages) counts[i] = run;
        run += v[a][e];
      }
    }
  }
  if (used) atomicAdd(&pages_used, used);
  __syncthreads();
  if (t == 0) {
    counts[n_pages] = carry;
    plan[0] = carry;
    plan[1] = n_seqs;
    plan[2] = max_pages;
    plan[3] = (2 * static_cast<int64_t>(carry) >= 3 * static_cast<int64_t>(pages_used) ? kPlanPageMajor : 0) |
              form_flag;
  }
}

}  // namespace gtkv
