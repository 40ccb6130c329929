// K4: block-table gather of one layer into packed [rows, H, D] K and V.
// Source: prhub report on sglang PR #34602, 功能与动机 -- with dense per-layer
// views every layer's K/V is read through one contiguous tensor and one shared
// block table -- and build_mha_views' view arithmetic (关键源码片段
// layout/page_major.py): token (page p, offset o) of layer l is K-view row
// p*ps*2L + o + 2l*ps, and its V row follows ps rows later.
//
// Work is split by OUTPUT row, which is what the caller's cu_out packs: a warp
// takes 32 consecutive output rows; lane k finds the sequence of row r0+k by
// binary search over cu_out, turns it into (page, offset) through the block
// table, and the warp then copies the 32 rows, each row's source shared by
// shuffle. Within a page the rows of one sequence are consecutive in the pool
// and in the output, so consecutive row groups touch consecutive memory.
#include "kv_common.cuh"

namespace gtkv {

namespace {

template <int G, int VPL, int U>
__global__ void __launch_bounds__(kBlock) k_gather(DevPool p, int32_t layer, const int32_t* __restrict__ bt,
                                                   int32_t n_seqs, int32_t max_pages,
                                                   const int32_t* __restrict__ seq_start,
                                                   const int32_t* __restrict__ seq_len,
                                                   const int64_t* __restrict__ cu, uint4* __restrict__ out_k,
                                                   uint4* __restrict__ out_v, int64_t out_rows) {
  constexpr int RPW = 32 / G;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t nthreads = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t ps = p.ps;

  // Metadata checks, one sequence per thread (they never gate the copies:
  // every access below is bounds-checked on its own).
  for (int64_t s = tid; s < n_seqs; s += nthreads) {
    const int64_t a = seq_start ? __ldg(seq_start + s) : 0;
    const int64_t b = __ldg(seq_len + s);
    const int64_t c0 = __ldg(cu + s), c1 = __ldg(cu + s + 1);
    if (a < 0 || b > static_cast<int64_t>(max_pages) * ps || c0 < 0 || c1 < c0 || c1 - c0 < b - a)
      atomicOr(p.err, KV_DEV_ERR_TABLE);
  }
  const int64_t cu_end = __ldg(cu + n_seqs);
  if (tid == 0 && cu_end > out_rows) atomicOr(p.err, KV_DEV_ERR_TABLE);
  const int64_t total = cu_end < out_rows ? cu_end : out_rows;
  const int64_t cu0 = __ldg(cu);

  const int lane = threadIdx.x & 31;
  const int g = lane % G;
  const int grp = lane / G;
  const int64_t vpr = VPL > 0 ? static_cast<int64_t>(G) * VPL : p.vpr;
  const int64_t warp = tid >> 5;
  const int64_t nwarps = nthreads >> 5;
  const int64_t koff = 2 * static_cast<int64_t>(layer) * ps;
  const L2Policy pol = make_l2_policy();

  for (int64_t r0 = warp * 32; r0 < total; r0 += nwarps * 32) {
    // lane's output row -> K-view source row (or -1: leave the row alone)
    const int64_t r = r0 + lane;
    long long src_row = -1;
    if (r < total && r >= cu0) {
      int lo = 0, hi = n_seqs;  // cu[lo] <= r < cu[hi] when cu is non-decreasing
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (__ldg(cu + mid) <= r) lo = mid; else hi = mid;
      }
      const int64_t a = seq_start ? __ldg(seq_start + lo) : 0;
      const int64_t j = a + (r - __ldg(cu + lo));
      if (j >= 0 && j < __ldg(seq_len + lo)) {
        const int64_t k = div_ps(p, j);
        int64_t o = j - k * ps;
        if (k < max_pages) {
          int64_t page = __ldg(bt + static_cast<int64_t>(lo) * max_pages + k);
          if (page < 0) {  // tombstoned entry reads the page-0 sink
            page = 0;
            o = 0;
          }
          if (page < p.num_pages) {
            src_row = page * p.stride + o + koff;
          } else {
            atomicOr(p.err, KV_DEV_ERR_ROW);
          }
        }
      }
    }
    const int cnt = static_cast<int>(total - r0 < 32 ? total - r0 : 32);
#pragma unroll 1
    for (int w0 = 0; w0 < cnt; w0 += RPW * U) {
      const uint4* src[2 * U];
      uint4* dst[2 * U];
      bool go[2 * U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int j = w0 + u * RPW + grp;  // row within this batch of 32
        const long long sr = __shfl_sync(kFull, src_row, j & 31);
        const bool ok = j < cnt && sr >= 0;
        const int64_t s_ = ok ? sr : 0;
        const int64_t o_ = ok ? r0 + j : 0;
        go[2 * u] = go[2 * u + 1] = ok;
        src[2 * u] = p.base + s_ * vpr;
        src[2 * u + 1] = p.base + (s_ + ps) * vpr;
        dst[2 * u] = out_k + o_ * vpr;
        dst[2 * u + 1] = out_v + o_ * vpr;
      }
      copy_rows<G, VPL, 2 * U, GTKV_GATHER_LD, GTKV_GATHER_ST>(src, dst, go, g, vpr, pol);
    }
  }
}

}  // namespace

cudaError_t launch_gather(const DevPool& p, int32_t layer, const int32_t* bt, int32_t n_seqs, int32_t max_pages,
                          const int32_t* seq_start, const int32_t* seq_len, const int64_t* cu, void* out_k,
                          void* out_v, int64_t out_rows, int sm_count, cudaStream_t s) {
  return dispatch_row(p.vpr, [&]<int G, int VPL>() -> cudaError_t {
    constexpr int U = VPL == 0 ? 1 : (VPL >= 4 ? 2 : 4 / VPL);
    auto kernel = k_gather<G, VPL, U>;
    // The row count lives on the device (cu_out[n_seqs]); out_rows bounds it.
    int64_t warps = (out_rows + 31) / 32;
    const int64_t seq_warps = (static_cast<int64_t>(n_seqs) + 31) / 32;
    if (warps < seq_warps) warps = seq_warps;
    const unsigned grid = grid_for(kernel, warps, sm_count);
    kernel<<<grid, kBlock, 0, s>>>(p, layer, bt, n_seqs, max_pages, seq_start, seq_len, cu,
                                   static_cast<uint4*>(out_k), static_cast<uint4*>(out_v), out_rows);
    return cudaGetLastError();
  });
}

}  // namespace gtkv
