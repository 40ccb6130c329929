// K4: block-table gather of one layer into packed [rows, H, D] K and V.
// Source: prhub report on sglang PR #34602, 功能与动机 -- with dense per-layer
// views every layer's K/V is read through one contiguous tensor and one shared
// block table -- and build_mha_views' view arithmetic (关键源码片段
// layout/page_major.py): token (page p, offset o) of layer l is K-view row
// p*ps*2L + o + 2l*ps, and its V row follows ps rows later.
//
// The block table is the work list. Entry (s, k) covers tokens
// [k*ps, (k+1)*ps) of sequence s; clipped to the window [start_s, len_s) it is
// a run of consecutive pool rows (one page's block 2l, then the same run in
// block 2l+1 for V) that lands on consecutive output rows cu_out[s] + j -
// start_s. So the gather is a set of contiguous copies: each run is cut into
// chunks of about 4 KiB, a warp takes one chunk at a time and copies its K
// and V bytes as 16-byte vectors, all loads issued before the stores. No
// search and no host synchronization: the item space is n_seqs x max_pages x
// chunks_per_page, and an entry outside a sequence's window is an empty item.
#include "kv_common.cuh"

namespace gtkv {

namespace {

#ifndef GTKV_GATHER_CHUNK
#define GTKV_GATHER_CHUNK 4096  // bytes of K (and of V) one warp copies per item
#endif

// Items = (sequence s, table entry k, chunk c). CHV 16-byte vectors per lane
// per round: one round moves 32*CHV vectors of K and as many of V.
template <int CHV>
__global__ void __launch_bounds__(kBlock) k_gather_runs(DevPool p, int32_t layer, const int32_t* __restrict__ bt,
                                                        int32_t n_seqs, int32_t max_pages,
                                                        const int32_t* __restrict__ seq_start,
                                                        const int32_t* __restrict__ seq_len,
                                                        const int64_t* __restrict__ cu, uint4* __restrict__ out_k,
                                                        uint4* __restrict__ out_v, int64_t out_rows,
                                                        int32_t chunk_rows, int32_t chunks_per_page) {
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
  if (tid == 0 && __ldg(cu + n_seqs) > out_rows) atomicOr(p.err, KV_DEV_ERR_TABLE);

  const int lane = threadIdx.x & 31;
  const int64_t vpr = p.vpr;
  const int64_t koff = 2 * static_cast<int64_t>(layer) * ps;
  const int64_t n_items = static_cast<int64_t>(n_seqs) * max_pages * chunks_per_page;
  const L2Policy pol = make_l2_policy();

  for (int64_t it = tid >> 5; it < n_items; it += nthreads >> 5) {
    const int64_t sk = it / chunks_per_page;  // block-table entry index s*max_pages + k
    const int64_t c = it - sk * chunks_per_page;
    const int64_t s = sk / max_pages;
    const int64_t k = sk - s * max_pages;
    const int64_t a = seq_start ? __ldg(seq_start + s) : 0;
    const int64_t b = __ldg(seq_len + s);
    const int64_t j0 = k * ps + c * chunk_rows;  // first token of this chunk
    int64_t jlo = j0 > a ? j0 : a;
    if (jlo < 0) jlo = 0;
    int64_t jhi = j0 + chunk_rows;
    if (jhi > (k + 1) * ps) jhi = (k + 1) * ps;
    if (jhi > b) jhi = b;
    if (jlo >= jhi) continue;  // entry outside the window: empty item
    int64_t page = __ldg(bt + sk);
    if (page >= p.num_pages) {
      if (lane == 0) atomicOr(p.err, KV_DEV_ERR_ROW);
      continue;
    }
    const int64_t cs = __ldg(cu + s);
    int64_t rlo = cs + (jlo - a);
    int64_t rhi = cs + (jhi - a);
    if (rlo < 0) {  // rows before 0 are never written (cu_out[s] < 0 is flagged)
      jlo -= rlo;
      rlo = 0;
    }
    if (rhi > out_rows) rhi = out_rows;
    if (rlo >= rhi) continue;
    const int64_t nvec = (rhi - rlo) * vpr;
    uint4* dk = out_k + rlo * vpr;
    uint4* dv = out_v + rlo * vpr;
    if (page >= 0) {
      const uint4* srck = p.base + (page * p.stride + koff + (jlo - k * ps)) * vpr;
      const uint4* srcv = srck + ps * vpr;
      for (int64_t v0 = 0; v0 < nvec; v0 += 32 * CHV) {
        uint4 bk[CHV], bv[CHV];
#pragma unroll
        for (int i = 0; i < CHV; ++i) {
          const int64_t v = v0 + lane + 32 * i;
          if (v < nvec) {
            bk[i] = ld16<GTKV_GATHER_LD>(srck + v, pol);
            bv[i] = ld16<GTKV_GATHER_LD>(srcv + v, pol);
          }
        }
#pragma unroll
        for (int i = 0; i < CHV; ++i) {
          const int64_t v = v0 + lane + 32 * i;
          if (v < nvec) {
            st16<GTKV_GATHER_ST>(dk + v, bk[i], pol);
            st16<GTKV_GATHER_ST>(dv + v, bv[i], pol);
          }
        }
      }
    } else {  // tombstoned entry: every token of the run reads the page-0 sink row
      const uint4* srck = p.base + koff * vpr;
      const uint4* srcv = srck + ps * vpr;
      for (int64_t v = lane; v < nvec; v += 32) {
        const int64_t col = v % vpr;
        st16<GTKV_GATHER_ST>(dk + v, ld16<GTKV_GATHER_LD>(srck + col, pol), pol);
        st16<GTKV_GATHER_ST>(dv + v, ld16<GTKV_GATHER_LD>(srcv + col, pol), pol);
      }
    }
  }
}

}  // namespace

cudaError_t launch_gather(const DevPool& p, int32_t layer, const int32_t* bt, int32_t n_seqs, int32_t max_pages,
                          const int32_t* seq_start, const int32_t* seq_len, const int64_t* cu, void* out_k,
                          void* out_v, int64_t out_rows, int sm_count, cudaStream_t s) {
  constexpr int CHV = 8;  // one round = 32 lanes x 8 vectors = 4 KiB of K and 4 KiB of V in flight per warp
  int64_t chunk_rows = GTKV_GATHER_CHUNK / (16 * p.vpr);
  if (chunk_rows < 1) chunk_rows = 1;
  if (chunk_rows > p.ps) chunk_rows = p.ps;
  const int64_t cpp = (p.ps + chunk_rows - 1) / chunk_rows;
  auto kernel = k_gather_runs<CHV>;
  int64_t warps = static_cast<int64_t>(n_seqs) * max_pages * cpp;
  const int64_t seq_warps = (static_cast<int64_t>(n_seqs) + 31) / 32;
  if (warps < seq_warps) warps = seq_warps;
  const unsigned grid = grid_for(kernel, warps, sm_count);
  kernel<<<grid, kBlock, 0, s>>>(p, layer, bt, n_seqs, max_pages, seq_start, seq_len, cu,
                                 static_cast<uint4*>(out_k), static_cast<uint4*>(out_v), out_rows,
                                 static_cast<int32_t>(chunk_rows), static_cast<int32_t>(cpp));
  return cudaGetLastError();
}

}  // namespace gtkv
