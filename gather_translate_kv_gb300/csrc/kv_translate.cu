// K1: token slots -> kernel-facing int32 ids.
// Source: prhub report on sglang PR #34602, 关键源码片段
// multi_ended_allocator.py, translate_kv_loc_for_kernel: split slots into
// pages and offsets, map pages virtual -> physical, scale by the page stride
// ps * 2L and clamp tombstones to 0 (the page-0 sink).
#include "kv_launch.h"

namespace gtkv {

namespace {

// One slot per thread per iteration, grid-stride. Reads 8 B (+4 B of page map)
// and writes 4 B per slot; launch-bound at the sizes a forward batch has.
__global__ void __launch_bounds__(kBlock) k_translate(DevPool p, const int64_t* __restrict__ slots, int64_t n,
                                                      const int32_t* __restrict__ v2p, int64_t v2p_len,
                                                      int32_t* __restrict__ ids) {
  int bits = 0;
  const int64_t step = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += step)
    ids[i] = static_cast<int32_t>(slot_to_id(p, __ldg(slots + i), v2p, v2p_len, bits));
  if (bits) atomicOr(p.err, bits);
}

// Kernel-facing block table, prefix only: one table entry per thread.
// Entry k of sequence s is translated when k < ceil(len_s / ps) (capped at
// max_pages): virtual page -> physical page through the map, scaled by the
// row-blocks per page (2L) so that entry * ps + offset is the kernel-facing
// id; tombstones and errors give 0, the sink page. Later entries are untouched.
// virt and out may be the same buffer (in place): each thread reads its own
// entry before writing it, so neither pointer is declared __restrict__.
__global__ void __launch_bounds__(kBlock) k_block_table(DevPool p, const int32_t* virt,
                                                        int32_t n_seqs, int32_t max_pages,
                                                        const int32_t* __restrict__ seq_len,
                                                        const int32_t* __restrict__ v2p, int64_t v2p_len,
                                                        int32_t* out) {
  int bits = 0;
  const int64_t n = static_cast<int64_t>(n_seqs) * max_pages;
  const int64_t step = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < n; e += step) {
    const int64_t s = e / max_pages;
    const int64_t k = e - s * max_pages;
    const int64_t len = __ldg(seq_len + s);
    int64_t np = len > 0 ? div_ps(p, len + p.ps - 1) : 0;
    if (np > max_pages) {
      if (k == 0) bits |= KV_DEV_ERR_TABLE;
      np = max_pages;
    }
    if (k >= np) continue;
    const int64_t vp = virt[e];
    int64_t phys = -1;
    if (vp >= 0) {
      if (vp < v2p_len) {
        phys = __ldg(v2p + vp);
      } else {
        bits |= KV_DEV_ERR_V2P;
      }
    }
    if (phys >= p.num_pages) {
      bits |= KV_DEV_ERR_ROW;
      phys = -1;
    }
    out[e] = static_cast<int32_t>(phys < 0 ? 0 : phys * p.blocks);
  }
  if (bits) atomicOr(p.err, bits);
}

// Full -> SWA token map, then translate (one slot per thread): t' = tmap[t]
// for 0 <= t < tmap_len (a negative t' is a cleared entry: the sink), t < 0
// is a tombstone, t >= tmap_len an error that also gives the sink.
__global__ void __launch_bounds__(kBlock) k_translate_mapped(DevPool p, const int64_t* __restrict__ slots, int64_t n,
                                                             const int64_t* __restrict__ tmap, int64_t tmap_len,
                                                             const int32_t* __restrict__ v2p, int64_t v2p_len,
                                                             int32_t* __restrict__ ids) {
  int bits = 0;
  const int64_t step = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += step) {
    const int64_t t = __ldg(slots + i);
    int64_t mapped = -1;
    if (t >= 0) {
      if (t < tmap_len) {
        mapped = __ldg(tmap + t);
      } else {
        bits |= KV_DEV_ERR_V2P;
      }
    }
    ids[i] = static_cast<int32_t>(slot_to_id(p, mapped, v2p, v2p_len, bits));
  }
  if (bits) atomicOr(p.err, bits);
}

}  // namespace

cudaError_t launch_translate_mapped(const DevPool& p, const int64_t* slots, int64_t n, const int64_t* tmap,
                                    int64_t tmap_len, const int32_t* v2p, int64_t v2p_len, int32_t* ids, int sm_count,
                                    cudaStream_t s) {
  const unsigned grid = grid_for(k_translate_mapped, (n + 31) / 32, sm_count);
  k_translate_mapped<<<grid, kBlock, 0, s>>>(p, slots, n, tmap, tmap_len, v2p, v2p_len, ids);
  return cudaGetLastError();
}

cudaError_t launch_block_table(const DevPool& p, const int32_t* virt, int32_t n_seqs, int32_t max_pages,
                               const int32_t* seq_len, const int32_t* v2p, int64_t v2p_len, int32_t* out,
                               int sm_count, cudaStream_t s) {
  const int64_t warps = (static_cast<int64_t>(n_seqs) * max_pages + 31) / 32;
  const unsigned grid = grid_for(k_block_table, warps, sm_count);
  k_block_table<<<grid, kBlock, 0, s>>>(p, virt, n_seqs, max_pages, seq_len, v2p, v2p_len, out);
  return cudaGetLastError();
}

cudaError_t launch_translate(const DevPool& p, const int64_t* slots, int64_t n, const int32_t* v2p,
                             int64_t v2p_len, int32_t* ids, int sm_count, cudaStream_t s) {
  const int64_t warps = (n + 31) / 32;
  const unsigned grid = grid_for(k_translate, warps, sm_count);
  k_translate<<<grid, kBlock, 0, s>>>(p, slots, n, v2p, v2p_len, ids);
  return cudaGetLastError();
}

}  // namespace gtkv
