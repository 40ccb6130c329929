// K1: token slots -> kernel-facing int32 ids.
// Source: prhub report on sglang PR #34602, 关键源码片段
// multi_ended_allocator.py, translate_kv_loc_for_kernel: split slots into
// pages and offsets, map pages virtual -> physical, scale by the page stride
// ps * 2L and clamp tombstones to 0 (the page-0 sink).
#include "kv_common.cuh"

namespace gtkv {

namespace {

// One slot per thread per iteration, grid-stride. Reads 8 B (+4 B of page map)
// and writes 4 B per slot; launch-bound at the sizes a forward batch has.
__global__ void __launch_bounds__(kBlock) k_translate(DevPool p, const int64_t* __restrict__ slots, int64_t n,
                                                      const int32_t* __restrict__ v2p, int64_t v2p_len,
                                                      int32_t* __restrict__ ids) {
  int bits = 0;
  const int64_t step = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += step) {
    const int64_t t = __ldg(slots + i);
    int64_t id = 0;
    if (t >= 0) {
      const int64_t page = div_ps(p, t);
      const int64_t off = t - page * p.ps;
      int64_t phys = page;
      if (v2p != nullptr) {
        if (page < v2p_len) {
          phys = __ldg(v2p + page);
        } else {
          phys = -1;
          bits |= KV_DEV_ERR_V2P;
        }
      }
      if (phys >= p.num_pages) {
        phys = -1;
        bits |= KV_DEV_ERR_ROW;
      }
      if (phys >= 0) id = phys * p.stride + off;
    }
    ids[i] = static_cast<int32_t>(id);
  }
  if (bits) atomicOr(p.err, bits);
}

}  // namespace

cudaError_t launch_translate(const DevPool& p, const int64_t* slots, int64_t n, const int32_t* v2p,
                             int64_t v2p_len, int32_t* ids, int sm_count, cudaStream_t s) {
  const int64_t warps = (n + 31) / 32;
  const unsigned grid = grid_for(k_translate, warps, sm_count);
  k_translate<<<grid, kBlock, 0, s>>>(p, slots, n, v2p, v2p_len, ids);
  return cudaGetLastError();
}

}  // namespace gtkv
