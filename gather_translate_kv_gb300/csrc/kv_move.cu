// K5: move every row-block (all layers' K and V) of token src to token dst.
// Source: prhub report on sglang PR #34602, 关键文件 memory_pool.py
// (_move_kv_cache_impl copies all layers' KV of the src tokens to the dst
// tokens) over the dense views of build_mha_views: block b of token id is
// view row id + b*ps, for b in [0, 2L).
//
// A task is one (pair, block) = one row; a warp takes (32/G)*U consecutive
// tasks, so the 2L rows of a pair are spread over consecutive row groups.
// Sources and destinations are disjoint by precondition, so loads use the
// coherent path (the pool is written by this kernel) and need no ordering.
#include "kv_common.cuh"

namespace gtkv {

namespace {

__device__ __forceinline__ int check_id(const DevPool& p, int32_t id) {
  if (id < 0 || id >= p.n_rows) return KV_DEV_ERR_ROW;
  if (id % p.stride >= p.ps) return KV_DEV_ERR_FORM;
  return 0;
}

template <int G, int VPL, int U>
__global__ void __launch_bounds__(kBlock) k_move(DevPool p, const int32_t* __restrict__ src_ids,
                                                 const int32_t* __restrict__ dst_ids, int64_t n_tasks) {
  constexpr int RPW = 32 / G;
  constexpr int TPU = RPW * U;
  const int lane = threadIdx.x & 31;
  const int g = lane % G;
  const int grp = lane / G;
  const int64_t vpr = VPL > 0 ? static_cast<int64_t>(G) * VPL : p.vpr;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int64_t blocks = p.blocks;
  const L2Policy pol = make_l2_policy();

  for (int64_t t0 = warp * TPU; t0 < n_tasks; t0 += nwarps * TPU) {
    const uint4* src[U];
    uint4* dst[U];
    bool go[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t t = t0 + u * RPW + grp;
      long long sr = -1, dr = -1;
      if (g == 0 && t < n_tasks) {
        const int64_t i = t / blocks;
        const int64_t b = t - i * blocks;
        const int32_t s_id = __ldg(src_ids + i);
        const int32_t d_id = __ldg(dst_ids + i);
        const int e = check_id(p, s_id) | check_id(p, d_id);
        if (e == 0) {
          sr = s_id + b * p.ps;
          dr = d_id + b * p.ps;
        } else if (b == 0) {
          atomicOr(p.err, e);
        }
      }
      const int leader = lane & ~(G - 1);
      sr = __shfl_sync(kFull, sr, leader);
      dr = __shfl_sync(kFull, dr, leader);
      go[u] = sr >= 0;
      src[u] = p.base + (sr >= 0 ? sr : 0) * vpr;
      dst[u] = p.base + (sr >= 0 ? dr : 0) * vpr;
    }
    copy_rows<G, VPL, U, kLdPlain, GTKV_MOVE_ST>(src, dst, go, g, vpr, pol);
  }
}

}  // namespace

cudaError_t launch_move(const DevPool& p, const int32_t* src, const int32_t* dst, int64_t n, int sm_count,
                        cudaStream_t s) {
  const int64_t n_tasks = n * p.blocks;
  return dispatch_row(p.vpr, [&]<int G, int VPL>() -> cudaError_t {
    constexpr int U = VPL == 0 ? 1 : (VPL >= 8 ? 1 : 8 / VPL);
    auto kernel = k_move<G, VPL, U>;
    const int64_t tpu = (32 / G) * U;
    const unsigned grid = grid_for(kernel, (n_tasks + tpu - 1) / tpu, sm_count);
    kernel<<<grid, kBlock, 0, s>>>(p, src, dst, n_tasks);
    return cudaGetLastError();
  });
}

}  // namespace gtkv
