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
#include "kv_launch.h"
#include "kv_tasks.cuh"

namespace gtkv {

namespace {

__device__ __forceinline__ int check_id(const DevPool& p, int32_t id) {
  if (id < 0 || id >= p.n_rows) return KV_DEV_ERR_ROW;
  if (id % p.stride >= p.ps) return KV_DEV_ERR_FORM;
  return 0;
}

// Tasks t = pair * 2L + block. A warp takes 32 consecutive tasks at a time;
// lane k decodes task t0 + k and reads its pair's ids (prefetched one batch
// ahead), then the warp copies the batch in waves of 32/G rows.
template <int G, int VPL, int U>
__global__ void __launch_bounds__(kBlock) k_move(DevPool p, const int32_t* __restrict__ src_ids,
                                                 const int32_t* __restrict__ dst_ids, int64_t n_tasks, int batch) {
  constexpr int RPW = 32 / G;
  const int lane = threadIdx.x & 31;
  const int g = lane % G;
  const int grp = lane / G;
  const int64_t vpr = VPL > 0 ? static_cast<int64_t>(G) * VPL : p.vpr;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t step = ((static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5) * batch;
  const int64_t blocks = p.blocks;
  const L2Policy pol = make_l2_policy();

  int64_t t0 = warp * batch;
  const bool mine = lane < batch;  // lane owns a task of the batch
  int32_t s_next = -1, d_next = -1;
  auto fetch = [&](int64_t t) {
    if (t < n_tasks) {
      const int64_t i = t / blocks;
      s_next = __ldg(src_ids + i);
      d_next = __ldg(dst_ids + i);
    }
  };
  fetch(mine ? t0 + lane : n_tasks);
  for (; t0 < n_tasks; t0 += step) {
    const int64_t t = mine ? t0 + lane : n_tasks;
    const int32_t s_id = s_next, d_id = d_next;
    fetch(mine ? t0 + step + lane : n_tasks);
    long long sr = -1, dr = -1;
    if (t < n_tasks) {
      const int64_t b = t % blocks;
      const int e = check_id(p, s_id) | check_id(p, d_id);
      if (e == 0) {
        sr = s_id + b * p.ps;
        dr = d_id + b * p.ps;
      } else if (b == 0) {
        atomicOr(p.err, e);
      }
    }
    const int cnt = static_cast<int>(n_tasks - t0 < batch ? n_tasks - t0 : batch);
#pragma unroll 1
    for (int w0 = 0; w0 < cnt; w0 += RPW * U) {
      const uint4* src[U];
      uint4* dst[U];
      bool go[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int j = w0 + u * RPW + grp;
        const long long a = __shfl_sync(kFull, sr, j & 31);
        const long long c = __shfl_sync(kFull, dr, j & 31);
        const bool ok = j < cnt && a >= 0;
        go[u] = ok;
        src[u] = p.base + (ok ? a : 0) * vpr;
        dst[u] = p.base + (ok ? c : 0) * vpr;
      }
      copy_rows<G, VPL, U, kLdPlain, GTKV_MOVE_ST>(src, dst, go, g, vpr, pol);
    }
  }
}

}  // namespace

cudaError_t launch_move(const DevPool& p, const int32_t* src, const int32_t* dst, int64_t n, int sm_count,
                        cudaStream_t s) {
  const int64_t n_tasks = n * p.blocks;
  return dispatch_row(p.vpr, [&]<int G, int VPL>() -> cudaError_t {
    constexpr int U0 = VPL == 0 ? 1 : (VPL >= GTKV_MOVE_VEC ? 1 : GTKV_MOVE_VEC / VPL);
    constexpr int U = U0 < G ? U0 : G;  // one wave set fits in a 32-task batch
    auto kernel = k_move<G, VPL, U>;
    const int batch = task_batch(kernel, n_tasks, (32 / G) * U, sm_count);
    const unsigned grid = grid_all((n_tasks + batch - 1) / batch);
    kernel<<<grid, kBlock, 0, s>>>(p, src, dst, n_tasks, batch);
    return cudaGetLastError();
  });
}

}  // namespace gtkv
