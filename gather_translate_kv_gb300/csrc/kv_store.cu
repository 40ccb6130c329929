// K2 / K3: scatter K and V rows into the pool, one layer or all layers.
// Source: prhub report on sglang PR #34602 -- 实现拆解 step 1 (layer l's K is
// row-block 2l, its V row-block 2l+1 of the page envelope) and the dense
// per-layer views of build_mha_views (关键源码片段 layout/page_major.py),
// through which _store_kv_layer's plain 3D assignment writes
// k_buffer[l][id] = k and v_buffer[l][id] = v.
//
// In view terms, token id's K row of layer l is pool row id + 2l*ps and its V
// row id + (2l+1)*ps. A task is one (layer, token) pair; it moves 2 rows in
// (contiguous K/V inputs) and 2 rows out (scattered pool rows).
#include "kv_common.cuh"

namespace gtkv {

namespace {

// Tasks t in [0, n_tasks), n_tasks = n_layers * n: layer = layer0 + t / n,
// token i = t % n; the input rows are K[t] and V[t] (a [n_layers, n, H, D]
// layout, n_layers = 1 for the per-layer call). A warp takes TPU = (32/G)*U
// consecutive tasks at a time; lane 0 of each row group reads the id and
// shares the destination row by shuffle.
template <int G, int VPL, int U>
__global__ void __launch_bounds__(kBlock) k_store(DevPool p, int32_t layer0, int64_t n, int64_t n_tasks,
                                                  const int32_t* __restrict__ ids, const uint4* __restrict__ K,
                                                  const uint4* __restrict__ V) {
  constexpr int RPW = 32 / G;
  constexpr int TPU = RPW * U;
  const int lane = threadIdx.x & 31;
  const int g = lane % G;
  const int grp = lane / G;
  const int64_t vpr = VPL > 0 ? static_cast<int64_t>(G) * VPL : p.vpr;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const bool one_layer = n_tasks == n;
  const L2Policy pol = make_l2_policy();

  for (int64_t t0 = warp * TPU; t0 < n_tasks; t0 += nwarps * TPU) {
    const uint4* src[2 * U];
    uint4* dst[2 * U];
    bool go[2 * U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t t = t0 + u * RPW + grp;
      long long row = -1;  // K row of this task, in view units; -1 = skip
      if (g == 0 && t < n_tasks) {
        const int64_t l = one_layer ? 0 : t / n;
        const int32_t id = __ldg(ids + (t - l * n));
        if (id >= 0 && id < p.n_rows) {
          row = id + 2 * (layer0 + l) * p.ps;
        } else {
          atomicOr(p.err, KV_DEV_ERR_ROW);
        }
      }
      row = __shfl_sync(kFull, row, lane & ~(G - 1));
      const bool ok = row >= 0;
      go[2 * u] = go[2 * u + 1] = ok;
      const int64_t tt = ok ? t : 0;
      const int64_t rr = ok ? row : 0;
      src[2 * u] = K + tt * vpr;
      src[2 * u + 1] = V + tt * vpr;
      dst[2 * u] = p.base + rr * vpr;
      dst[2 * u + 1] = p.base + (rr + p.ps) * vpr;
    }
    copy_rows<G, VPL, 2 * U, GTKV_STORE_LD, GTKV_STORE_ST>(src, dst, go, g, vpr, pol);
  }
}

}  // namespace

cudaError_t launch_store(const DevPool& p, int32_t layer0, int32_t n_layers, const int32_t* ids, int64_t n,
                         const void* k, const void* v, int sm_count, cudaStream_t s) {
  const int64_t n_tasks = n * n_layers;
  return dispatch_row(p.vpr, [&]<int G, int VPL>() -> cudaError_t {
    // about 8 row vectors in flight per lane (K and V of U tasks)
    constexpr int U = VPL == 0 ? 1 : (VPL >= 4 ? 1 : 4 / VPL);
    auto kernel = k_store<G, VPL, U>;
    const int64_t tpu = (32 / G) * U;
    const unsigned grid = grid_for(kernel, (n_tasks + tpu - 1) / tpu, sm_count);
    kernel<<<grid, kBlock, 0, s>>>(p, layer0, n, n_tasks, ids, static_cast<const uint4*>(k),
                                   static_cast<const uint4*>(v));
    return cudaGetLastError();
  });
}

}  // namespace gtkv
