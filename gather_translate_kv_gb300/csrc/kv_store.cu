// K2 / K3: scatter K and V rows into the pool, one layer or all layers.
// Source: prhub report on sglang PR #34602 -- 实现拆解 step 1 (layer l's K is
// row-block 2l, its V row-block 2l+1 of the page envelope) and the dense
// per-layer views of build_mha_views (关键源码片段 layout/page_major.py),
// through which _store_kv_layer's plain 3D assignment writes
// k_buffer[l][id] = k and v_buffer[l][id] = v.
//
// In view terms, token id's K row of layer l is pool row id + 2l*ps and its V
// row id + (2l+1)*ps. A task is one (layer, token) pair; it moves 2 rows in
// (contiguous K/V inputs) and 2 rows out (scattered pool rows). In an MLA pool
// (one latent row per layer, blocks_per_page = L) the row is id + l*ps and
// there is no V.
#include "kv_launch.h"
#include "kv_tasks.cuh"

namespace gtkv {

namespace {

// The two halves of copy_rows for callers that can issue their loads before
// the destinations are known (fixed-size rows only, VPL > 0).
template <int G, int VPL, int N, int LD>
__device__ __forceinline__ void load_rows(uint4 (&buf)[N][VPL], const uint4* const (&src)[N], const bool (&go)[N],
                                          int g, const L2Policy& pol) {
#pragma unroll
  for (int i = 0; i < N; ++i)
    if (go[i]) {
#pragma unroll
      for (int v = 0; v < VPL; ++v) buf[i][v] = ld16<LD>(src[i] + g + v * G, pol);
    }
}

template <int G, int VPL, int N, int ST>
__device__ __forceinline__ void store_rows(uint4* const (&dst)[N], const uint4 (&buf)[N][VPL], const bool (&go)[N],
                                           int g, const L2Policy& pol) {
#pragma unroll
  for (int i = 0; i < N; ++i)
    if (go[i]) {
#pragma unroll
      for (int v = 0; v < VPL; ++v) st16<ST>(dst[i] + g + v * G, buf[i][v], pol);
    }
}

// Tasks t in [0, n_tasks), n_tasks = n_layers * n: layer = layer0 + t / n,
// token i = t % n; the input rows are K[t] and V[t] (a [n_layers, n, H, D]
// layout, n_layers = 1 for the per-layer call). A warp takes 32 consecutive
// tasks at a time: lane k reads the id of task t0 + k (one coalesced load for
// the batch, issued one batch ahead so its latency hides behind the copies),
// then the warp copies the batch in waves of 32/G tasks, each task's
// destination row shared by shuffle from the lane that owns it.
//
// With SLOTS the tasks carry token slots instead of ids, and each lane
// translates its own (translate fused into the store: one launch, no id
// buffer); a tombstone then lands on the sink exactly as kv_translate's id 0
// would.
template <int G, int VPL, int U, bool SLOTS>
__global__ void __launch_bounds__(kBlock) k_store(DevPool p, int32_t layer0, int64_t n, int64_t n_tasks,
                                                  const int32_t* __restrict__ ids, const int64_t* __restrict__ slots,
                                                  const int32_t* __restrict__ v2p, int64_t v2p_len,
                                                  const uint4* __restrict__ K, const uint4* __restrict__ V,
                                                  int batch) {
  constexpr int RPW = 32 / G;
  const int lane = threadIdx.x & 31;
  const int g = lane % G;
  const int grp = lane / G;
  const int64_t vpr = VPL > 0 ? static_cast<int64_t>(G) * VPL : p.vpr;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t step = ((static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5) * batch;
  const bool one_layer = n_tasks == n;
  const L2Policy pol = make_l2_policy();

  int64_t t0 = warp * batch;
  const bool mine = lane < batch;  // lane owns a task of the batch
  int64_t l_next = 0;
  int64_t id_next = -1;
  int bits = 0;
  auto fetch = [&](int64_t t) {
    l_next = (one_layer || t >= n_tasks) ? 0 : t / n;
    if (t >= n_tasks) {
      id_next = -1;
    } else if constexpr (SLOTS) {
      id_next = __ldg(slots + (t - l_next * n));  // translated below, once the load has landed
    } else {
      id_next = __ldg(ids + (t - l_next * n));
    }
  };
  fetch(mine ? t0 + lane : n_tasks);
  for (; t0 < n_tasks; t0 += step) {
    const int64_t t = mine ? t0 + lane : n_tasks;
    const int64_t id_raw = id_next;
    const int64_t l = l_next;
    fetch(mine ? t0 + step + lane : n_tasks);  // next batch's ids, in flight during this batch's copies
    // K row of this lane's task in view units (-1 = skip); worked out after
    // the first wave's data loads are issued, so a batch whose ids are still
    // in flight overlaps the two loads
    long long row = -1;
    auto resolve = [&]() {
      int64_t id = id_raw;
      if constexpr (SLOTS) {
        if (t < n_tasks) id = slot_to_id(p, id, v2p, v2p_len, bits);
      }
      if (t < n_tasks) {
        if (id < 0 || id >= p.n_rows) {
          atomicOr(p.err, KV_DEV_ERR_ROW);
        } else if (!SLOTS && static_cast<uint32_t>(id) % static_cast<uint32_t>(p.stride) >= p.ps) {
          // not of the form page * ps * 2L + o with o < ps: its rows would land
          // in another layer's row-block, so the task is skipped
          atomicOr(p.err, KV_DEV_ERR_FORM);
        } else {
          row = id + (layer0 + l) * p.kv_rows * p.ps;
        }
      }
    };
    const int cnt = static_cast<int>(n_tasks - t0 < batch ? n_tasks - t0 : batch);
#pragma unroll 1
    for (int w0 = 0; w0 < cnt; w0 += RPW * U) {
      const uint4* src[2 * U];
      uint4* dst[2 * U];
      bool go[2 * U];
      bool ld[2 * U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int j = w0 + u * RPW + grp;  // task within the batch
        const int64_t tt = j < cnt ? t0 + j : 0;
        ld[2 * u] = j < cnt;
        ld[2 * u + 1] = j < cnt && V != nullptr;  // an MLA pool has no V rows
        src[2 * u] = K + tt * vpr;
        src[2 * u + 1] = (V != nullptr ? V : K) + tt * vpr;
      }
      if constexpr (VPL > 0) {
        uint4 buf[2 * U][VPL];
        load_rows<G, VPL, 2 * U, GTKV_STORE_LD>(buf, src, ld, g, pol);  // sources do not depend on the ids
        if (w0 == 0) resolve();
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int j = w0 + u * RPW + grp;
          const long long rr = __shfl_sync(kFull, row, j & 31);
          const int64_t r_ = rr >= 0 ? rr : 0;
          go[2 * u] = ld[2 * u] && rr >= 0;
          go[2 * u + 1] = ld[2 * u + 1] && rr >= 0;
          dst[2 * u] = p.base + r_ * vpr;
          dst[2 * u + 1] = p.base + (r_ + p.ps) * vpr;
        }
        store_rows<G, VPL, 2 * U, GTKV_STORE_ST>(dst, buf, go, g, pol);
      } else {
        if (w0 == 0) resolve();
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int j = w0 + u * RPW + grp;
          const long long rr = __shfl_sync(kFull, row, j & 31);
          const int64_t r_ = rr >= 0 ? rr : 0;
          go[2 * u] = ld[2 * u] && rr >= 0;
          go[2 * u + 1] = ld[2 * u + 1] && rr >= 0;
          dst[2 * u] = p.base + r_ * vpr;
          dst[2 * u + 1] = p.base + (r_ + p.ps) * vpr;
        }
        copy_rows<G, VPL, 2 * U, GTKV_STORE_LD, GTKV_STORE_ST>(src, dst, go, g, vpr, pol);
      }
    }
  }
  if constexpr (SLOTS) {
    if (bits) atomicOr(p.err, bits);
  }
}

template <bool SLOTS>
cudaError_t launch(const DevPool& p, int32_t layer0, int32_t n_layers, const int32_t* ids, const int64_t* slots,
                   int64_t n, const int32_t* v2p, int64_t v2p_len, const void* k, const void* v, int sm_count,
                   cudaStream_t s) {
  const int64_t n_tasks = n * n_layers;
  return dispatch_row(p.vpr, [&]<int G, int VPL>() -> cudaError_t {
    // GTKV_STORE_VEC row vectors in flight per lane (K and V of U tasks)
    // (U capped at G so that one wave set, (32/G)*U tasks, fits in a 32-task batch)
    constexpr int U0 = VPL == 0 ? 1 : (2 * VPL >= GTKV_STORE_VEC ? 1 : GTKV_STORE_VEC / (2 * VPL));
    constexpr int U = U0 < G ? U0 : G;
    auto kernel = k_store<G, VPL, U, SLOTS>;
    const int batch = task_batch(kernel, n_tasks, (32 / G) * U, sm_count);
    const unsigned grid = grid_all((n_tasks + batch - 1) / batch);
    kernel<<<grid, kBlock, 0, s>>>(p, layer0, n, n_tasks, ids, slots, v2p, v2p_len, static_cast<const uint4*>(k),
                                   static_cast<const uint4*>(v), batch);
    return cudaGetLastError();
  });
}

}  // namespace

cudaError_t launch_store(const DevPool& p, int32_t layer0, int32_t n_layers, const int32_t* ids, int64_t n,
                         const void* k, const void* v, int sm_count, cudaStream_t s) {
  return launch<false>(p, layer0, n_layers, ids, nullptr, n, nullptr, 0, k, v, sm_count, s);
}

cudaError_t launch_store_slots(const DevPool& p, int32_t layer0, int32_t n_layers, const int64_t* slots, int64_t n,
                               const int32_t* v2p, int64_t v2p_len, const void* k, const void* v, int sm_count,
                               cudaStream_t s) {
  return launch<true>(p, layer0, n_layers, nullptr, slots, n, v2p, v2p_len, k, v, sm_count, s);
}

}  // namespace gtkv
