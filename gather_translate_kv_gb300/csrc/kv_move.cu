// K5: move every row-block (all layers' K and V) of token src to token dst.
// Source: prhub report on sglang PR #34602, 关键文件 memory_pool.py
// (_move_kv_cache_impl copies all layers' KV of the src tokens to the dst
// tokens) over the dense views of build_mha_views: block b of token id is
// view row id + b*ps, for b in [0, 2L).
//
// Vector form: a task is one (pair, block) = one row; a warp takes (32/G)*U
// consecutive tasks, so the 2L rows of a pair are spread over consecutive row
// groups. Sources and destinations are disjoint by precondition, so loads use
// the coherent path (the pool is written by this kernel) and need no ordering.
// Rows of at least 128 bytes take the bulk-copy form below instead (one warp
// per pair, or per chunk of at most 18 KiB of it, through shared memory).
#include "kv_bulk.cuh"
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

// Bulk-copy form: one block of one warp per pair, or per chunk of a pair's
// row-blocks when the pair holds more than GTKV_MOVE_BULK_MAX_BYTES (grid-
// stride beyond the grid). Lane j issues the bulk loads of rows b0 + j,
// b0 + j + 32, ... of token src into shared memory, counted on one mbarrier,
// and once they have landed their bulk stores to the same rows of token dst.
// Measured against the vector kernel over 8192 random pairs on 2 GB pools
// (us): rows of 128 to 2048 bytes with up to 36 KiB per pair 2-10 % faster
// (512-byte rows x 24 row-blocks 74.7 -> 70.8, the SWA move 67.7 -> 63.9);
// whole pairs of 64 to 72 KiB (3 in flight per SM) the same or up to 12 %
// slower, but split into chunks 0.4-3 % faster (the decode move 353 -> 348);
// 64-byte rows 15 % slower. Chunks of 18 KiB against 36 KiB: the SWA move
// 64.6 -> 62.8, the MLA move ~1 % faster, the rest within noise. So the
// launcher takes this form for rows of at least 128 bytes, in chunks of at
// most 18 KiB.
#ifndef GTKV_MOVE_BULK
#define GTKV_MOVE_BULK 1  // 0: every move takes the vector kernel
#endif
#ifndef GTKV_MOVE_BULK_MAX_BYTES
#define GTKV_MOVE_BULK_MAX_BYTES 18432  // bytes of a pair's rows per block (chunk)
#endif
#ifndef GTKV_MOVE_BULK_MIN_ROW
#define GTKV_MOVE_BULK_MIN_ROW 128
#endif
#ifndef GTKV_MOVE_BULK_SPLIT
#define GTKV_MOVE_BULK_SPLIT 1  // 0: pairs over GTKV_MOVE_BULK_MAX_BYTES keep the vector kernel
#endif

__global__ void __launch_bounds__(32) k_move_bulk(DevPool p, const int32_t* __restrict__ src_ids,
                                                  const int32_t* __restrict__ dst_ids, int64_t n, int chunks,
                                                  int chunk_rows) {
  extern __shared__ __align__(128) uint4 sbuf[];  // one chunk of the pair's row-blocks, in block order
  __shared__ __align__(8) uint64_t bar;
  const int lane = threadIdx.x;
  const int64_t vpr = p.vpr;
  const int blocks = p.blocks;
  const uint32_t rbytes = static_cast<uint32_t>(vpr * 16);
  const L2Policy pol = make_l2_policy();
  if (lane == 0) mbar_init(&bar);
  __syncwarp();
  uint32_t parity = 0;
  const int64_t n_units = n * chunks;
  for (int64_t w = blockIdx.x; w < n_units; w += gridDim.x) {
    const int64_t i = w / chunks;
    const int b0 = static_cast<int>(w - i * chunks) * chunk_rows;
    const int b1 = b0 + chunk_rows < blocks ? b0 + chunk_rows : blocks;
    const int32_t s_id = __ldg(src_ids + i), d_id = __ldg(dst_ids + i);
    const int e = check_id(p, s_id) | check_id(p, d_id);
    if (e != 0) {
      if (lane == 0 && b0 == 0) atomicOr(p.err, e);
      continue;
    }
    if (lane == 0) mbar_expect(&bar, rbytes * static_cast<uint32_t>(b1 - b0));
    __syncwarp();  // the phase expects its bytes before any load can complete it
    for (int b = b0 + lane; b < b1; b += 32)
      bulk_load(sbuf + (b - b0) * vpr, p.base + (s_id + static_cast<int64_t>(b) * p.ps) * vpr, rbytes, &bar,
                pol.first);
    if (!__all_sync(kFull, mbar_wait_bounded(&bar, parity))) {
      if (lane == 0) atomicOr(p.err, KV_DEV_ERR_TIMEOUT);
      mbar_wait_bounded(&bar, parity);
      bulk_wait_all();
      return;
    }
    parity ^= 1;
    for (int b = b0 + lane; b < b1; b += 32)
      bulk_store(p.base + (d_id + static_cast<int64_t>(b) * p.ps) * vpr, sbuf + (b - b0) * vpr, rbytes,
                 pol.first);
    bulk_commit();
    bulk_wait_read();  // the next unit's loads reuse the buffer
    __syncwarp();
  }
}

}  // namespace

cudaError_t launch_move(const DevPool& p, const int32_t* src, const int32_t* dst, int64_t n, int sm_count,
                        cudaStream_t s) {
  const int64_t n_tasks = n * p.blocks;
  const int64_t pair_bytes = static_cast<int64_t>(p.blocks) * p.vpr * 16;
  const int64_t R = p.vpr * 16;
  if (GTKV_MOVE_BULK && R >= GTKV_MOVE_BULK_MIN_ROW &&
      (pair_bytes <= GTKV_MOVE_BULK_MAX_BYTES || GTKV_MOVE_BULK_SPLIT)) {
    static_assert(GTKV_MOVE_BULK_MAX_BYTES <= 48 * 1024, "within the default dynamic shared memory limit");
    // a pair over GTKV_MOVE_BULK_MAX_BYTES is split into equal chunks of row-blocks, one block each
    int64_t chunks = (pair_bytes + GTKV_MOVE_BULK_MAX_BYTES - 1) / GTKV_MOVE_BULK_MAX_BYTES;
    if (chunks > p.blocks) chunks = p.blocks;
    const int64_t chunk_rows = (p.blocks + chunks - 1) / chunks;
    chunks = (p.blocks + chunk_rows - 1) / chunk_rows;
    if (chunk_rows * R <= GTKV_MOVE_BULK_MAX_BYTES) {
      const int smem = static_cast<int>(chunk_rows * R);
      const int64_t units = n * chunks;
      const unsigned grid = static_cast<unsigned>(units < 0x7fffffff ? units : 0x7fffffff);
      k_move_bulk<<<grid, 32, smem, s>>>(p, src, dst, n, static_cast<int>(chunks), static_cast<int>(chunk_rows));
      return cudaGetLastError();
    }
  }
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
