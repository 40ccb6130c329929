// Launch shapes of the row-task kernels (kv_store.cu, kv_move.cu): one warp
// per batch of tasks on an uncapped grid. Host code only.
#pragma once

#include "kv_common.cuh"

namespace gtkv {

// Grid for `warps_needed` warps of work, one warp per batch of tasks and no
// cap: the hardware block scheduler hands blocks to SMs as they free up, so
// SMs whose memory traffic drains faster take more of the work. Used by the
// store and the move. A persistent grid with a fixed share per warp
// measured 4-10 % slower on them: on this GPU some SMs finish an equal share
// of a write stream several times sooner than others, and the launch lasts
// as long as the slowest.
inline unsigned grid_all(int64_t warps_needed) {
  const int64_t per_block = kBlock / 32;
  int64_t blocks = (warps_needed + per_block - 1) / per_block;
  if (blocks < 1) blocks = 1;
  if (blocks > 0x7fffffff) blocks = 0x7fffffff;  // the kernels loop grid-stride beyond this
  return static_cast<unsigned>(blocks);
}

// Tasks per warp batch for the row-task kernels (store, move): lanes hold the
// metadata of up to 32 tasks, copied in waves of `wave` tasks. The batch is
// sized so that the (uncapped) grid holds about kTaskWaves times the warps
// the SMs keep resident, up to full 32-task batches: blocks stay short, so
// the launch ends with a short tail. Small calls shrink the batch (to a
// multiple of the wave) so that the work still spreads over every SM.
// Measured against one wave: the per-layer prefill store 43.0 -> 39.7 us,
// the decode move 353 -> 350 us, the MLA move 115.5 -> 114 us; eight waves
// cost the SWA move 3 %.
#ifndef GTKV_TASK_WAVES
#define GTKV_TASK_WAVES 4
#endif
constexpr int kTaskWaves = GTKV_TASK_WAVES;

template <class K>
inline int task_batch(K kernel, int64_t n_tasks, int wave, int sm_count) {
  const int64_t warps_full =
      static_cast<int64_t>(sm_count) * blocks_per_sm(kernel) * (kBlock / 32) * kTaskWaves;
  int64_t b = (n_tasks + warps_full - 1) / warps_full;
  if (wave > 32) wave = 32;
  b = (b + wave - 1) / wave * wave;
  if (b < wave) b = wave;
  if (b > 32) b = 32 / wave * wave;
  return static_cast<int>(b);
}

}  // namespace gtkv
