// Host-side layout arithmetic and start-up gates of the page-major KV pool.
// Layout source: prhub report on sglang PR #34602, 关键源码片段
// layout/page_major.py (build_mha_views) and unified_memory_pool.py
// (view_tail_pad_bytes, _assert_kernel_id_bound).
#pragma once

#include <stdint.h>

#include "kv_pool.h"

namespace gtkv {

struct Layout {
  int64_t R;              // row bytes, H * D * itemsize
  int64_t blocks;         // row-blocks per page: 2L (MHA/SWA) or L (MLA)
  int64_t kv_rows;        // rows per layer per token: 2 (K, V) or 1 (MLA latent)
  int64_t page_bytes;     // ps * blocks * R
  int64_t total;          // num_pages * page_bytes
  int64_t tail_pad;       // ps * 2L * R (one page envelope)
  int64_t n_rows;         // num_pages * 2L * ps
  int64_t stride;         // rows per page, ps * 2L
  int64_t last_view_end;  // anchor + (2L-1)*ps*R + n_rows*R
  int64_t alloc_bytes;    // anchor + total + tail_pad
};

// Validates the descriptor (every gate but the buffer size) and fills *out.
// Returns KV_OK or a KV_ERR_* code. Overflow-safe for any input.
int compute_layout(const kv_pool_desc* d, Layout* out);

}  // namespace gtkv
