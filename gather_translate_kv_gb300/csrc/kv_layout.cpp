// Host-side layout arithmetic and start-up gates (see kv_layout.h).
#include "kv_layout.h"

namespace gtkv {

namespace {

bool mul(int64_t a, int64_t b, int64_t* out) { return !__builtin_mul_overflow(a, b, out); }
bool add(int64_t a, int64_t b, int64_t* out) { return !__builtin_add_overflow(a, b, out); }

}  // namespace

int compute_layout(const kv_pool_desc* d, Layout* out) {
  if (d == nullptr || out == nullptr) return KV_ERR_INVALID;
  if (d->layer_num < 1 || d->head_num < 1 || d->head_dim < 1 || d->page_size < 1 ||
      d->num_pages < 1 || d->anchor_bytes < 0)
    return KV_ERR_INVALID;
  if (d->itemsize != 1 && d->itemsize != 2 && d->itemsize != 4) return KV_ERR_INVALID;
  if ((d->latent_only != 0 && d->latent_only != 1) || d->reserved != 0) return KV_ERR_INVALID;
  // build_mha_views: the row-block array exists only for uniform K/V rows;
  // unified_memory_supported_for_model admits MLA (one latent row) regardless.
  if (!d->latent_only && d->head_dim != d->v_head_dim) return KV_ERR_ASYMMETRIC;

  Layout L{};
  L.kv_rows = d->latent_only ? 1 : 2;
  L.blocks = L.kv_rows * static_cast<int64_t>(d->layer_num);
  if (!mul(static_cast<int64_t>(d->head_num) * d->head_dim, d->itemsize, &L.R)) return KV_ERR_INVALID;
  // _assert_kernel_id_bound: kernel-facing rows num_pages * 2L * ps < 2^31.
  if (!mul(L.blocks, d->page_size, &L.stride)) return KV_ERR_ID_BOUND;
  if (!mul(d->num_pages, L.stride, &L.n_rows) || L.n_rows >= (int64_t(1) << 31))
    return KV_ERR_ID_BOUND;
  // build_mha_views asserts anchor % itemsize; every kernel here also moves
  // rows as 16-byte vectors, so rows and the anchor must be 16-byte multiples.
  if (d->anchor_bytes % d->itemsize != 0) return KV_ERR_ALIGN;
  if (L.R % 16 != 0 || d->anchor_bytes % 16 != 0) return KV_ERR_ALIGN;

  int64_t rows_bytes, reach;
  if (!mul(L.stride, L.R, &L.page_bytes)) return KV_ERR_INVALID;
  if (!mul(d->num_pages, L.page_bytes, &L.total)) return KV_ERR_INVALID;
  L.tail_pad = L.page_bytes;  // ps * entry_bytes with entry_bytes = blocks * R
  if (!mul(L.n_rows, L.R, &rows_bytes)) return KV_ERR_INVALID;
  if (!mul((L.blocks - 1) * d->page_size, L.R, &reach)) return KV_ERR_INVALID;
  if (!add(d->anchor_bytes, reach, &L.last_view_end) || !add(L.last_view_end, rows_bytes, &L.last_view_end))
    return KV_ERR_INVALID;
  if (!add(d->anchor_bytes, L.total, &L.alloc_bytes) || !add(L.alloc_bytes, L.tail_pad, &L.alloc_bytes))
    return KV_ERR_INVALID;
  *out = L;
  return KV_OK;
}

}  // namespace gtkv
