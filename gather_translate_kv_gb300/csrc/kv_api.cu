// The C ABI of include/kv_pool.h: argument checks, pool bookkeeping and
// kernel launches. Nothing here touches K/V bytes; every step of the path runs
// in the kernels of kv_translate.cu, kv_store.cu, kv_gather.cu and kv_move.cu.
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>
#include <stdint.h>

#include <new>

#include "kv_launch.h"
#include "kv_layout.h"
#include "kv_pool.h"
#include "kv_pool_internal.h"

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// An NVTX range around one API call, so profilers show which entry point
// enqueued which kernel (a no-op when no tool is attached).
struct Range {
  explicit Range(const char* name) { nvtxRangePushA(name); }
  ~Range() { nvtxRangePop(); }
  Range(const Range&) = delete;
  Range& operator=(const Range&) = delete;
};

int ps_shift_of(int64_t ps) {
  if ((ps & (ps - 1)) != 0) return -1;
  int s = 0;
  while ((int64_t(1) << s) < ps) ++s;
  return s;
}

// Current device must be the pool's.
int enter(const kv_pool_t* pool) {
  if (pool == nullptr) return KV_ERR_INVALID;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return KV_ERR_CUDA;
  return dev == pool->device ? KV_OK : KV_ERR_DEVICE;
}

// Status of an enqueue. A failed runtime call also leaves its error in the
// runtime's last-error slot, where the next launch's check would find it;
// take it out so that it is reported once, here.
int launched(cudaError_t e) {
  if (e == cudaSuccess) return KV_OK;
  cudaGetLastError();
  return KV_ERR_CUDA;
}

// A runtime call of pool set-up failed: take its error out of the runtime's
// last-error slot (it would otherwise surface as the status of the next
// launch, through cudaGetLastError) and report KV_ERR_CUDA.
int failed_call() {
  cudaGetLastError();
  return KV_ERR_CUDA;
}

// The pool's device words: [0] the error word the kernels OR bits into,
// [1] where kv_pool_last_error parks the value it took.
constexpr size_t kErrWords = 2;

// Read and clear the error word in one step, so a bit that work on another
// stream raises meanwhile is kept for the next read instead of being lost.
__global__ void k_take_error(int32_t* err) { err[1] = atomicExch(err, 0); }

cudaStream_t as_stream(kv_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

}  // namespace

extern "C" {

const char* kv_status_string(int status) {
  switch (status) {
    case KV_OK: return "KV_OK";
    case KV_ERR_INVALID: return "KV_ERR_INVALID";
    case KV_ERR_ASYMMETRIC: return "KV_ERR_ASYMMETRIC";
    case KV_ERR_ID_BOUND: return "KV_ERR_ID_BOUND";
    case KV_ERR_TAIL_PAD: return "KV_ERR_TAIL_PAD";
    case KV_ERR_ALIGN: return "KV_ERR_ALIGN";
    case KV_ERR_CUDA: return "KV_ERR_CUDA";
    case KV_ERR_DEVICE: return "KV_ERR_DEVICE";
    case KV_ERR_CAPACITY: return "KV_ERR_CAPACITY";
    default: return "KV_ERR_UNKNOWN";
  }
}

int kv_pool_required_bytes(const kv_pool_desc* desc, int64_t* total_bytes, int64_t* tail_pad_bytes) {
  gtkv::Layout lay;
  const int rc = gtkv::compute_layout(desc, &lay);
  if (rc != KV_OK) return rc;
  if (total_bytes) *total_bytes = lay.total;
  if (tail_pad_bytes) *tail_pad_bytes = lay.tail_pad;
  return KV_OK;
}

int kv_pool_create(const kv_pool_desc* desc, void* raw_dev, int64_t raw_bytes, kv_pool_t** out) {
  if (out == nullptr) return KV_ERR_INVALID;
  *out = nullptr;
  gtkv::Layout lay;
  int rc = gtkv::compute_layout(desc, &lay);
  if (rc != KV_OK) return rc;
  if (raw_dev != nullptr) {
    if (!aligned16(raw_dev)) return KV_ERR_ALIGN;
    // build_mha_views: the last view must end inside the raw buffer.
    if (raw_bytes < lay.last_view_end) return KV_ERR_TAIL_PAD;
  }

  int dev = -1, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return failed_call();
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
    return failed_call();
  if (gtkv::prepare_gather() != cudaSuccess) return failed_call();
  if (raw_dev != nullptr) {
    // a borrowed buffer must be device (or managed) memory of this device:
    // anything else would only show up later, as a fault in a kernel
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, raw_dev) != cudaSuccess) {
      cudaGetLastError();  // a failed query leaves its error for the next cudaGetLastError: clear it
      return KV_ERR_INVALID;
    }
    if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) {
      if (a.device != dev) return KV_ERR_DEVICE;
    } else {
      return KV_ERR_INVALID;
    }
  }

  kv_pool* p = new (std::nothrow) kv_pool{};
  if (p == nullptr) return KV_ERR_INVALID;
  p->desc = *desc;
  p->lay = lay;
  p->device = dev;
  p->sm_count = sms;
  if (raw_dev == nullptr) {
    void* mem = nullptr;
    if (cudaMalloc(&mem, static_cast<size_t>(lay.alloc_bytes)) != cudaSuccess) {
      delete p;
      return failed_call();
    }
    p->raw = static_cast<uint8_t*>(mem);
    p->raw_bytes = lay.alloc_bytes;
    p->owns_raw = 1;
  } else {
    p->raw = static_cast<uint8_t*>(raw_dev);
    p->raw_bytes = raw_bytes;
    p->owns_raw = 0;
  }
  void* err = nullptr;
  if (cudaMalloc(&err, kErrWords * sizeof(int32_t)) != cudaSuccess ||
      cudaMemset(err, 0, kErrWords * sizeof(int32_t)) != cudaSuccess) {
    if (err) cudaFree(err);
    if (p->owns_raw) cudaFree(p->raw);
    delete p;
    return failed_call();
  }
  p->d_err = static_cast<int32_t*>(err);

  gtkv::DevPool& d = p->dev;
  d.base = reinterpret_cast<uint4*>(p->raw + desc->anchor_bytes);
  d.vpr = lay.R / 16;
  d.ps = desc->page_size;
  d.stride = lay.stride;
  d.n_rows = lay.n_rows;
  d.num_pages = desc->num_pages;
  d.blocks = static_cast<int32_t>(lay.blocks);
  d.kv_rows = static_cast<int32_t>(lay.kv_rows);
  d.ps_shift = ps_shift_of(desc->page_size);
  d.err = p->d_err;
  *out = p;
  return KV_OK;
}

int kv_pool_destroy(kv_pool_t* pool) {
  if (pool == nullptr) return KV_OK;
  int rc = KV_OK;
  if (cudaFree(pool->d_err) != cudaSuccess) rc = KV_ERR_CUDA;
  if (pool->owns_raw && cudaFree(pool->raw) != cudaSuccess) rc = KV_ERR_CUDA;
  delete pool;
  return rc;
}

int kv_pool_info(const kv_pool_t* pool, kv_pool_info_t* out) {
  if (pool == nullptr || out == nullptr) return KV_ERR_INVALID;
  out->raw_dev = pool->raw;
  out->raw_bytes = pool->raw_bytes;
  out->row_bytes = pool->lay.R;
  out->page_bytes = pool->lay.page_bytes;
  out->total_bytes = pool->lay.total;
  out->tail_pad_bytes = pool->lay.tail_pad;
  out->n_rows = pool->lay.n_rows;
  out->last_view_end = pool->lay.last_view_end;
  out->device = pool->device;
  out->owns_raw = pool->owns_raw;
  out->blocks_per_page = static_cast<int32_t>(pool->lay.blocks);
  out->latent_only = pool->desc.latent_only;
  return KV_OK;
}

int kv_translate(const kv_pool_t* pool, const int64_t* slots_dev, int64_t n, const int32_t* v2p_dev,
                 int64_t v2p_len, int32_t* ids_dev, kv_stream_t stream) {
  Range nvtx("kv_translate");
  int rc = enter(pool);
  if (rc != KV_OK) return rc;
  if (n < 0 || v2p_len < 0) return KV_ERR_INVALID;
  if (n == 0) return KV_OK;
  if (slots_dev == nullptr || ids_dev == nullptr || (v2p_dev == nullptr && v2p_len > 0)) return KV_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(slots_dev) & 7u) || (reinterpret_cast<uintptr_t>(ids_dev) & 3u))
    return KV_ERR_ALIGN;
  // ids (int32) must not overlap slots (int64): no in-place translation.
  const uintptr_t s0 = reinterpret_cast<uintptr_t>(slots_dev), s1 = s0 + 8 * static_cast<uintptr_t>(n);
  const uintptr_t i0 = reinterpret_cast<uintptr_t>(ids_dev), i1 = i0 + 4 * static_cast<uintptr_t>(n);
  if (i0 < s1 && s0 < i1) return KV_ERR_INVALID;
  return launched(gtkv::launch_translate(pool->dev, slots_dev, n, v2p_dev, v2p_len, ids_dev, pool->sm_count,
                                         as_stream(stream)));
}

int kv_store_layer(const kv_pool_t* pool, int32_t layer, const int32_t* ids_dev, int64_t n, const void* k_dev,
                   const void* v_dev, kv_stream_t stream) {
  Range nvtx("kv_store_layer");
  int rc = enter(pool);
  if (rc != KV_OK) return rc;
  if (n < 0 || layer < 0 || layer >= pool->desc.layer_num) return KV_ERR_INVALID;
  if (n == 0) return KV_OK;
  if (pool->desc.latent_only) v_dev = nullptr;  // MLA: no V rows
  if (ids_dev == nullptr || k_dev == nullptr || (v_dev == nullptr && !pool->desc.latent_only)) return KV_ERR_INVALID;
  if (!aligned16(k_dev) || !aligned16(v_dev) || (reinterpret_cast<uintptr_t>(ids_dev) & 3u)) return KV_ERR_ALIGN;
  return launched(gtkv::launch_store(pool->dev, layer, 1, ids_dev, n, k_dev, v_dev, pool->sm_count,
                                     as_stream(stream)));
}

int kv_store_all_layers(const kv_pool_t* pool, const int32_t* ids_dev, int64_t n, const void* k_all_dev,
                        const void* v_all_dev, kv_stream_t stream) {
  Range nvtx("kv_store_all_layers");
  int rc = enter(pool);
  if (rc != KV_OK) return rc;
  if (n < 0) return KV_ERR_INVALID;
  if (n == 0) return KV_OK;
  if (pool->desc.latent_only) v_all_dev = nullptr;
  if (ids_dev == nullptr || k_all_dev == nullptr || (v_all_dev == nullptr && !pool->desc.latent_only))
    return KV_ERR_INVALID;
  if (!aligned16(k_all_dev) || !aligned16(v_all_dev) || (reinterpret_cast<uintptr_t>(ids_dev) & 3u))
    return KV_ERR_ALIGN;
  return launched(gtkv::launch_store(pool->dev, 0, pool->desc.layer_num, ids_dev, n, k_all_dev, v_all_dev,
                                     pool->sm_count, as_stream(stream)));
}

int kv_translate_mapped(const kv_pool_t* pool, const int64_t* slots_dev, int64_t n, const int64_t* tmap_dev,
                        int64_t tmap_len, const int32_t* v2p_dev, int64_t v2p_len, int32_t* ids_dev,
                        kv_stream_t stream) {
  Range nvtx("kv_translate_mapped");
  int rc = enter(pool);
  if (rc != KV_OK) return rc;
  if (n < 0 || tmap_len < 0 || v2p_len < 0) return KV_ERR_INVALID;
  if (n == 0) return KV_OK;
  if (slots_dev == nullptr || ids_dev == nullptr || (tmap_dev == nullptr && tmap_len > 0) ||
      (v2p_dev == nullptr && v2p_len > 0))
    return KV_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(slots_dev) & 7u) || (reinterpret_cast<uintptr_t>(tmap_dev) & 7u) ||
      (reinterpret_cast<uintptr_t>(ids_dev) & 3u) || (reinterpret_cast<uintptr_t>(v2p_dev) & 3u))
    return KV_ERR_ALIGN;
  const uintptr_t s0 = reinterpret_cast<uintptr_t>(slots_dev), s1 = s0 + 8 * static_cast<uintptr_t>(n);
  const uintptr_t i0 = reinterpret_cast<uintptr_t>(ids_dev), i1 = i0 + 4 * static_cast<uintptr_t>(n);
  if (i0 < s1 && s0 < i1) return KV_ERR_INVALID;
  return launched(gtkv::launch_translate_mapped(pool->dev, slots_dev, n, tmap_dev, tmap_len, v2p_dev, v2p_len, ids_dev,
                                                pool->sm_count, as_stream(stream)));
}

static int store_slots(const kv_pool_t* pool, int32_t layer0, int32_t n_layers, const int64_t* slots_dev, int64_t n,
                       const int32_t* v2p_dev, int64_t v2p_len, const void* k_dev, const void* v_dev,
                       kv_stream_t stream) {
  int rc = enter(pool);
  if (rc != KV_OK) return rc;
  if (n < 0 || v2p_len < 0) return KV_ERR_INVALID;
  if (n == 0) return KV_OK;
  if (pool->desc.latent_only) v_dev = nullptr;
  if (slots_dev == nullptr || k_dev == nullptr || (v_dev == nullptr && !pool->desc.latent_only) ||
      (v2p_dev == nullptr && v2p_len > 0))
    return KV_ERR_INVALID;
  if (!aligned16(k_dev) || !aligned16(v_dev) || (reinterpret_cast<uintptr_t>(slots_dev) & 7u) ||
      (reinterpret_cast<uintptr_t>(v2p_dev) & 3u))
    return KV_ERR_ALIGN;
  return launched(gtkv::launch_store_slots(pool->dev, layer0, n_layers, slots_dev, n, v2p_dev, v2p_len, k_dev,
                                           v_dev, pool->sm_count, as_stream(stream)));
}

int kv_store_layer_slots(const kv_pool_t* pool, int32_t layer, const int64_t* slots_dev, int64_t n,
                         const int32_t* v2p_dev, int64_t v2p_len, const void* k_dev, const void* v_dev,
                         kv_stream_t stream) {
  Range nvtx("kv_store_layer_slots");
  if (pool != nullptr && (layer < 0 || layer >= pool->desc.layer_num)) return KV_ERR_INVALID;
  return store_slots(pool, layer, 1, slots_dev, n, v2p_dev, v2p_len, k_dev, v_dev, stream);
}

int kv_store_all_layers_slots(const kv_pool_t* pool, const int64_t* slots_dev, int64_t n, const int32_t* v2p_dev,
                              int64_t v2p_len, const void* k_all_dev, const void* v_all_dev, kv_stream_t stream) {
  Range nvtx("kv_store_all_layers_slots");
  if (pool == nullptr) return KV_ERR_INVALID;
  return store_slots(pool, 0, pool->desc.layer_num, slots_dev, n, v2p_dev, v2p_len, k_all_dev, v_all_dev, stream);
}

static int gather(const kv_pool_t* pool, int32_t layer, const void* plan_dev, const int32_t* block_table_dev,
                  bool kernel_facing, int32_t n_seqs, int32_t max_pages, const int32_t* seq_start_dev,
                  const int32_t* seq_len_dev, const int64_t* cu_out_dev, void* out_k_dev, void* out_v_dev,
                  int64_t out_rows, kv_stream_t stream) {
  int rc = enter(pool);
  if (rc != KV_OK) return rc;
  if (layer < 0 || layer >= pool->desc.layer_num || n_seqs < 0 || max_pages < 0 || out_rows < 0)
    return KV_ERR_INVALID;
  if (static_cast<int64_t>(n_seqs) * max_pages >= (int64_t(1) << 31)) return KV_ERR_INVALID;
  if (n_seqs == 0) return KV_OK;
  if (seq_len_dev == nullptr || cu_out_dev == nullptr || (block_table_dev == nullptr && max_pages > 0))
    return KV_ERR_INVALID;
  if (pool->desc.latent_only) out_v_dev = nullptr;  // MLA: no V output
  if (out_rows > 0 && (out_k_dev == nullptr || (out_v_dev == nullptr && !pool->desc.latent_only)))
    return KV_ERR_INVALID;
  if ((out_k_dev && !aligned16(out_k_dev)) || (out_v_dev && !aligned16(out_v_dev)) ||
      (reinterpret_cast<uintptr_t>(cu_out_dev) & 7u) || (reinterpret_cast<uintptr_t>(seq_len_dev) & 3u) ||
      (reinterpret_cast<uintptr_t>(block_table_dev) & 3u) || (reinterpret_cast<uintptr_t>(seq_start_dev) & 3u) ||
      (reinterpret_cast<uintptr_t>(plan_dev) & 3u))
    return KV_ERR_ALIGN;
  return launched(gtkv::launch_gather(pool->dev, layer, block_table_dev, n_seqs, max_pages, seq_start_dev,
                                      seq_len_dev, cu_out_dev, out_k_dev, out_v_dev, out_rows,
                                      static_cast<const int32_t*>(plan_dev), kernel_facing, pool->sm_count,
                                      as_stream(stream)));
}

int kv_gather_layer(const kv_pool_t* pool, int32_t layer, const int32_t* block_table_dev, int32_t n_seqs,
                    int32_t max_pages, const int32_t* seq_start_dev, const int32_t* seq_len_dev,
                    const int64_t* cu_out_dev, void* out_k_dev, void* out_v_dev, int64_t out_rows,
                    kv_stream_t stream) {
  Range nvtx("kv_gather_layer");
  return gather(pool, layer, nullptr, block_table_dev, false, n_seqs, max_pages, seq_start_dev, seq_len_dev,
                cu_out_dev, out_k_dev, out_v_dev, out_rows, stream);
}

int kv_gather_layer_kf(const kv_pool_t* pool, int32_t layer, const int32_t* kf_table_dev, int32_t n_seqs,
                       int32_t max_pages, const int32_t* seq_start_dev, const int32_t* seq_len_dev,
                       const int64_t* cu_out_dev, void* out_k_dev, void* out_v_dev, int64_t out_rows,
                       kv_stream_t stream) {
  Range nvtx("kv_gather_layer_kf");
  return gather(pool, layer, nullptr, kf_table_dev, true, n_seqs, max_pages, seq_start_dev, seq_len_dev,
                cu_out_dev, out_k_dev, out_v_dev, out_rows, stream);
}

int kv_gather_plan_bytes(const kv_pool_t* pool, int32_t n_seqs, int32_t max_pages, int64_t* plan_bytes) {
  if (pool == nullptr || plan_bytes == nullptr || n_seqs < 0 || max_pages < 0) return KV_ERR_INVALID;
  if (static_cast<int64_t>(n_seqs) * max_pages >= (int64_t(1) << 31)) return KV_ERR_INVALID;
  *plan_bytes = 4 * gtkv::plan_words(pool->dev, n_seqs, max_pages);
  return KV_OK;
}

static int gather_plan(const kv_pool_t* pool, const int32_t* block_table_dev, bool kernel_facing, int32_t n_seqs,
                       int32_t max_pages, const int32_t* seq_start_dev, const int32_t* seq_len_dev, void* plan_dev,
                       int64_t plan_bytes, kv_stream_t stream) {
  int rc = enter(pool);
  if (rc != KV_OK) return rc;
  int64_t need = 0;
  if ((rc = kv_gather_plan_bytes(pool, n_seqs, max_pages, &need)) != KV_OK) return rc;
  if (plan_dev == nullptr || plan_bytes < need) return KV_ERR_INVALID;
  if (n_seqs > 0 && (seq_len_dev == nullptr || (block_table_dev == nullptr && max_pages > 0)))
    return KV_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(plan_dev) & 3u) || (reinterpret_cast<uintptr_t>(seq_len_dev) & 3u) ||
      (reinterpret_cast<uintptr_t>(block_table_dev) & 3u) || (reinterpret_cast<uintptr_t>(seq_start_dev) & 3u))
    return KV_ERR_ALIGN;
  return launched(gtkv::launch_gather_plan(pool->dev, block_table_dev, n_seqs, max_pages, seq_start_dev,
                                           seq_len_dev, static_cast<int32_t*>(plan_dev), kernel_facing,
                                           pool->sm_count, as_stream(stream)));
}

int kv_gather_plan(const kv_pool_t* pool, const int32_t* block_table_dev, int32_t n_seqs, int32_t max_pages,
                   const int32_t* seq_start_dev, const int32_t* seq_len_dev, void* plan_dev, int64_t plan_bytes,
                   kv_stream_t stream) {
  Range nvtx("kv_gather_plan");
  return gather_plan(pool, block_table_dev, false, n_seqs, max_pages, seq_start_dev, seq_len_dev, plan_dev,
                     plan_bytes, stream);
}

int kv_gather_plan_kf(const kv_pool_t* pool, const int32_t* kf_table_dev, int32_t n_seqs, int32_t max_pages,
                      const int32_t* seq_start_dev, const int32_t* seq_len_dev, void* plan_dev, int64_t plan_bytes,
                      kv_stream_t stream) {
  Range nvtx("kv_gather_plan_kf");
  return gather_plan(pool, kf_table_dev, true, n_seqs, max_pages, seq_start_dev, seq_len_dev, plan_dev,
                     plan_bytes, stream);
}

static int gather_planned(const kv_pool_t* pool, int32_t layer, const void* plan_dev, int64_t plan_bytes,
                          const int32_t* block_table_dev, bool kernel_facing, int32_t n_seqs, int32_t max_pages,
                          const int32_t* seq_start_dev, const int32_t* seq_len_dev, const int64_t* cu_out_dev,
                          void* out_k_dev, void* out_v_dev, int64_t out_rows, kv_stream_t stream) {
  if (plan_dev == nullptr) return KV_ERR_INVALID;
  int64_t need = 0;
  const int rc = kv_gather_plan_bytes(pool, n_seqs, max_pages, &need);
  if (rc != KV_OK) return rc;
  if (plan_bytes < need) return KV_ERR_INVALID;  // the kernel reads up to `need` bytes of the plan
  return gather(pool, layer, plan_dev, block_table_dev, kernel_facing, n_seqs, max_pages, seq_start_dev,
                seq_len_dev, cu_out_dev, out_k_dev, out_v_dev, out_rows, stream);
}

int kv_gather_layer_planned(const kv_pool_t* pool, int32_t layer, const void* plan_dev, int64_t plan_bytes,
                            const int32_t* block_table_dev, int32_t n_seqs, int32_t max_pages,
                            const int32_t* seq_start_dev, const int32_t* seq_len_dev, const int64_t* cu_out_dev,
                            void* out_k_dev, void* out_v_dev, int64_t out_rows, kv_stream_t stream) {
  Range nvtx("kv_gather_layer_planned");
  return gather_planned(pool, layer, plan_dev, plan_bytes, block_table_dev, false, n_seqs, max_pages, seq_start_dev,
                        seq_len_dev, cu_out_dev, out_k_dev, out_v_dev, out_rows, stream);
}

int kv_gather_layer_planned_kf(const kv_pool_t* pool, int32_t layer, const void* plan_dev, int64_t plan_bytes,
                               const int32_t* kf_table_dev, int32_t n_seqs, int32_t max_pages,
                               const int32_t* seq_start_dev, const int32_t* seq_len_dev, const int64_t* cu_out_dev,
                               void* out_k_dev, void* out_v_dev, int64_t out_rows, kv_stream_t stream) {
  Range nvtx("kv_gather_layer_planned_kf");
  return gather_planned(pool, layer, plan_dev, plan_bytes, kf_table_dev, true, n_seqs, max_pages, seq_start_dev,
                        seq_len_dev, cu_out_dev, out_k_dev, out_v_dev, out_rows, stream);
}

int kv_move(const kv_pool_t* pool, const int32_t* src_ids_dev, const int32_t* dst_ids_dev, int64_t n,
            kv_stream_t stream) {
  Range nvtx("kv_move");
  int rc = enter(pool);
  if (rc != KV_OK) return rc;
  if (n < 0) return KV_ERR_INVALID;
  if (n == 0) return KV_OK;
  if (src_ids_dev == nullptr || dst_ids_dev == nullptr) return KV_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(src_ids_dev) & 3u) || (reinterpret_cast<uintptr_t>(dst_ids_dev) & 3u))
    return KV_ERR_ALIGN;
  return launched(gtkv::launch_move(pool->dev, src_ids_dev, dst_ids_dev, n, pool->sm_count, as_stream(stream)));
}

int kv_translate_block_table(const kv_pool_t* pool, const int32_t* virt_bt_dev, int32_t n_seqs, int32_t max_pages,
                             const int32_t* seq_len_dev, const int32_t* v2p_dev, int64_t v2p_len,
                             int32_t* out_bt_dev, kv_stream_t stream) {
  Range nvtx("kv_translate_block_table");
  int rc = enter(pool);
  if (rc != KV_OK) return rc;
  if (n_seqs < 0 || max_pages < 0 || v2p_len < 0) return KV_ERR_INVALID;
  if (n_seqs == 0 || max_pages == 0) return KV_OK;
  if (virt_bt_dev == nullptr || seq_len_dev == nullptr || out_bt_dev == nullptr || (v2p_dev == nullptr && v2p_len > 0))
    return KV_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(virt_bt_dev) & 3u) || (reinterpret_cast<uintptr_t>(out_bt_dev) & 3u) ||
      (reinterpret_cast<uintptr_t>(seq_len_dev) & 3u) || (reinterpret_cast<uintptr_t>(v2p_dev) & 3u))
    return KV_ERR_ALIGN;
  return launched(gtkv::launch_block_table(pool->dev, virt_bt_dev, n_seqs, max_pages, seq_len_dev, v2p_dev, v2p_len,
                                           out_bt_dev, pool->sm_count, as_stream(stream)));
}

int kv_pool_last_error(const kv_pool_t* pool, kv_stream_t stream, int32_t* dev_code) {
  Range nvtx("kv_pool_last_error");
  int rc = enter(pool);
  if (rc != KV_OK) return rc;
  if (dev_code == nullptr) return KV_ERR_INVALID;
  int32_t h = 0;
  cudaStream_t s = as_stream(stream);
  k_take_error<<<1, 1, 0, s>>>(pool->d_err);
  if (cudaGetLastError() != cudaSuccess) return KV_ERR_CUDA;
  if (cudaMemcpyAsync(&h, pool->d_err + 1, sizeof(h), cudaMemcpyDeviceToHost, s) != cudaSuccess) return KV_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return KV_ERR_CUDA;
  *dev_code = h;
  return KV_OK;
}

}  // extern "C"
