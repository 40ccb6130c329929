// Host launchers of the pool kernels, one translation unit each; every one
// enqueues its kernel on `s` and returns the launch status.
#pragma once

#include "kv_common.cuh"

namespace gtkv {

cudaError_t launch_translate(const DevPool& p, const int64_t* slots, int64_t n, const int32_t* v2p,
                             int64_t v2p_len, int32_t* ids, int sm_count, cudaStream_t s);
cudaError_t launch_store(const DevPool& p, int32_t layer0, int32_t n_layers, const int32_t* ids, int64_t n,
                         const void* k, const void* v, int sm_count, cudaStream_t s);
cudaError_t launch_store_slots(const DevPool& p, int32_t layer0, int32_t n_layers, const int64_t* slots, int64_t n,
                               const int32_t* v2p, int64_t v2p_len, const void* k, const void* v, int sm_count,
                               cudaStream_t s);
// Per-device set-up of the gather kernels (their shared-memory limit); called by kv_pool_create.
cudaError_t prepare_gather();
cudaError_t launch_gather(const DevPool& p, int32_t layer, const int32_t* bt, int32_t n_seqs, int32_t max_pages,
                          const int32_t* seq_start, const int32_t* seq_len, const int64_t* cu, void* out_k,
                          void* out_v, int64_t out_rows, const int32_t* plan, bool kernel_facing, int sm_count,
                          cudaStream_t s);
// Page-major gather plan (kv_plan.cu): its size in int32 words, and its build.
// kernel_facing: the table holds kernel-facing entries phys * 2L.
int64_t plan_words(const DevPool& p, int32_t n_seqs, int32_t max_pages);
cudaError_t launch_gather_plan(const DevPool& p, const int32_t* bt, int32_t n_seqs, int32_t max_pages,
                               const int32_t* seq_start, const int32_t* seq_len, int32_t* plan, bool kernel_facing,
                               int sm_count, cudaStream_t s);
cudaError_t launch_translate_mapped(const DevPool& p, const int64_t* slots, int64_t n, const int64_t* tmap,
                                    int64_t tmap_len, const int32_t* v2p, int64_t v2p_len, int32_t* ids, int sm_count,
                                    cudaStream_t s);
cudaError_t launch_block_table(const DevPool& p, const int32_t* virt, int32_t n_seqs, int32_t max_pages,
                               const int32_t* seq_len, const int32_t* v2p, int64_t v2p_len, int32_t* out,
                               int sm_count, cudaStream_t s);
cudaError_t launch_move(const DevPool& p, const int32_t* src, const int32_t* dst, int64_t n, int sm_count,
                        cudaStream_t s);

}  // namespace gtkv
