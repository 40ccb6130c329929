/*
 * A plain C99 caller of the library: it includes only include/kv_pool.h and
 * links libgtkv.so (plus the CUDA runtime for its own buffers).
 *
 *   c_abi_roundtrip        host-only checks: sizes and start-up gates
 *   c_abi_roundtrip gpu    + a translate -> store -> gather round trip on the
 *                          current device, with the library owning the pool,
 *                          the same gather through a page-major plan, and
 *                          through a kernel-facing table built from virtual
 *                          pages and a page map
 *
 * Pool: 2 layers, 2 KV heads, head_dim 8, bf16 (R = 32 bytes), page size 4,
 * 64 pages. Exit status 0 = every check passed.
 */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "kv_pool.h"

#ifdef WITH_CUDA
#include <cuda_runtime_api.h>
#endif

static int fail(const char* what, int rc) {
  fprintf(stderr, "FAILED: %s (%d)\n", what, rc);
  return 1;
}

static kv_pool_desc tiny(void) {
  kv_pool_desc d;
  memset(&d, 0, sizeof d);
  d.layer_num = 2;
  d.head_num = 2;
  d.head_dim = 8;
  d.v_head_dim = 8;
  d.itemsize = 2;
  d.page_size = 4;
  d.num_pages = 64;
  return d;
}

static int host_checks(void) {
  kv_pool_desc d = tiny();
  int64_t total = 0, pad = 0;
  int rc = kv_pool_required_bytes(&d, &total, &pad);
  /* page_bytes = 4 * 2L * 32 = 512; total = 64 * 512; tail pad = one envelope */
  if (rc != KV_OK || total != 32768 || pad != 512) return fail("required bytes", rc);
  d.v_head_dim = 16;
  if ((rc = kv_pool_required_bytes(&d, NULL, NULL)) != KV_ERR_ASYMMETRIC) return fail("asymmetric gate", rc);
  d = tiny();
  d.layer_num = 80;
  d.head_num = 1;
  d.head_dim = 64;
  d.v_head_dim = 64;
  d.itemsize = 1;
  d.page_size = 256;
  d.num_pages = 52429; /* 52429 * 2 * 80 * 256 >= 2^31 */
  if ((rc = kv_pool_required_bytes(&d, NULL, NULL)) != KV_ERR_ID_BOUND) return fail("id bound gate", rc);
  d.num_pages = 52428;
  if ((rc = kv_pool_required_bytes(&d, NULL, NULL)) != KV_OK) return fail("largest legal pool", rc);
  d = tiny();
  kv_pool_t* pool = NULL;
  /* a buffer one byte short of the last view's end (anchor + (2L-1)*ps*R + n_rows*R = 33152) */
  rc = kv_pool_create(&d, (void*)(uintptr_t)(1u << 20), 33151, &pool);
  if (rc != KV_ERR_TAIL_PAD || pool != NULL) return fail("tail pad gate", rc);
  if (strcmp(kv_status_string(KV_ERR_ALIGN), "KV_ERR_ALIGN") != 0) return fail("status string", 0);
  return 0;
}

#ifdef WITH_CUDA
static int gpu_roundtrip(void) {
  kv_pool_desc d = tiny();
  kv_pool_t* pool = NULL;
  int rc = kv_pool_create(&d, NULL, 0, &pool); /* the library allocates the buffer */
  if (rc != KV_OK) return fail("create", rc);
  enum { N = 16, R = 32, PAGES = 4 };
  int64_t slots[N];
  int32_t table[PAGES] = {7, 3, 12, 40}; /* the sequence's pages */
  for (int j = 0; j < N; ++j) slots[j] = (int64_t)table[j / 4] * 4 + j % 4;
  uint8_t k[N * R], v[N * R], gk[N * R], gv[N * R];
  for (int i = 0; i < N * R; ++i) {
    k[i] = (uint8_t)(i * 7 + 1);
    v[i] = (uint8_t)(i * 13 + 5);
  }
  int32_t seq_len = N;
  int64_t cu[2] = {0, N};
  int64_t* d_slots;
  int32_t *d_ids, *d_table, *d_len;
  int64_t* d_cu;
  void *d_k, *d_v, *d_gk, *d_gv;
  if (cudaMalloc((void**)&d_slots, sizeof slots) || cudaMalloc((void**)&d_ids, N * 4) ||
      cudaMalloc((void**)&d_table, sizeof table) || cudaMalloc((void**)&d_len, 4) || cudaMalloc((void**)&d_cu, 16) ||
      cudaMalloc(&d_k, sizeof k) || cudaMalloc(&d_v, sizeof v) || cudaMalloc(&d_gk, sizeof gk) ||
      cudaMalloc(&d_gv, sizeof gv))
    return fail("cudaMalloc", 0);
  cudaMemcpy(d_slots, slots, sizeof slots, cudaMemcpyHostToDevice);
  cudaMemcpy(d_table, table, sizeof table, cudaMemcpyHostToDevice);
  cudaMemcpy(d_len, &seq_len, 4, cudaMemcpyHostToDevice);
  cudaMemcpy(d_cu, cu, sizeof cu, cudaMemcpyHostToDevice);
  cudaMemcpy(d_k, k, sizeof k, cudaMemcpyHostToDevice);
  cudaMemcpy(d_v, v, sizeof v, cudaMemcpyHostToDevice);
  if ((rc = kv_translate(pool, d_slots, N, NULL, 0, d_ids, NULL)) != KV_OK) return fail("translate", rc);
  if ((rc = kv_store_layer(pool, 1, d_ids, N, d_k, d_v, NULL)) != KV_OK) return fail("store", rc);
  if ((rc = kv_gather_layer(pool, 1, d_table, 1, PAGES, NULL, d_len, d_cu, d_gk, d_gv, N, NULL)) != KV_OK)
    return fail("gather", rc);
  int32_t bits = -1;
  if ((rc = kv_pool_last_error(pool, NULL, &bits)) != KV_OK || bits != 0) return fail("device errors", bits);
  int32_t ids[N];
  cudaMemcpy(ids, d_ids, sizeof ids, cudaMemcpyDeviceToHost);
  cudaMemcpy(gk, d_gk, sizeof gk, cudaMemcpyDeviceToHost);
  cudaMemcpy(gv, d_gv, sizeof gv, cudaMemcpyDeviceToHost);
  /* kernel_id = page * (ps * 2L) + offset = page * 16 + offset */
  for (int j = 0; j < N; ++j)
    if (ids[j] != table[j / 4] * 16 + j % 4) return fail("kernel id", ids[j]);
  if (memcmp(gk, k, sizeof k) != 0 || memcmp(gv, v, sizeof v) != 0) return fail("round trip bytes", 0);

  /* the same gather through a page-major plan: 4 * (4 + 64 + 1 + 1 * 4) bytes */
  int64_t plan_bytes = 0;
  if ((rc = kv_gather_plan_bytes(pool, 1, PAGES, &plan_bytes)) != KV_OK || plan_bytes != 4 * (4 + 64 + 1 + 4))
    return fail("plan bytes", rc);
  void* d_plan;
  if (cudaMalloc(&d_plan, (size_t)plan_bytes)) return fail("cudaMalloc plan", 0);
  cudaMemset(d_gk, 0, sizeof gk);
  cudaMemset(d_gv, 0, sizeof gv);
  if ((rc = kv_gather_plan(pool, d_table, 1, PAGES, NULL, d_len, d_plan, plan_bytes, NULL)) != KV_OK)
    return fail("plan", rc);
  if ((rc = kv_gather_layer_planned(pool, 1, d_plan, plan_bytes - 4, d_table, 1, PAGES, NULL, d_len, d_cu, d_gk,
                                    d_gv, N, NULL)) != KV_ERR_INVALID)
    return fail("short plan buffer accepted", rc);
  if ((rc = kv_gather_layer_planned(pool, 1, d_plan, plan_bytes, d_table, 1, PAGES, NULL, d_len, d_cu, d_gk, d_gv,
                                    N, NULL)) != KV_OK)
    return fail("planned gather", rc);
  if ((rc = kv_pool_last_error(pool, NULL, &bits)) != KV_OK || bits != 0) return fail("device errors (plan)", bits);
  cudaMemcpy(gk, d_gk, sizeof gk, cudaMemcpyDeviceToHost);
  cudaMemcpy(gv, d_gv, sizeof gv, cudaMemcpyDeviceToHost);
  if (memcmp(gk, k, sizeof k) != 0 || memcmp(gv, v, sizeof v) != 0) return fail("planned round trip bytes", 0);

  /* the read path through a kernel-facing table: virtual pages 0..3 map to
   * the physical pages above; the table build writes phys * 2L = phys * 4 */
  int32_t virt[PAGES] = {0, 1, 2, 3}, v2p[PAGES] = {7, 3, 12, 40}, kf[PAGES];
  int32_t *d_virt, *d_v2p, *d_kf;
  if (cudaMalloc((void**)&d_virt, sizeof virt) || cudaMalloc((void**)&d_v2p, sizeof v2p) ||
      cudaMalloc((void**)&d_kf, sizeof kf))
    return fail("cudaMalloc kf", 0);
  cudaMemcpy(d_virt, virt, sizeof virt, cudaMemcpyHostToDevice);
  cudaMemcpy(d_v2p, v2p, sizeof v2p, cudaMemcpyHostToDevice);
  if ((rc = kv_translate_block_table(pool, d_virt, 1, PAGES, d_len, d_v2p, PAGES, d_kf, NULL)) != KV_OK)
    return fail("kernel-facing table", rc);
  cudaMemcpy(kf, d_kf, sizeof kf, cudaMemcpyDeviceToHost);
  for (int i = 0; i < PAGES; ++i)
    if (kf[i] != table[i] * 4) return fail("kernel-facing entry", kf[i]);
  cudaMemset(d_gk, 0, sizeof gk);
  cudaMemset(d_gv, 0, sizeof gv);
  if ((rc = kv_gather_layer_kf(pool, 1, d_kf, 1, PAGES, NULL, d_len, d_cu, d_gk, d_gv, N, NULL)) != KV_OK)
    return fail("kernel-facing gather", rc);
  cudaMemcpy(gk, d_gk, sizeof gk, cudaMemcpyDeviceToHost);
  cudaMemcpy(gv, d_gv, sizeof gv, cudaMemcpyDeviceToHost);
  if (memcmp(gk, k, sizeof k) != 0 || memcmp(gv, v, sizeof v) != 0) return fail("kernel-facing round trip", 0);
  cudaMemset(d_gk, 0, sizeof gk);
  cudaMemset(d_gv, 0, sizeof gv);
  if ((rc = kv_gather_plan_kf(pool, d_kf, 1, PAGES, NULL, d_len, d_plan, plan_bytes, NULL)) != KV_OK)
    return fail("kernel-facing plan", rc);
  if ((rc = kv_gather_layer_planned_kf(pool, 1, d_plan, plan_bytes, d_kf, 1, PAGES, NULL, d_len, d_cu, d_gk, d_gv,
                                       N, NULL)) != KV_OK)
    return fail("planned kernel-facing gather", rc);
  if ((rc = kv_pool_last_error(pool, NULL, &bits)) != KV_OK || bits != 0) return fail("device errors (kf)", bits);
  cudaMemcpy(gk, d_gk, sizeof gk, cudaMemcpyDeviceToHost);
  cudaMemcpy(gv, d_gv, sizeof gv, cudaMemcpyDeviceToHost);
  if (memcmp(gk, k, sizeof k) != 0 || memcmp(gv, v, sizeof v) != 0) return fail("planned kf round trip", 0);
  cudaFree(d_virt);
  cudaFree(d_v2p);
  cudaFree(d_kf);
  cudaFree(d_plan);
  cudaFree(d_slots);
  cudaFree(d_ids);
  cudaFree(d_table);
  cudaFree(d_len);
  cudaFree(d_cu);
  cudaFree(d_k);
  cudaFree(d_v);
  cudaFree(d_gk);
  cudaFree(d_gv);
  if ((rc = kv_pool_destroy(pool)) != KV_OK) return fail("destroy", rc);
  return 0;
}
#endif

int main(int argc, char** argv) {
  if (host_checks() != 0) return 1;
  if (argc > 1 && strcmp(argv[1], "gpu") == 0) {
#ifdef WITH_CUDA
    if (gpu_roundtrip() != 0) return 2;
#else
    return fail("built without CUDA", 0);
#endif
  }
  printf("c abi: ok\n");
  return 0;
}
