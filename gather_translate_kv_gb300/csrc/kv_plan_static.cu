// kv_gather_plan_noalloc: the page-major gather plan of kv_plan.cu, built
// without device memory from the caller beyond the plan itself.
//
// Some callers of this library cannot call cudaMalloc: code inside a host
// framework whose allocator reserved the device's memory at start-up and owns
// it, or a serving loop that must keep allocations (and the device-wide
// synchronization cudaMalloc and cudaFree may cause) out of its steady state.
// kv_gather_plan counts the entries of each page inside the caller's plan
// buffer; this variant counts in g_plan_counts, a fixed array in the
// library's device image, and copies the finished per-page offsets into the
// plan, so the plan matches kv_gather_plan's up to the order of the entries
// within one page.
//
// g_plan_counts holds kMaxPages + 1 int32 counters (256 KiB + 4 bytes); every
// GPU that loads the library keeps it until the process exits. All calls
// share it and it keeps the last call's contents, so each call clears the
// counters it uses first, on its own stream. Calls that overlap on the GPU
// (other streams, threads or pools on the same device) race on it.
#include <cuda.h>  // CUcontext and the driver's function types only: the functions are looked up at run time
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>
#include <stdint.h>

#include <mutex>

#include "kv_launch.h"
#include "kv_plan.cuh"
#include "kv_pool.h"
#include "kv_pool_internal.h"

namespace gtkv {
namespace {

constexpr int64_t kMaxPages = 65536;
constexpr int kMaxDevices = 128;

// One counter per page, then the total. In host code this name is only a
// stand-in for the array; kernels get its device address from counts_on().
static __device__ __align__(256) int32_t g_plan_counts[kMaxPages + 1];

// The array's address per device, with the id of the context it was looked
// up in: a context the runtime creates anew (after cudaDeviceReset, for
// instance) loads the module again, and the array may move.
struct CountsAddr {
  int32_t* ptr;
  unsigned long long ctx_id;
};
CountsAddr g_counts_addr[kMaxDevices] = {};
std::mutex g_counts_mu;

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);
CtxGetCurrentFn g_ctx_get_current = nullptr;
CtxGetIdFn g_ctx_get_id = nullptr;

// Process-unique id of the calling thread's current context (the driver
// never reuses one), or an error when the thread has none bound yet.
// Called with g_counts_mu held.
cudaError_t current_context_id(unsigned long long* id) {
  if (g_ctx_get_current == nullptr || g_ctx_get_id == nullptr) {
    void* f0 = nullptr;
    void* f1 = nullptr;
    cudaDriverEntryPointQueryResult q0, q1;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f0, 12000, cudaEnableDefault, &q0) != cudaSuccess ||
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &f1, 12000, cudaEnableDefault, &q1) != cudaSuccess ||
        q0 != cudaDriverEntryPointSuccess || q1 != cudaDriverEntryPointSuccess)
      return cudaErrorNotSupported;
    g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(f0);
    g_ctx_get_id = reinterpret_cast<CtxGetIdFn>(f1);
  }
  CUcontext ctx = nullptr;
  if (g_ctx_get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return cudaErrorDeviceUninitialized;
  return g_ctx_get_id(ctx, id) == CUDA_SUCCESS ? cudaSuccess : cudaErrorDeviceUninitialized;
}

// Device address of g_plan_counts on `device`, which must be current. Looked
// up with cudaGetSymbolAddress on the first call per device, and again only
// when the device's current context is not the one of the last lookup.
cudaError_t counts_on(int device, int32_t** out) {
  if (device < 0 || device >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_counts_mu);
  CountsAddr& c = g_counts_addr[device];
  unsigned long long ctx = 0;
  const bool have_ctx = current_context_id(&ctx) == cudaSuccess;
  if (c.ptr == nullptr || !have_ctx || ctx != c.ctx_id) {
    void* ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&ptr, g_plan_counts);  // binds the device's context if need be
    if (e != cudaSuccess) return e;
    if (!have_ctx && current_context_id(&ctx) != cudaSuccess) return cudaErrorDeviceUninitialized;
    c.ptr = static_cast<int32_t*>(ptr);
    c.ctx_id = ctx;
  }
  *out = c.ptr;
  return cudaSuccess;
}

__global__ void __launch_bounds__(kBlock) k_noalloc_count(DevPool p, const int32_t* __restrict__ bt,
                                                          int64_t n_entries, int32_t max_pages,
                                                          const int32_t* __restrict__ seq_start,
                                                          const int32_t* __restrict__ seq_len, int32_t* counts) {
  int bits = 0;
  const int64_t step = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < n_entries; e += step) {
    const int64_t b = plan_bucket(p, e, bt, max_pages, seq_start, seq_len, 1, bits);
    if (b >= 0) atomicAdd(counts + b, 1);
  }
  if (bits) atomicOr(p.err, bits);
}

// Counts -> start offsets (in place) and the plan header.
__global__ void __launch_bounds__(kScanThreads) k_noalloc_scan(int64_t n_pages, int32_t n_seqs, int32_t max_pages,
                                                               int32_t* counts, int32_t* __restrict__ plan) {
  scan_plan_counts(counts, n_pages, n_seqs, max_pages, 0, plan);
}

// Each entry takes the next position of its page; afterwards counts[b] is the
// end offset of page b, as in kv_gather_plan's plan.
__global__ void __launch_bounds__(kBlock) k_noalloc_scatter(DevPool p, const int32_t* __restrict__ bt,
                                                            int64_t n_entries, int32_t max_pages,
                                                            const int32_t* __restrict__ seq_start,
                                                            const int32_t* __restrict__ seq_len, int32_t* counts,
                                                            int32_t* __restrict__ entries) {
  int bits = 0;
  const int64_t step = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < n_entries; e += step) {
    const int64_t b = plan_bucket(p, e, bt, max_pages, seq_start, seq_len, 1, bits);
    if (b >= 0) plan_place(entries, counts + b, n_entries, e, bits);
  }
  if (bits & KV_DEV_ERR_TABLE) atomicOr(p.err, KV_DEV_ERR_TABLE);
}

}  // namespace
}  // namespace gtkv

extern "C" int kv_gather_plan_noalloc(const kv_pool_t* pool, const int32_t* block_table_dev, int32_t n_seqs,
                                      int32_t max_pages, const int32_t* seq_start_dev, const int32_t* seq_len_dev,
                                      void* plan_dev, int64_t plan_bytes, kv_stream_t stream) {
  using namespace gtkv;
  if (pool == nullptr) return KV_ERR_INVALID;
  int device = -1;
  if (cudaGetDevice(&device) != cudaSuccess) return KV_ERR_CUDA;
  if (device != pool->device) return KV_ERR_DEVICE;
  int64_t need = 0;
  int rc = kv_gather_plan_bytes(pool, n_seqs, max_pages, &need);
  if (rc != KV_OK) return rc;
  const int64_t n_pages = pool->dev.num_pages;
  if (n_pages > kMaxPages) return KV_ERR_CAPACITY;
  if (plan_dev == nullptr || plan_bytes < need) return KV_ERR_INVALID;
  if (n_seqs > 0 && (seq_len_dev == nullptr || (block_table_dev == nullptr && max_pages > 0)))
    return KV_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(plan_dev) & 3u) || (reinterpret_cast<uintptr_t>(seq_len_dev) & 3u) ||
      (reinterpret_cast<uintptr_t>(block_table_dev) & 3u) || (reinterpret_cast<uintptr_t>(seq_start_dev) & 3u))
    return KV_ERR_ALIGN;
  int32_t* counts = nullptr;
  if (counts_on(device, &counts) != cudaSuccess) {
    cudaGetLastError();  // a failed look-up must not surface as the status of a later launch
    return KV_ERR_CUDA;
  }

  nvtxRangePushA("kv_gather_plan_noalloc");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int32_t* plan = static_cast<int32_t*>(plan_dev);
  const int64_t n_entries = static_cast<int64_t>(n_seqs) * max_pages;
  const size_t count_bytes = sizeof(int32_t) * static_cast<size_t>(n_pages + 1);
  const unsigned grid = grid_for(k_noalloc_count, (n_entries + 31) / 32, pool->sm_count);
  cudaError_t e = cudaMemsetAsync(counts, 0, count_bytes, s);  // the last call's counts are still there
  if (e == cudaSuccess) {
    k_noalloc_count<<<grid, kBlock, 0, s>>>(pool->dev, block_table_dev, n_entries, max_pages, seq_start_dev,
                                            seq_len_dev, counts);
    k_noalloc_scan<<<1, kScanThreads, 0, s>>>(n_pages, n_seqs, max_pages, counts, plan);
    k_noalloc_scatter<<<grid, kBlock, 0, s>>>(pool->dev, block_table_dev, n_entries, max_pages, seq_start_dev,
                                              seq_len_dev, counts, plan + kPlanHeaderWords + n_pages + 1);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) e = cudaMemcpyAsync(plan + kPlanHeaderWords, counts, count_bytes, cudaMemcpyDeviceToDevice, s);
  nvtxRangePop();
  if (e == cudaSuccess) return KV_OK;
  cudaGetLastError();  // reported here, not again by a later launch
  return KV_ERR_CUDA;
}
