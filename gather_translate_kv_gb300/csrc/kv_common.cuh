// Shared device-side pieces of the page-major KV pool kernels (sm_103a).
//
// Every kernel here is a row mover: a row is R = H*D*itemsize bytes (one
// token's K or V for one layer), copied as R/16 16-byte vectors. G lanes of a
// warp cooperate on one row (G = min(32, R/16) for the common power-of-two
// rows; 8 lanes x 9 vectors for 1152-byte MLA latents), each lane holding
// VPL vectors of it; a warp thus covers 32/G rows
// per wave, and U waves are loaded into registers before any is stored so
// that every lane keeps several 16-byte loads in flight. All byte offsets are
// 64-bit: a pool reaches 1.3e11 bytes while ids stay below 2^31.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <utility>
#include <vector>

#include "kv_layout.h"
#include "kv_pool.h"

namespace gtkv {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kBlock = 256;  // threads per block for every row-moving kernel

// Device view of a pool, passed by value to every kernel.
struct DevPool {
  uint4* base;        // raw + anchor (16-byte aligned)
  int64_t vpr;        // 16-byte vectors per row, R / 16
  int64_t ps;         // page size
  int64_t stride;     // rows per page envelope, ps * 2L
  int64_t n_rows;     // num_pages * 2L * ps
  int64_t num_pages;  // P
  int32_t blocks;     // row-blocks per page: 2L, or L for an MLA pool
  int32_t kv_rows;    // rows per layer per token: 2 (K then V) or 1 (MLA latent)
  int32_t ps_shift;   // log2(ps) when ps is a power of two, else -1
  int32_t* err;       // device error word (KV_DEV_ERR_* bits)
};

__device__ __forceinline__ int64_t div_ps(const DevPool& p, int64_t j) {
  return p.ps_shift >= 0 ? (j >> p.ps_shift) : j / p.ps;
}

// Token slot -> kernel-facing id, as translate_kv_loc_for_kernel computes it
// (prhub report on sglang PR #34602, 关键源码片段 multi_ended_allocator.py):
// page = t / ps, off = t % ps, phys = v2p[page] when a page map is given,
// id = phys * (ps * 2L) + off, and 0 (the page-0 sink) for a negative slot or
// a negative phys. A page index past the map or a phys >= P also gives 0 and
// ORs an error bit into `bits`.
__device__ __forceinline__ int64_t slot_to_id(const DevPool& p, int64_t t, const int32_t* __restrict__ v2p,
                                              int64_t v2p_len, int& bits) {
  if (t < 0) return 0;
  const int64_t page = div_ps(p, t);
  const int64_t off = t - page * p.ps;
  int64_t phys = page;
  if (v2p != nullptr) {
    if (page >= v2p_len) {
      bits |= KV_DEV_ERR_V2P;
      return 0;
    }
    phys = __ldg(v2p + page);
  }
  if (phys < 0) return 0;
  if (phys >= p.num_pages) {
    bits |= KV_DEV_ERR_ROW;
    return 0;
  }
  return phys * p.stride + off;
}

// ---- 16-byte loads / stores with explicit cache behaviour ---------------

enum : int {
  kLdNc = 0,      // read-only for the whole kernel: non-coherent path, no L1 allocation
  kLdPlain = 1,   // buffer is also written by the kernel (move): coherent load, no L1 allocation
  kLdNcKeep = 2,  // as kLdNc, and ask L2 to keep the line (evict_last): rows other warps re-read
  kLdNcFirst = 3, // as kLdNc, and let L2 drop the line first (evict_first): rows read once
  kLdNcPf = 4,    // as kLdNc, with a 256-byte L2 prefetch hint
};
enum : int {
  kStPlain = 0,   // write-back store
  kStStream = 1,  // st.cs: streaming store for outputs the kernel never reads back
  kStFirst = 2,   // write-back store with an L2 evict_first hint
};

// L2 cache-policy operands for the .L2::cache_hint forms.
struct L2Policy {
  uint64_t keep;   // evict_last
  uint64_t first;  // evict_first
};

__device__ __forceinline__ L2Policy make_l2_policy() {
  L2Policy c;
  asm("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(c.keep));
  asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(c.first));
  return c;
}

template <int LD>
__device__ __forceinline__ uint4 ld16(const uint4* p, const L2Policy& pol) {
  uint4 v;
  if constexpr (LD == kLdNc) {
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
  } else if constexpr (LD == kLdNcKeep) {
    asm("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p), "l"(pol.keep));
  } else if constexpr (LD == kLdNcFirst) {
    asm("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p), "l"(pol.first));
  } else if constexpr (LD == kLdNcPf) {
    asm("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
  } else {
    asm volatile("ld.global.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p)
                 : "memory");
  }
  return v;
}

template <int ST>
__device__ __forceinline__ void st16(uint4* p, const uint4& v, const L2Policy& pol) {
  if constexpr (ST == kStStream) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
  } else if constexpr (ST == kStFirst) {
    asm volatile("st.global.L1::no_allocate.L2::cache_hint.v4.u32 [%0], {%1,%2,%3,%4}, %5;" ::"l"(p), "r"(v.x),
                 "r"(v.y), "r"(v.z), "r"(v.w), "l"(pol.first)
                 : "memory");
  } else {
    asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
  }
}

// ---- copy N rows, all loads before all stores ------------------------------
//
// src[i]/dst[i] point at the first vector of row i (not yet offset by the
// lane); go[i] says whether row i is copied. With VPL > 0 the row holds
// exactly G*VPL vectors and lane g copies vectors g, g+G, ...; with VPL == 0
// (rows of any other size, G == 32) the row has vpr vectors and is copied in
// chunks of 4 vectors per lane.
template <int G, int VPL, int N, int LD, int ST>
__device__ __forceinline__ void copy_rows(const uint4* const (&src)[N], uint4* const (&dst)[N],
                                          const bool (&go)[N], int g, int64_t vpr, const L2Policy& pol) {
  if constexpr (VPL > 0) {
    uint4 buf[N][VPL];
#pragma unroll
    for (int i = 0; i < N; ++i)
      if (go[i]) {
#pragma unroll
        for (int v = 0; v < VPL; ++v) buf[i][v] = ld16<LD>(src[i] + g + v * G, pol);
      }
#pragma unroll
    for (int i = 0; i < N; ++i)
      if (go[i]) {
#pragma unroll
        for (int v = 0; v < VPL; ++v) st16<ST>(dst[i] + g + v * G, buf[i][v], pol);
      }
  } else {
    static_assert(G == 32, "dynamic rows use whole warps");
#pragma unroll 1
    for (int i = 0; i < N; ++i) {
      if (!go[i]) continue;
#pragma unroll 1
      for (int64_t c0 = 0; c0 < vpr; c0 += 4 * 32) {
        uint4 buf[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int64_t c = c0 + g + 32 * k;
          if (c < vpr) buf[k] = ld16<LD>(src[i] + c, pol);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int64_t c = c0 + g + 32 * k;
          if (c < vpr) st16<ST>(dst[i] + c, buf[k], pol);
        }
      }
    }
  }
}

// Cache behaviour and depth of each kernel: the measured choices on GB300.
// Gather: block-table pages are often shared by many sequences (common
// prefixes), so its reads ask L2 to keep lines (evict_last) and its output,
// which it never re-reads, is streamed (st.cs); on the decode workload this
// was worth ~2.5% over plain reads, and neutral where pages are read once.
#ifndef GTKV_GATHER_LD
#define GTKV_GATHER_LD kLdNcKeep
#endif
#ifndef GTKV_GATHER_ST
#define GTKV_GATHER_ST kStStream
#endif
#ifndef GTKV_STORE_LD
#define GTKV_STORE_LD kLdNc
#endif
#ifndef GTKV_STORE_ST
#define GTKV_STORE_ST kStPlain
#endif
#ifndef GTKV_MOVE_ST
#define GTKV_MOVE_ST kStPlain
#endif
// 16-byte vectors each lane keeps in flight (loads issued before stores)
#ifndef GTKV_STORE_VEC
#define GTKV_STORE_VEC 16
#endif
#ifndef GTKV_MOVE_VEC
#define GTKV_MOVE_VEC 8
#endif

// Row geometry chosen on the host from R/16; the list of instantiations.
enum class RowKind { V4, V8, V16, V32, V64, V72, V96, V128, V256, Dyn };

inline RowKind row_kind(int64_t vpr) {
  switch (vpr) {
    case 4: return RowKind::V4;
    case 8: return RowKind::V8;
    case 16: return RowKind::V16;
    case 32: return RowKind::V32;
    case 64: return RowKind::V64;
    case 72: return RowKind::V72;   // 1152-byte rows: an MLA latent of 576 bf16
    case 96: return RowKind::V96;   // 1536-byte rows
    case 128: return RowKind::V128;
    case 256: return RowKind::V256;
    default: return RowKind::Dyn;
  }
}

// Calls f.template operator()<G, VPL>() for the row kind.
template <class F>
inline cudaError_t dispatch_row(int64_t vpr, F&& f) {
  switch (row_kind(vpr)) {
    case RowKind::V4: return f.template operator()<4, 1>();
    case RowKind::V8: return f.template operator()<8, 1>();
    case RowKind::V16: return f.template operator()<16, 1>();
    case RowKind::V32: return f.template operator()<32, 1>();
    case RowKind::V64: return f.template operator()<32, 2>();
    case RowKind::V72: return f.template operator()<8, 9>();
    case RowKind::V96: return f.template operator()<32, 3>();
    case RowKind::V128: return f.template operator()<32, 4>();
    case RowKind::V256: return f.template operator()<32, 8>();
    default: return f.template operator()<32, 0>();
  }
}

// Blocks per SM a kernel reaches at kBlock threads, looked up once per kernel.
// The cache is keyed by the kernel's address: the instances of one template
// share a function-pointer type but not their register counts.
template <class K>
inline int blocks_per_sm(K kernel) {
  static std::mutex mu;
  static std::vector<std::pair<const void*, int>> cache;
  const void* key = reinterpret_cast<const void*>(kernel);
  std::lock_guard<std::mutex> lock(mu);
  for (const auto& e : cache)
    if (e.first == key) return e.second;
  int nb = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kernel, kBlock, 0) != cudaSuccess || nb < 1) nb = 1;
  cache.emplace_back(key, nb);
  return nb;
}

// Grid for `warps_needed` warps of work, capped at one full wave of resident
// blocks (the kernels loop grid-stride over the rest).
template <class K>
inline unsigned grid_for(K kernel, int64_t warps_needed, int sm_count) {
  const int64_t per_block = kBlock / 32;
  int64_t blocks = (warps_needed + per_block - 1) / per_block;
  const int64_t cap = static_cast<int64_t>(sm_count) * blocks_per_sm(kernel);
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return static_cast<unsigned>(blocks);
}

}  // namespace gtkv
