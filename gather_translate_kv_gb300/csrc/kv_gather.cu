// K4: block-table gather of one layer into packed [rows, H, D] K and V.
// Source: prhub report on sglang PR #34602, 功能与动机 -- with dense per-layer
// views every layer's K/V is read through one contiguous tensor and one shared
// block table -- and build_mha_views' view arithmetic (关键源码片段
// layout/page_major.py): token (page p, offset o) of layer l is K-view row
// p*ps*2L + o + 2l*ps, and its V row follows ps rows later.
//
// In an MLA pool (one latent row per layer, L row-blocks per page) layer l is
// block l and there is no V output.
//
// The block table is the work list. Entry (s, k) covers tokens
// [k*ps, (k+1)*ps) of sequence s; clipped to the window [start_s, len_s) it is
// a run of consecutive pool rows (one page's block 2l, then the same run in
// block 2l+1 for V) that lands on consecutive output rows cu_out[s] + j -
// start_s. So the gather is a set of contiguous copies: each run is cut into
// chunks of about 4 KiB; a warp works out the runs of up to 8 consecutive
// chunks at once (one per lane), then copies them in turn, K and V bytes as 16-byte
// vectors, all loads of a round issued before its stores. No
// search and no host synchronization: the item space is n_seqs x max_pages x
// chunks_per_page, and an entry outside a sequence's window is an empty item.
//
// Where one page's rows of a layer fit in 72 KiB of shared memory, gathers take
// the fan-out form instead (k_gather_fan, below): a block stages each page it
// needs once in shared memory and bulk-copies it to its readers -- with a
// page-major plan over a table of at least num_pages entries, the readers of
// a page among its two plan positions; otherwise a single table entry.
#include "kv_bulk.cuh"
#include "kv_launch.h"
#include "kv_plan.cuh"

namespace gtkv {

namespace {

#ifndef GTKV_GATHER_CHUNK
#define GTKV_GATHER_CHUNK 4096  // bytes of K (and of V) one warp copies per item
#endif
#ifndef GTKV_GATHER_MAX_BATCH
#define GTKV_GATHER_MAX_BATCH 8  // consecutive items a warp takes at once (1..32)
#endif
#ifndef GTKV_GATHER_CHV
#define GTKV_GATHER_CHV 8  // 16-byte vectors of K (and as many of V) each lane keeps in flight
#endif
// Latent rows of 1152 bytes (the 576-element bf16 latent of DeepSeek-like
// MLA pools, 72 vectors) fit 7 to a round of 32 x 16 vectors, so a 64-row
// page takes 10 rounds, the last one for a single row. Rounds whose vectors
// hold whole rows do better, measured on the 128 x 4096-token MLA gather:
// in table order rounds of 32 x 18 vectors (8 rows) take it from 184 to
// 176 us; the planned gather is best with rounds of 32 x 9 vectors (4 rows,
// 80 registers: 3 blocks per SM), 154 -> 144 us (18-vector rounds spill
// there and were slower, 164 us).
#ifndef GTKV_GATHER_V72
#define GTKV_GATHER_V72 1
#endif
#ifndef GTKV_GATHER_V72_TABLE_CHV
#define GTKV_GATHER_V72_TABLE_CHV 18  // vectors per lane per round, table order (a multiple of 9)
#endif
#ifndef GTKV_GATHER_V72_PLANNED_CHV
#define GTKV_GATHER_V72_PLANNED_CHV 9  // vectors per lane per round, page-major plan (a multiple of 9)
#endif
// Blocks per SM the register allocation must allow (0: left to the compiler,
// which keeps these kernels at 2 blocks of 256 threads per SM; 3 or 4 blocks
// with fewer vectors per lane measured 5-15 % slower on the decode gather).
#ifndef GTKV_GATHER_MINB
#define GTKV_GATHER_MINB 0
#endif
#if GTKV_GATHER_MINB > 0
#define GTKV_GATHER_BOUNDS __launch_bounds__(kBlock, GTKV_GATHER_MINB)
#else
#define GTKV_GATHER_BOUNDS __launch_bounds__(kBlock)
#endif

// Metadata checks, one sequence per thread, grid-stride (they never gate the
// copies: every access is bounds-checked on its own): KV_DEV_ERR_TABLE when
// start < 0, len > max_pages * ps, cu_out not non-decreasing from 0 or a span
// shorter than its tokens, or cu_out[n_seqs] > out_rows.
__device__ __forceinline__ void check_gather_meta(const DevPool& p, int32_t n_seqs, int32_t max_pages,
                                                  const int32_t* __restrict__ seq_start,
                                                  const int32_t* __restrict__ seq_len,
                                                  const int64_t* __restrict__ cu, int64_t out_rows, int64_t tid,
                                                  int64_t nthreads) {
  for (int64_t s = tid; s < n_seqs; s += nthreads) {
    const int64_t a = seq_start ? __ldg(seq_start + s) : 0;
    const int64_t b = __ldg(seq_len + s);
    const int64_t c0 = __ldg(cu + s), c1 = __ldg(cu + s + 1);
    if (a < 0 || b > static_cast<int64_t>(max_pages) * p.ps || c0 < 0 || c1 < c0 || c1 - c0 < b - a)
      atomicOr(p.err, KV_DEV_ERR_TABLE);
  }
  if (tid == 0 && __ldg(cu + n_seqs) > out_rows) atomicOr(p.err, KV_DEV_ERR_TABLE);
}

// One work item: chunk c of block-table entry sk = s*max_pages + k, clipped to
// the window [start_s, len_s), to tokens >= 0 and to output rows [0, out_rows).
// With KF the table holds kernel-facing entries phys * 2L (2L = the
// row-blocks per page, L for MLA: the prefix-only table of
// kv_translate_block_table): entry * ps + o is then the token's kernel-facing
// id, so the page is entry / 2L and an entry off that grid is a form error.
struct Run {
  int64_t src;   // 16-byte vector index (from p.base) of its first K row; V is ps rows later
  int64_t row;   // first output row
  int64_t nvec;  // 16-byte vectors of K (and of V)
  int kind;      // 0: nothing to copy; 1: rows of a page; 2: tombstoned entry, every row reads the sink
};

template <bool KF>
__device__ __forceinline__ Run gather_item(const DevPool& p, int64_t sk, int64_t c, int64_t koff,
                                           const int32_t* __restrict__ bt, int32_t max_pages,
                                           const int32_t* __restrict__ seq_start,
                                           const int32_t* __restrict__ seq_len, const int64_t* __restrict__ cu,
                                           int64_t out_rows, int32_t chunk_rows, bool report) {
  Run r{0, 0, 0, 0};
  const int64_t ps = p.ps;
  const int64_t s = sk / max_pages;
  const int64_t k = sk - s * max_pages;
  const int64_t a = seq_start ? __ldg(seq_start + s) : 0;
  const int64_t b = __ldg(seq_len + s);
  const int64_t j0 = k * ps + c * chunk_rows;  // first token of this chunk
  int64_t jlo = j0 > a ? j0 : a;
  if (jlo < 0) jlo = 0;
  int64_t jhi = j0 + chunk_rows;
  if (jhi > (k + 1) * ps) jhi = (k + 1) * ps;
  if (jhi > b) jhi = b;
  if (jlo >= jhi) return r;  // entry outside the window: empty item
  int64_t page = __ldg(bt + sk);
  if (page >= p.num_pages * (KF ? p.blocks : 1)) {  // a page (or kernel-facing entry) past the pool
    if (report) atomicOr(p.err, KV_DEV_ERR_ROW);
    return r;
  }
  if (KF && page > 0) {  // 0 < entry < P * 2L < 2^31: 32-bit arithmetic
    const uint32_t e = static_cast<uint32_t>(page), b = static_cast<uint32_t>(p.blocks);
    const uint32_t phys = e / b;
    if (phys * b != e) {
      if (report) atomicOr(p.err, KV_DEV_ERR_FORM);
      return r;
    }
    page = phys;
  }
  const int64_t cs = __ldg(cu + s);
  int64_t rlo = cs + (jlo - a);
  int64_t rhi = cs + (jhi - a);
  if (rlo < 0) {  // rows before 0 are never written (cu_out[s] < 0 is flagged)
    jlo -= rlo;
    rlo = 0;
  }
  if (rhi > out_rows) rhi = out_rows;
  if (rlo >= rhi) return r;
  r.row = rlo;
  r.nvec = (rhi - rlo) * p.vpr;
  if (page < 0) {
    r.kind = 2;
    r.src = koff * p.vpr;
  } else {
    r.kind = 1;
    r.src = (page * p.stride + koff + (jlo - k * ps)) * p.vpr;
  }
  return r;
}


// Items = (table entry sk, chunk c), taken in table order, or in the order of
// a page-major plan (PLANNED: kv_plan.cu). CHV 16-byte vectors per lane per
// round: one round moves 32*CHV vectors of K and, with HAS_V, as many of V
// (a latent-only pool has no V rows). KF: the table holds kernel-facing
// entries (see gather_item).
template <int CHV, bool PLANNED, bool HAS_V, bool KF>
__global__ void GTKV_GATHER_BOUNDS k_gather_runs(DevPool p, int32_t layer, const int32_t* __restrict__ bt,
                                                        int32_t n_seqs, int32_t max_pages,
                                                        const int32_t* __restrict__ seq_start,
                                                        const int32_t* __restrict__ seq_len,
                                                        const int64_t* __restrict__ cu, uint4* __restrict__ out_k,
                                                        uint4* __restrict__ out_v, int64_t out_rows,
                                                        int32_t chunk_rows, int32_t chunks_per_page,
                                                        const int32_t* __restrict__ plan, int batch) {
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t nthreads = static_cast<int64_t>(gridDim.x) * blockDim.x;
  check_gather_meta(p, n_seqs, max_pages, seq_start, seq_len, cu, out_rows, tid, nthreads);
  const int64_t n_entries = static_cast<int64_t>(n_seqs) * max_pages;
  int64_t n_units = n_entries;  // entries (table order) or plan positions
  const int32_t* order = nullptr;
  if constexpr (PLANNED) {
    // the plan must have been built for a table of this shape and form; its
    // entries are bounds-checked one by one below, so a stale plan can only
    // give wrong rows (flagged), never an access outside the buffers
    const int32_t flags = __ldg(plan + 3);
    if (__ldg(plan + 1) != n_seqs || __ldg(plan + 2) != max_pages ||
        ((flags & kPlanKernelFacing) != 0) != KF) {
      if (tid == 0) atomicOr(p.err, KV_DEV_ERR_TABLE);
      return;
    }
    if (flags & kPlanPageMajor) {  // page-major order pays; else keep the table's order
      const int64_t np = __ldg(plan);
      n_units = np < 0 ? 0 : (np > n_entries ? n_entries : np);
      order = plan + 4 + p.num_pages + 1;
    }
  }

  const int lane = threadIdx.x & 31;
  const int64_t vpr = p.vpr;
  const int64_t ps_vec = p.ps * vpr;                                      // K -> V distance, in vectors
  const int64_t koff = static_cast<int64_t>(layer) * p.kv_rows * p.ps;  // K (or latent) block of the layer
  constexpr bool has_v = HAS_V;
  const int64_t n_items = n_units * chunks_per_page;
  const L2Policy pol = make_l2_policy();

  // A warp takes `batch` consecutive items at a time (8 chunks of 4 KiB: a
  // whole 16-token entry of 2 KiB rows, read and written as one stream) and
  // works their runs out at once: lane j takes
  // item it0 + j (its plan position, table entry, window and output rows: a
  // chain of dependent loads), so one chain's latency serves the whole batch;
  // the warp then copies the runs in turn, each broadcast by shuffle.
  const int64_t n_warps = nthreads >> 5;
  for (int64_t it0 = (tid >> 5) * batch; it0 < n_items; it0 += n_warps * batch) {
    Run mine{0, 0, 0, 0};
    const int64_t it = it0 + lane;
    if (lane < batch && it < n_items) {
      const int64_t u = it / chunks_per_page;
      const int64_t c = it - u * chunks_per_page;
      int64_t sk = u;
      bool ok = true;
      if (PLANNED && order != nullptr) {
        sk = __ldg(order + u);
        if (sk < 0 || sk >= n_entries) {
          atomicOr(p.err, KV_DEV_ERR_TABLE);
          ok = false;
        }
      }
      if (ok)
        mine = gather_item<KF>(p, sk, c, koff, bt, max_pages, seq_start, seq_len, cu, out_rows, chunk_rows, true);
    }
    const int nb = n_items - it0 < batch ? static_cast<int>(n_items - it0) : batch;
    for (int j = 0; j < nb; ++j) {
      const int kind = __shfl_sync(kFull, mine.kind, j);
      if (kind == 0) continue;
      const int64_t row = __shfl_sync(kFull, mine.row, j);
      const int64_t nvec = __shfl_sync(kFull, mine.nvec, j);
      const uint4* srck = p.base + __shfl_sync(kFull, mine.src, j);
      const uint4* srcv = srck + ps_vec;
      uint4* dk = out_k + row * vpr;
      uint4* dv = has_v ? out_v + row * vpr : nullptr;
      if (kind == 1) {
        for (int64_t v0 = 0; v0 < nvec; v0 += 32 * CHV) {
          uint4 bk[CHV], bv[CHV];
#pragma unroll
          for (int i = 0; i < CHV; ++i) {
            const int64_t v = v0 + lane + 32 * i;
            if (v < nvec) {
              bk[i] = ld16<GTKV_GATHER_LD>(srck + v, pol);
              if (has_v) bv[i] = ld16<GTKV_GATHER_LD>(srcv + v, pol);
            }
          }
#pragma unroll
          for (int i = 0; i < CHV; ++i) {
            const int64_t v = v0 + lane + 32 * i;
            if (v < nvec) {
              st16<GTKV_GATHER_ST>(dk + v, bk[i], pol);
              if (has_v) st16<GTKV_GATHER_ST>(dv + v, bv[i], pol);
            }
          }
        }
      } else {  // tombstoned entry: every token of the run reads the page-0 sink row
        for (int64_t v = lane; v < nvec; v += 32) {
          const int64_t col = v % vpr;
          st16<GTKV_GATHER_ST>(dk + v, ld16<GTKV_GATHER_LD>(srck + col, pol), pol);
          if (has_v) st16<GTKV_GATHER_ST>(dv + v, ld16<GTKV_GATHER_LD>(srcv + col, pol), pol);
        }
      }
    }
  }
}

// ---- fan-out form of the gather -------------------------------------------
//
// With a page-major plan the readers of a page are consecutive plan
// positions. A block of one warp takes `group` consecutive positions (whole
// table entries), loads the rows of each page they name into shared memory
// once (bulk copy, completion counted on an mbarrier) and writes them to every
// reader's output rows with bulk stores: a page shared by n readers is read
// from L2 n / group times instead of n times, and the output leaves through
// the bulk-copy engine in whole-entry runs. The grid is not persistent (one
// block per `group` positions, balanced over the SMs by the hardware block
// scheduler): on this GPU a persistent grid writes at ~6.5 TB/s whatever its
// store form, short blocks at ~7.5 TB/s. A block whose positions name several
// pages keeps up to `nbuf` page loads in flight (one buffer and one mbarrier
// each), issued in the order the pages are written.
//
// Positions per block, measured: on the decode gather (256 x 4096 tokens over
// tables that name every page ~16 times) 2 positions per block take the
// page-major walk from 742 to 708 us against the vector kernel (3 or 4: the
// same; 1: 757 us, every reader reloading its page) and the MLA gather from 142
// to 131 us. Where pages are read about once, a block of two entries ends with
// the later of two loads (the SWA gather +5 %), and one entry per block is as
// fast as the vector kernel or faster (stress gather 42.1 -> 41.0 us). So a
// block takes 2 positions when the table has at least as many entries as the
// pool has pages (its entries then name pages several times over), else 1;
// gathers without a plan take 1 table entry per block (decode tables 1241 ->
// 1169 us, MLA 175 -> 170 us, stress 41.6 -> 40.8 us, SWA unchanged). Pages
// whose rows of a layer exceed GTKV_FAN_MAX_BYTES keep the vector kernel.

#ifndef GTKV_GATHER_FANOUT
#define GTKV_GATHER_FANOUT 1  // 0: every gather takes the vector kernel
#endif
#ifndef GTKV_FAN_GROUP
#define GTKV_FAN_GROUP 2  // plan positions per block for tables of >= num_pages entries (1..32)
#endif
#ifndef GTKV_FAN_MAX_BYTES
#define GTKV_FAN_MAX_BYTES 73728  // shared memory per block for page buffers (a 64-row 1152-byte latent page)
#endif
// L2 eviction priority of the page loads (pages have other readers in
// nearby blocks) and of the output stores (never read back by the gather).
#ifndef GTKV_FAN_LD_PRIO
#define GTKV_FAN_LD_PRIO "evict_last"
#endif
#ifndef GTKV_FAN_ST_PRIO
#define GTKV_FAN_ST_PRIO "evict_first"
#endif
static_assert(GTKV_FAN_GROUP >= 1 && GTKV_FAN_GROUP <= 32, "one warp per block");

template <bool HAS_V, bool KF>
__global__ void __launch_bounds__(32) k_gather_fan(DevPool p, int32_t layer, const int32_t* __restrict__ bt,
                                                   int32_t n_seqs, int32_t max_pages,
                                                   const int32_t* __restrict__ seq_start,
                                                   const int32_t* __restrict__ seq_len,
                                                   const int64_t* __restrict__ cu, uint4* __restrict__ out_k,
                                                   uint4* __restrict__ out_v, int64_t out_rows,
                                                   const int32_t* __restrict__ plan, int group, int nbuf) {
  extern __shared__ __align__(128) uint4 sbuf[];  // nbuf buffers: a page's K rows of the layer, then its V rows
  __shared__ __align__(8) uint64_t bars[32];
  const int lane = threadIdx.x;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * 32 + lane;
  check_gather_meta(p, n_seqs, max_pages, seq_start, seq_len, cu, out_rows, tid,
                    static_cast<int64_t>(gridDim.x) * 32);
  const int64_t n_entries = static_cast<int64_t>(n_seqs) * max_pages;
  int64_t n_units = n_entries;  // table order, unless a page-major plan is given
  const int32_t* order = nullptr;
  if (plan != nullptr) {
    const int32_t flags = __ldg(plan + 3);
    if (__ldg(plan + 1) != n_seqs || __ldg(plan + 2) != max_pages || ((flags & kPlanKernelFacing) != 0) != KF) {
      if (tid == 0) atomicOr(p.err, KV_DEV_ERR_TABLE);
      return;
    }
    if (flags & kPlanPageMajor) {
      const int64_t np = __ldg(plan);
      n_units = np < 0 ? 0 : (np > n_entries ? n_entries : np);
      order = plan + kPlanHeaderWords + p.num_pages + 1;
    }
  }
  const int64_t vpr = p.vpr;
  const int64_t koff = static_cast<int64_t>(layer) * p.kv_rows * p.ps;
  const L2Policy pol = make_l2_policy();
  uint64_t ld_pol, st_pol;
  asm("createpolicy.fractional.L2::" GTKV_FAN_LD_PRIO ".b64 %0, 1.0;" : "=l"(ld_pol));
  asm("createpolicy.fractional.L2::" GTKV_FAN_ST_PRIO ".b64 %0, 1.0;" : "=l"(st_pol));

  // lane j < group: plan position blockIdx.x * group + j, a whole table entry
  Run mine{0, 0, 0, 0};
  const int64_t u = static_cast<int64_t>(blockIdx.x) * group + lane;
  if (lane < group && u < n_units) {
    int64_t sk = u;
    bool ok = true;
    if (order != nullptr) {
      sk = __ldg(order + u);
      if (sk < 0 || sk >= n_entries) {
        atomicOr(p.err, KV_DEV_ERR_TABLE);
        ok = false;
      }
    }
    if (ok)
      mine = gather_item<KF>(p, sk, 0, koff, bt, max_pages, seq_start, seq_len, cu, out_rows,
                             static_cast<int32_t>(p.ps), true);
  }
  // a page run: page pg, rows [off, off + nrows) of the layer's block
  int64_t pg = -1;
  int32_t off = 0, nrows = 0;
  if (mine.kind == 1) {
    const int64_t r = mine.src / vpr;
    pg = r / p.stride;
    off = static_cast<int32_t>(r - pg * p.stride - koff);
    nrows = static_cast<int32_t>(mine.nvec / vpr);
  }

  // Page groups: the block's runs that name one page, numbered in the order
  // of their lowest lane; group g's rows [lo, hi) of the page go to buffer
  // g % nbuf, and its lowest lane issues that load.
  int my_g = -1, lead_g = -1, ng = 0;
  int32_t g_lo = 0, g_hi = 0;
  int64_t g_pg = 0;
  for (unsigned t = __ballot_sync(kFull, mine.kind == 1); t; ++ng) {
    const int lead = __ffs(t) - 1;
    const int64_t gp = __shfl_sync(kFull, pg, lead);
    const bool in = mine.kind == 1 && pg == gp;
    const unsigned members = __ballot_sync(kFull, in);
    const int32_t lo = __reduce_min_sync(kFull, in ? off : INT32_MAX);
    const int32_t hi = __reduce_max_sync(kFull, in ? off + nrows : 0);
    if (in) my_g = ng;
    if (lane == lead) {
      lead_g = ng;
      g_lo = lo;
      g_hi = hi;
      g_pg = gp;
    }
    t &= ~members;
  }
  if (ng > 0) {
    const int64_t buf_vecs = p.kv_rows * p.ps * vpr;
    if (lane < nbuf) mbar_init(bars + lane);
    __syncwarp();
    auto issue = [&](int b) {  // by the lane that leads the group
      const uint32_t bytes = static_cast<uint32_t>((g_hi - g_lo) * vpr * 16);
      uint4* sb = sbuf + b * buf_vecs;
      mbar_expect(bars + b, HAS_V ? 2 * bytes : bytes);
      const uint4* src = p.base + (g_pg * p.stride + koff + g_lo) * vpr;
      bulk_load(sb + g_lo * vpr, src, bytes, bars + b, ld_pol);
      if (HAS_V) bulk_load(sb + (p.ps + g_lo) * vpr, src + p.ps * vpr, bytes, bars + b, ld_pol);
    };
    if (lead_g >= 0 && lead_g < nbuf) issue(lead_g);
    for (int g = 0; g < ng; ++g) {
      const int b = g % nbuf;
      if (!__all_sync(kFull, mbar_wait_bounded(bars + b, (g / nbuf) & 1))) {
        // a load that never landed: flag it, give the loads in flight one more
        // bounded wait, then leave
        if (lane == 0) atomicOr(p.err, KV_DEV_ERR_TIMEOUT);
        for (int q = g; q < ng && q < g + nbuf; ++q) mbar_wait_bounded(bars + q % nbuf, (q / nbuf) & 1);
        bulk_wait_all();
        return;
      }
      if (my_g == g) {
        const uint32_t run = static_cast<uint32_t>(nrows * vpr * 16);
        const uint4* sb = sbuf + b * buf_vecs;
        bulk_store(out_k + mine.row * vpr, sb + off * vpr, run, st_pol);
        if (HAS_V) bulk_store(out_v + mine.row * vpr, sb + (p.ps + off) * vpr, run, st_pol);
        bulk_commit();
      }
      if (g + nbuf < ng) {  // group g + nbuf reuses buffer b: group g's stores must have read it
        if (my_g == g) bulk_wait_read();
        __syncwarp();
        if (lead_g == g + nbuf) issue(b);
      }
    }
  }
  // tombstoned entries: every token of the run reads the page-0 sink row
  const unsigned sinks = __ballot_sync(kFull, mine.kind == 2);
  for (unsigned m = sinks; m; m &= m - 1) {
    const int j = __ffs(m) - 1;
    const int64_t row = __shfl_sync(kFull, mine.row, j);
    const int64_t nvec = __shfl_sync(kFull, mine.nvec, j);
    const uint4* srck = p.base + __shfl_sync(kFull, mine.src, j);
    for (int64_t v = lane; v < nvec; v += 32) {
      const int64_t col = v % vpr;
      st16<GTKV_GATHER_ST>(out_k + row * vpr + v, ld16<GTKV_GATHER_LD>(srck + col, pol), pol);
      if (HAS_V)
        st16<GTKV_GATHER_ST>(out_v + row * vpr + v, ld16<GTKV_GATHER_LD>(srck + p.ps * vpr + col, pol), pol);
    }
  }
  bulk_wait_read();  // shared memory must outlive the stores' reads
}

}  // namespace

// The fan-out kernels take up to GTKV_FAN_MAX_BYTES of dynamic shared memory,
// more than the 48 KiB a launch gets by default; the limit is a property of
// the function on the current device, raised here once per pool (from
// kv_pool_create, outside any stream capture) so that no launch has to.
cudaError_t prepare_gather() {
  const void* fans[] = {reinterpret_cast<const void*>(k_gather_fan<true, false>),
                        reinterpret_cast<const void*>(k_gather_fan<true, true>),
                        reinterpret_cast<const void*>(k_gather_fan<false, false>),
                        reinterpret_cast<const void*>(k_gather_fan<false, true>)};
  for (const void* f : fans) {
    const cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, GTKV_FAN_MAX_BYTES);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_gather(const DevPool& p, int32_t layer, const int32_t* bt, int32_t n_seqs, int32_t max_pages,
                          const int32_t* seq_start, const int32_t* seq_len, const int64_t* cu, void* out_k,
                          void* out_v, int64_t out_rows, const int32_t* plan, bool kernel_facing, int sm_count,
                          cudaStream_t s) {
  // rows per item: GTKV_GATHER_CHUNK bytes of K (and as many of V); a
  // latent-only pool has no V, so its items take twice the K bytes and keep
  // the same bytes in flight per warp
  const bool latent = p.kv_rows == 1;
  const int64_t page_layer_bytes = static_cast<int64_t>(p.kv_rows) * p.ps * p.vpr * 16;
  const int64_t n_table = static_cast<int64_t>(n_seqs) * max_pages;
  if (GTKV_GATHER_FANOUT && page_layer_bytes <= GTKV_FAN_MAX_BYTES) {
    using FanKernel = decltype(&k_gather_fan<true, false>);
    const FanKernel fans[2][2] = {{k_gather_fan<true, false>, k_gather_fan<true, true>},
                                  {k_gather_fan<false, false>, k_gather_fan<false, true>}};
    const FanKernel fan = fans[latent][kernel_facing];
    const int group = plan != nullptr && n_table >= p.num_pages ? GTKV_FAN_GROUP : 1;
    // page buffers per block: as many as GTKV_FAN_MAX_BYTES holds, at most one per position
    int64_t nbuf = GTKV_FAN_MAX_BYTES / page_layer_bytes;
    if (nbuf > group) nbuf = group;
    if (nbuf < 1) nbuf = 1;
    const int smem = static_cast<int>(nbuf * page_layer_bytes);  // <= GTKV_FAN_MAX_BYTES: see prepare_gather
    int64_t blocks = (n_table + group - 1) / group;
    const int64_t seq_blocks = (static_cast<int64_t>(n_seqs) + 31) / 32;  // the metadata checks
    if (blocks < seq_blocks) blocks = seq_blocks;
    if (blocks < 1) blocks = 1;
    fan<<<static_cast<unsigned>(blocks), 32, smem, s>>>(p, layer, bt, n_seqs, max_pages, seq_start, seq_len, cu,
                                                       static_cast<uint4*>(out_k), static_cast<uint4*>(out_v),
                                                       out_rows, plan, group, static_cast<int>(nbuf));
    return cudaGetLastError();
  }
  auto rows_per_item = [&](int64_t bytes) {
    int64_t r = bytes / (16 * p.vpr);
    if (r < 1) r = 1;
    if (r > p.ps) r = p.ps;
    return r;
  };
  int64_t chunk_rows = rows_per_item(GTKV_GATHER_CHUNK);
  int64_t cpp = (p.ps + chunk_rows - 1) / chunk_rows;
  // one round: 32 lanes x 8 vectors = 4 KiB of K and 4 KiB of V (latent: 8 KiB of K) in flight per warp
  constexpr int CHV = GTKV_GATHER_CHV;
  const int kind = !latent ? 0 : (GTKV_GATHER_V72 && p.vpr == 72 ? 2 : 1);
  constexpr int V72T = GTKV_GATHER_V72_TABLE_CHV, V72P = GTKV_GATHER_V72_PLANNED_CHV;
  using Kernel = decltype(&k_gather_runs<CHV, true, true, false>);
  const Kernel kernels[3][2][2] = {  // [MHA / latent / 1152-byte latent][plan][kernel_facing]
      {{k_gather_runs<CHV, false, true, false>, k_gather_runs<CHV, false, true, true>},
       {k_gather_runs<CHV, true, true, false>, k_gather_runs<CHV, true, true, true>}},
      {{k_gather_runs<2 * CHV, false, false, false>, k_gather_runs<2 * CHV, false, false, true>},
       {k_gather_runs<2 * CHV, true, false, false>, k_gather_runs<2 * CHV, true, false, true>}},
      {{k_gather_runs<V72T, false, false, false>, k_gather_runs<V72T, false, false, true>},
       {k_gather_runs<V72P, true, false, false>, k_gather_runs<V72P, true, false, true>}}};
  const Kernel kernel = kernels[kind][plan != nullptr][kernel_facing];
  if (latent) {
    chunk_rows = rows_per_item(kind == 2 ? 32 * 16 * (plan != nullptr ? V72P : V72T) : 2 * GTKV_GATHER_CHUNK);
    cpp = (p.ps + chunk_rows - 1) / chunk_rows;
  }
  int64_t warps = static_cast<int64_t>(n_seqs) * max_pages * cpp;
  const int64_t seq_warps = (static_cast<int64_t>(n_seqs) + 31) / 32;
  if (warps < seq_warps) warps = seq_warps;
  const unsigned grid = grid_for(kernel, warps, sm_count);
  // items per warp batch: up to GTKV_GATHER_MAX_BATCH, fewer when the grid's
  // warps would not all get a full batch
  const int64_t grid_warps = static_cast<int64_t>(grid) * (kBlock / 32);
  const int64_t n_items = static_cast<int64_t>(n_seqs) * max_pages * cpp;
  int64_t batch = (n_items + grid_warps - 1) / grid_warps;
  if (batch > GTKV_GATHER_MAX_BATCH) batch = GTKV_GATHER_MAX_BATCH;
  if (batch < 1) batch = 1;
  kernel<<<grid, kBlock, 0, s>>>(p, layer, bt, n_seqs, max_pages, seq_start, seq_len, cu,
                                 static_cast<uint4*>(out_k), static_cast<uint4*>(out_v), out_rows,
                                 static_cast<int32_t>(chunk_rows), static_cast<int32_t>(cpp), plan,
                                 static_cast<int>(batch));
  return cudaGetLastError();
}

}  // namespace gtkv
