/*
 * kv_pool.h -- C ABI of a unified page-major KV-cache pool for uniform-row
 * MHA / sliding-window attention models, with hand-written CUDA kernels for
 * NVIDIA GB300 (sm_103a).
 *
 * Source of the layout and of every operation: the prhub report on sglang PR
 * #34602, "feat(unified-memory): dense KV views for uniform-row MHA/SWA
 * models" (cited below as "the report", by section).
 *
 * Layout (实现拆解 step 1; 关键源码片段 layout/page_major.py build_mha_views).
 * One raw byte buffer holds [anchor | pool | tail pad]. The pool is num_pages
 * page envelopes; each envelope is 2L equal row-blocks of page_size rows,
 * [L0_K | L0_V | L1_K | L1_V | ...], so layer l's K is block 2l and its V is
 * block 2l+1. A row is R = head_num * head_dim * itemsize bytes (one token's
 * K, or V, for one layer). A token slot t (physical page t/ps, offset t%ps)
 * has the kernel-facing id
 *
 *      kernel_id(t) = (t / ps) * (ps * 2L) + t % ps
 *
 * and block b of that token is the row at byte
 *
 *      anchor + (kernel_id + b * ps) * R.
 *
 * Sizes: page_bytes = ps * 2L * R, total = num_pages * page_bytes,
 * tail_pad = ps * 2L * R (one page envelope: MHASubPoolSpec.
 * view_tail_pad_bytes returns page_size * entry_bytes, entry_bytes read as
 * 2L * R), n_rows = num_pages * 2L * ps (kernel-facing rows, must be < 2^31:
 * _assert_kernel_id_bound, 实现拆解 step 2 and 风险与影响 item 5).
 *
 * Conventions for every call below.
 *  - Pointers named *_dev are device memory of the pool's device; the others
 *    are host memory. Nothing is retained after a call returns: the caller
 *    owns every buffer it passes.
 *  - Compute calls are asynchronous on `stream` (a cudaStream_t; NULL is the
 *    legacy default stream), launch only this library's kernels, allocate
 *    nothing and never synchronize. kv_translate, kv_translate_mapped, the
 *    stores, kv_translate_block_table, kv_gather_plan, kv_gather_plan_kf,
 *    the gathers and kv_move can be captured in a CUDA graph.
 *    kv_pool_last_error is the one call that synchronizes.
 *  - The calling thread's current device must be the pool's device.
 *  - Return value: KV_OK (0) or a negative KV_ERR_* code. These are argument,
 *    layout and launch errors, found on the host before anything is enqueued
 *    (KV_ERR_CUDA also covers a failed launch).
 *  - Data-dependent errors (an id, page or table entry pointing outside the
 *    pool) are never a trap: the kernel skips that row and ORs a
 *    KV_DEV_ERR_* bit into the pool's device error word, which
 *    kv_pool_last_error returns and clears.
 *  - K/V bytes are opaque: no call converts, rounds or inspects them.
 *
 * MLA pools (latent_only = 1). The report's MLA sub-pools use the same dense
 * per-layer views with blocks_per_page() = layer_num (实现拆解 step 2): the
 * envelope is [L0 | L1 | ...], one latent row per layer per token, layer l
 * in block l, kernel_id(t) = (t / ps) * (ps * L) + t % ps. Everything above
 * holds with 2L replaced by L; every V argument is ignored (may be NULL).
 */
#ifndef GATHER_TRANSLATE_KV_GB300_KV_POOL_H
#define GATHER_TRANSLATE_KV_GB300_KV_POOL_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Host status codes. */
enum {
  KV_OK = 0,
  KV_ERR_INVALID = -1,    /* bad argument: null pointer, negative count, layer out of range */
  KV_ERR_ASYMMETRIC = -2, /* head_dim != v_head_dim: no uniform row-block array exists */
  KV_ERR_ID_BOUND = -3,   /* num_pages * 2L * page_size >= 2^31 */
  KV_ERR_TAIL_PAD = -4,   /* raw buffer ends before the last view does */
  KV_ERR_ALIGN = -5,      /* a pointer, the anchor or the row size breaks 16-byte alignment */
  KV_ERR_CUDA = -6,       /* a CUDA runtime call or a kernel launch failed */
  KV_ERR_DEVICE = -7,     /* current device is not the pool's, or a buffer is another device's */
  KV_ERR_CAPACITY = -8    /* more pages than kv_gather_plan_noalloc's fixed workspace holds */
};

/* Bits of the device error word (kv_pool_last_error). */
#define KV_DEV_ERR_ROW 1   /* an id / page addressed a row outside the pool; row skipped   */
#define KV_DEV_ERR_V2P 2   /* translate: a virtual page index was past the page map        */
#define KV_DEV_ERR_TABLE 4 /* gather: sequence metadata inconsistent (see kv_gather_layer);
                              plan: the table changed while the plan was built */
#define KV_DEV_ERR_FORM 8  /* store / move: an id was not p * ps * 2L + o with o < ps (token or
                              pair skipped);
                              kernel-facing gather / plan: an entry was not a multiple of 2L
                              (its tokens skipped) */
#define KV_DEV_ERR_TIMEOUT 16 /* gather / move: a load into shared memory did not complete
                                 within its bounded wait (~1 s); that block's remaining rows
                                 are left untouched. Not expected on a healthy GPU. */

typedef struct kv_pool kv_pool_t; /* opaque, host-side, owned by the library */

/* A cudaStream_t without requiring the CUDA headers. */
typedef struct CUstream_st* kv_stream_t;

/* Pool geometry in the report's notation (build_mha_views' arguments). */
typedef struct {
  int32_t layer_num;    /* L >= 1                                                  */
  int32_t head_num;     /* H >= 1, KV heads                                        */
  int32_t head_dim;     /* D >= 1                                                  */
  int32_t v_head_dim;   /* must equal head_dim                                     */
  int32_t itemsize;     /* bytes per element: 1 (fp8), 2 (bf16/fp16) or 4          */
  int32_t page_size;    /* ps >= 1 tokens per page                                 */
  int64_t num_pages;    /* P >= 1; page 0 is the tombstone sink                    */
  int64_t anchor_bytes; /* byte offset of the pool in the raw buffer, % 16 == 0    */
  int32_t latent_only;  /* 0: MHA/SWA pool, a K and a V row per layer (2L blocks)  */
                        /* 1: MLA pool, one latent row per layer (L blocks, no V;  */
                        /*    v_head_dim is ignored). Zero-initialised = MHA.      */
  int32_t reserved;     /* must be 0                                               */
} kv_pool_desc;

/* Derived layout of a pool (kv_pool_info). */
typedef struct {
  void* raw_dev;         /* start of the raw buffer                       */
  int64_t raw_bytes;     /* its size                                      */
  int64_t row_bytes;     /* R                                             */
  int64_t page_bytes;    /* ps * 2L * R                                   */
  int64_t total_bytes;   /* num_pages * page_bytes                        */
  int64_t tail_pad_bytes;/* ps * 2L * R                                   */
  int64_t n_rows;        /* num_pages * 2L * ps                           */
  int64_t last_view_end; /* anchor + (2L-1)*ps*R + n_rows*R               */
  int32_t device;        /* CUDA device ordinal the pool lives on         */
  int32_t owns_raw;      /* 1 when kv_pool_create allocated the buffer    */
  int32_t blocks_per_page; /* 2L (MHA/SWA) or L (MLA)                     */
  int32_t latent_only;   /* the descriptor's flag                         */
} kv_pool_info_t;

/* Sizes of a pool, host only, no CUDA call.
 * Source: UnifiedKVPool.__init__ allocates total_bytes + view_tail_pad_bytes
 * (关键源码片段 unified_memory_pool.py); page_bytes and n_rows from
 * build_mha_views (关键源码片段 page_major.py).
 * Writes *total_bytes = num_pages * ps * 2L * R and *tail_pad_bytes =
 * ps * 2L * R; the raw buffer a caller allocates is anchor_bytes +
 * total_bytes + tail_pad_bytes. Either output may be NULL. Runs every gate of
 * kv_pool_create except the buffer-size one and returns its code. */
int kv_pool_required_bytes(const kv_pool_desc* desc, int64_t* total_bytes, int64_t* tail_pad_bytes);

/* Create a pool on the current device.
 * Source: UnifiedKVPool.__init__ and build_mha_views (关键源码片段) with the
 * start-up gates of 实现拆解 step 2: uniform rows (KV_ERR_ASYMMETRIC), the
 * kernel-facing id bound (KV_ERR_ID_BOUND), and the last view fitting in the
 * raw buffer (KV_ERR_TAIL_PAD).
 *  raw_dev == NULL: the library allocates anchor + total + tail_pad bytes
 *    (cudaMalloc, contents undefined) and frees them in kv_pool_destroy.
 *  raw_dev != NULL: the pool borrows the caller's buffer (16-byte aligned,
 *    raw_bytes long, device or managed memory of the current device: host
 *    memory gives KV_ERR_INVALID, another device's memory KV_ERR_DEVICE) for
 *    its whole life; raw_bytes must reach
 *    last_view_end = anchor + (2L-1)*ps*R + n_rows*R, which build_mha_views
 *    asserts, else KV_ERR_TAIL_PAD. A buffer of anchor + total + tail_pad
 *    bytes always suffices.
 * Additionally requires R % 16 == 0 and anchor_bytes % 16 == 0
 * (KV_ERR_ALIGN): every kernel moves rows as 16-byte vectors.
 * Also allocates the pool's device error word (8 bytes) and raises the
 * gather kernels' shared-memory limit on the current device (a property of
 * the functions, set here so that no later call has to; create pools outside
 * stream capture). Launches no kernel.
 * On success *out receives the handle; on failure *out is set to NULL and
 * nothing stays allocated. */
int kv_pool_create(const kv_pool_desc* desc, void* raw_dev, int64_t raw_bytes, kv_pool_t** out);

/* Free a pool: the error word, and the raw buffer if the library allocated
 * it. Synchronizes nothing; the caller must ensure no work using the pool is
 * still in flight. NULL is accepted. */
int kv_pool_destroy(kv_pool_t* pool);

/* Copy the derived layout of a pool into *out (host only). */
int kv_pool_info(const kv_pool_t* pool, kv_pool_info_t* out);

/* Token slots -> kernel-facing int32 ids.
 * Source: MultiEndedAllocator.translate_kv_loc_for_kernel (关键源码片段
 * multi_ended_allocator.py; 实现拆解 step 3): page = t / ps, off = t % ps,
 * phys = v2p[page] when a page map is given (else phys = page),
 * id = phys * (ps * 2L) + off, clamped to 0 (the page-0 sink) when t < 0 or
 * phys < 0. kernel_page_multiplier is always blocks_per_page() = 2L.
 *  slots_dev  int64 [n]
 *  v2p_dev    int32 [v2p_len] virtual -> physical page map, or NULL
 *  ids_dev    int32 [n] output; must not overlap slots_dev (the report's
 *             in-place aliasing case is not supported)
 * Device errors: a page index >= v2p_len sets KV_DEV_ERR_V2P, a physical page
 * >= num_pages sets KV_DEV_ERR_ROW; both write id 0. n == 0 is a no-op. */
int kv_translate(const kv_pool_t* pool, const int64_t* slots_dev, int64_t n, const int32_t* v2p_dev,
                 int64_t v2p_len, int32_t* ids_dev, kv_stream_t stream);

/* Full -> SWA token mapping, then translate: for slot t of the full-attention
 * sub-pool, t' = tmap[t] is the token's slot in this (sliding-window)
 * sub-pool, and ids[i] is kv_translate of t' (with the optional page map).
 * Source: SWA sub-pools share the dense id space (实现拆解 step 2,
 * init_unified_swa_pools) and are addressed through the full -> SWA token
 * mapping, whose cleared entries are tombstones (关联脉络: PR #35773,
 * clear_full_to_swa_mapping).
 *  slots_dev  int64 [n] full-pool slots (negative = tombstone)
 *  tmap_dev   int64 [tmap_len] full slot -> SWA slot (negative = cleared)
 *  v2p_dev    int32 [v2p_len] page map of this pool, or NULL
 *  ids_dev    int32 [n] output; must not overlap slots_dev
 * A tombstone or cleared entry gives id 0 (the sink). Device errors: a slot
 * >= tmap_len sets KV_DEV_ERR_V2P (id 0); then as kv_translate. */
int kv_translate_mapped(const kv_pool_t* pool, const int64_t* slots_dev, int64_t n, const int64_t* tmap_dev,
                        int64_t tmap_len, const int32_t* v2p_dev, int64_t v2p_len, int32_t* ids_dev,
                        kv_stream_t stream);

/* Per-layer store: row i of K goes to block 2*layer and row i of V to block
 * 2*layer+1 of token ids_dev[i], i.e. bytes anchor + (id + 2*layer*ps) * R and
 * anchor + (id + (2*layer+1)*ps) * R.
 * Source: _store_kv_layer's plain 3D assignment through the dense per-layer
 * views k_buffer[l][ids] = k, v_buffer[l][ids] = v (关键文件 memory_pool.py
 * and cache_move.py; build_mha_views' view bases).
 *  ids_dev  int32 [n] kernel-facing ids (kv_translate's output)
 *  k_dev    [n, H, D] contiguous, R bytes per row, 16-byte aligned
 *  v_dev    [n, H, D] contiguous, R bytes per row, 16-byte aligned
 * Duplicate ids (tombstones all map to id 0, the sink) leave the row with
 * some mix of the duplicates' words: which one wins is unspecified.
 * Device errors: an id outside [0, n_rows) sets KV_DEV_ERR_ROW, and an id
 * that kv_translate cannot produce (id % (ps*2L) >= ps, whose rows would land
 * in another layer's row-block) sets KV_DEV_ERR_FORM; its rows are skipped. */
int kv_store_layer(const kv_pool_t* pool, int32_t layer, const int32_t* ids_dev, int64_t n,
                   const void* k_dev, const void* v_dev, kv_stream_t stream);

/* All-layer store: kv_store_layer for every layer l in one launch, with
 * K_all[l] and V_all[l] as layer l's rows.
 * Source: the same assignment as kv_store_layer, over all 2L row-blocks of
 * the envelope (实现拆解 step 1).
 *  k_all_dev, v_all_dev  [L, n, H, D] contiguous (layer-major), 16-byte aligned
 * Device errors: as kv_store_layer. */
int kv_store_all_layers(const kv_pool_t* pool, const int32_t* ids_dev, int64_t n, const void* k_all_dev,
                        const void* v_all_dev, kv_stream_t stream);

/* Fused translate + per-layer store: exactly kv_translate of slots_dev (with
 * the optional page map) followed by kv_store_layer, in one launch and with
 * no id buffer: each task translates its own slot.
 * Source: translate_kv_loc_for_kernel (关键源码片段 multi_ended_allocator.py)
 * and _store_kv_layer (关键文件 memory_pool.py); the report's related
 * write-path change (关联脉络, PR #35245) translates the write location once
 * per forward batch, which this call folds into the store itself.
 *  slots_dev  int64 [n] token slots (negative = tombstone -> page-0 sink)
 *  v2p_dev    int32 [v2p_len] virtual -> physical page map, or NULL
 *  k_dev, v_dev  as kv_store_layer
 * Device errors: as kv_translate (KV_DEV_ERR_V2P, KV_DEV_ERR_ROW; the token
 * is then stored to the sink, as kv_translate's id 0 would be). */
int kv_store_layer_slots(const kv_pool_t* pool, int32_t layer, const int64_t* slots_dev, int64_t n,
                         const int32_t* v2p_dev, int64_t v2p_len, const void* k_dev, const void* v_dev,
                         kv_stream_t stream);

/* Fused translate + all-layer store: kv_translate followed by
 * kv_store_all_layers, in one launch.
 *  k_all_dev, v_all_dev  [L, n, H, D] contiguous (layer-major), 16-byte aligned */
int kv_store_all_layers_slots(const kv_pool_t* pool, const int64_t* slots_dev, int64_t n, const int32_t* v2p_dev,
                              int64_t v2p_len, const void* k_all_dev, const void* v_all_dev, kv_stream_t stream);

/* Block-table gather of one layer into packed K and V outputs.
 * Source: the read path the report describes -- each layer's K/V read
 * "through one contiguous tensor and one shared block table" (功能与动机) --
 * over build_mha_views' dense views.
 * For sequence s and every token j in [start_s, len_s):
 *    p = block_table[s * max_pages + j / ps]   (a physical page)
 *    o = j % ps; if p < 0 the token reads the sink (p = 0, o = 0)
 *    out_k[cu_out[s] + j - start_s] = K row of (p, o) for `layer`
 *    out_v[cu_out[s] + j - start_s] = V row of (p, o) for `layer`
 *  block_table_dev int32 [n_seqs, max_pages]
 *  seq_start_dev   int32 [n_seqs] first token of each window, or NULL for 0
 *  seq_len_dev     int32 [n_seqs] one past the last token
 *  cu_out_dev      int64 [n_seqs + 1] output row of each sequence's first
 *                  token; non-decreasing, cu_out[0] >= 0, and
 *                  cu_out[s+1] - cu_out[s] >= len_s - start_s
 *  out_k_dev, out_v_dev  [out_rows, H, D], 16-byte aligned
 * Output rows not covered by a token (gaps between sequences) are left
 * untouched. The kernel reads the row count cu_out[n_seqs] on the device, so
 * the call needs no host synchronization.
 * Device errors: KV_DEV_ERR_TABLE when some sequence has start_s < 0,
 * len_s > max_pages * ps, cu_out[s] < 0, cu_out[s+1] < cu_out[s] or a span
 * shorter than its token count, or when cu_out[n_seqs] > out_rows (rows past
 * out_rows are not written); KV_DEV_ERR_ROW when a page is >= num_pages (that
 * token is skipped). Every access stays in bounds whatever the metadata.
 * Where one page's rows of a layer (ps * 2R bytes, ps * R for MLA) fit in
 * 72 KiB, each table entry's rows are staged in shared memory by bulk copy and
 * bulk-copied out, with a bounded wait for the load (KV_DEV_ERR_TIMEOUT);
 * otherwise warps copy them through registers. The output is the same. */
int kv_gather_layer(const kv_pool_t* pool, int32_t layer, const int32_t* block_table_dev, int32_t n_seqs,
                    int32_t max_pages, const int32_t* seq_start_dev, const int32_t* seq_len_dev,
                    const int64_t* cu_out_dev, void* out_k_dev, void* out_v_dev, int64_t out_rows,
                    kv_stream_t stream);

/* Page-major gather plan. Many sequences often share pages (common
 * prefixes); a gather that visits the block table sequence by sequence reads
 * a shared page at unrelated times. kv_gather_plan orders the entries of a
 * block table by the page they name (a counting sort), and
 * kv_gather_layer_planned then visits them in that order, so all readers of a
 * page run together and L2 serves the repeats. The plan depends only on the
 * table and the windows, so one plan serves every layer of a step.
 * Source: the read path of the report (功能与动机: one contiguous tensor and
 * one shared block table per layer); the ordering is this library's.
 *
 * kv_gather_plan_bytes: size of the plan buffer for a table of n_seqs x
 *   max_pages entries: 4 * (4 + num_pages + 1 + n_seqs * max_pages) bytes
 *   (host only). n_seqs * max_pages must be < 2^31.
 * kv_gather_plan: builds the plan into plan_dev (device, plan_bytes long,
 *   4-byte aligned; the caller owns it and may reuse it until the table
 *   changes). Layout (int32): [0] entries in the plan, [1] n_seqs,
 *   [2] max_pages, [3] flags: bit 0 set when the page-major order pays
 *   (entries >= 1.5 x distinct pages), bit 1 set when the plan was built
 *   from a kernel-facing table (kv_gather_plan_kf); then num_pages + 1
 *   per-page offsets (the sort's workspace), then the entry indices
 *   s * max_pages + k grouped by page. With bit 0 clear (pages hardly
 *   shared) the planned gather keeps the table's own order, whose output
 *   writes stay sequential.
 *   Only entries holding tokens of [start_s, len_s) enter the plan; an entry
 *   naming a page >= num_pages sets KV_DEV_ERR_ROW and is left out. The
 *   table must not change while the plan builds (it is read twice, to count
 *   and to place); if it does, no write lands outside the plan, and an entry
 *   without a place sets KV_DEV_ERR_TABLE.
 * kv_gather_layer_planned: kv_gather_layer with the same arguments plus the
 *   plan built from the same block table, starts and lengths (plan_bytes: the
 *   size of its buffer, at least kv_gather_plan_bytes(), else KV_ERR_INVALID);
 *   the output is identical. A plan built for another table shape, or from
 *   a kernel-facing table, sets KV_DEV_ERR_TABLE and writes nothing; plan
 *   entries are bounds-checked one by one, so a stale or foreign plan never
 *   reads outside its buffer. Where one page's rows of a layer (ps * 2R
 *   bytes, ps * R for MLA) fit in 72 KiB, blocks of one warp stage each page
 *   once in shared memory and bulk-copy it to their readers (bounded waits
 *   for those loads: KV_DEV_ERR_TIMEOUT), two plan positions per block when
 *   n_seqs * max_pages >= num_pages (pages are then named several times
 *   over), one otherwise; larger pages are copied through registers by
 *   warps. The output is the same. */
int kv_gather_plan_bytes(const kv_pool_t* pool, int32_t n_seqs, int32_t max_pages, int64_t* plan_bytes);
int kv_gather_plan(const kv_pool_t* pool, const int32_t* block_table_dev, int32_t n_seqs, int32_t max_pages,
                   const int32_t* seq_start_dev, const int32_t* seq_len_dev, void* plan_dev, int64_t plan_bytes,
                   kv_stream_t stream);
int kv_gather_layer_planned(const kv_pool_t* pool, int32_t layer, const void* plan_dev, int64_t plan_bytes,
                            const int32_t* block_table_dev, int32_t n_seqs, int32_t max_pages,
                            const int32_t* seq_start_dev, const int32_t* seq_len_dev, const int64_t* cu_out_dev,
                            void* out_k_dev, void* out_v_dev, int64_t out_rows, kv_stream_t stream);

/* kv_gather_plan without any device memory from the caller beyond the plan.
 * The paper has no counterpart: this entry point exists for callers of this
 * library that cannot call cudaMalloc, such as code running inside a host
 * framework whose allocator reserved the device's memory up front and owns
 * it, or a serving loop that must not let an allocation (or the device-wide
 * synchronization a cudaMalloc or cudaFree may bring) into its steady state.
 * kv_gather_plan counts entries per page in the plan buffer itself; this
 * variant counts in a fixed array inside the library's device image and then
 * copies the resulting per-page offsets into the plan.
 *
 * Arguments, plan layout and device error bits are those of kv_gather_plan,
 * and plan_bytes must still be at least kv_gather_plan_bytes(). The plan
 * written is kv_gather_plan's up to the order of entries within one page
 * (that order is not fixed in either), and kv_gather_layer_planned takes it
 * unchanged. Calls no cudaMalloc or cudaFree and allocates nothing.
 *
 * Limit: pools of at most 65536 pages; larger pools return KV_ERR_CAPACITY
 * before anything is enqueued. The array (65537 int32 counters, 256 KiB + 4 B)
 * is held by every GPU that loads the library until the process exits.
 * Set-up: the first call on each device looks up the array's device address
 * with that device current (cudaGetSymbolAddress), and so does the first
 * call after the device's context was created anew (cudaDeviceReset); make
 * that first call before any stream capture. Sharing: every call uses the
 * same array, which keeps the previous call's contents; each call clears the
 * counters it uses on its stream first, so calls ordered on the GPU are
 * independent, but calls that overlap on the GPU (different streams, threads
 * or pools on one device) race on the array and give wrong plans: order them. */
int kv_gather_plan_noalloc(const kv_pool_t* pool, const int32_t* block_table_dev, int32_t n_seqs,
                           int32_t max_pages, const int32_t* seq_start_dev, const int32_t* seq_len_dev,
                           void* plan_dev, int64_t plan_bytes, kv_stream_t stream);

/* Move: copy every row-block (all layers' K and V, 2L rows) of token
 * src_ids[i] to token dst_ids[i].
 * Source: move_kv_cache / _move_kv_cache_impl (关键文件 memory_pool.py).
 *  src_ids_dev, dst_ids_dev  int32 [n] kernel-facing ids
 * Precondition: the src set and the dst set are disjoint and dst ids are
 * distinct; otherwise the result is unspecified (still in bounds).
 * Device errors: an id outside [0, n_rows) sets KV_DEV_ERR_ROW and an id
 * whose offset id % (ps*2L) is >= ps sets KV_DEV_ERR_FORM; that pair is
 * skipped. With rows of at least 128 bytes a pair's 2L rows are copied
 * through shared memory by bulk copies, in chunks of at most 18 KiB, with a
 * bounded wait for the loads (KV_DEV_ERR_TIMEOUT); smaller rows are copied
 * row by row through registers. */
int kv_move(const kv_pool_t* pool, const int32_t* src_ids_dev, const int32_t* dst_ids_dev, int64_t n,
            kv_stream_t stream);

/* Kernel-facing block table, prefix only: for each sequence s, the first
 * ceil(seq_len[s] / ps) entries (at most max_pages) of its virtual page list
 * are mapped through the virtual -> physical page map and scaled by the
 * row-blocks per page, out = phys * 2L, so that out * ps + offset is the
 * token's kernel-facing id (the id kv_translate gives the same virtual slot).
 * Entries past the prefix are left untouched.
 * Source: the report's read-path change (关联脉络, PR #35247: the read path's
 * kernel-facing page table is built once, translating only the prefix a
 * sequence uses) over translate_kv_loc_for_kernel's page arithmetic
 * (关键源码片段 multi_ended_allocator.py).
 *  virt_bt_dev  int32 [n_seqs, max_pages] virtual pages (negative = tombstone)
 *  seq_len_dev  int32 [n_seqs] tokens per sequence
 *  v2p_dev      int32 [v2p_len] virtual -> physical page map (negative = tombstone)
 *  out_bt_dev   int32 [n_seqs, max_pages]; may be virt_bt_dev itself (in place)
 * A tombstone becomes 0, the sink page (reads of it land in the sink, like a
 * clamped id). Device errors: a virtual page >= v2p_len sets KV_DEV_ERR_V2P,
 * a physical page >= num_pages sets KV_DEV_ERR_ROW (both write 0), and
 * seq_len[s] > max_pages * ps sets KV_DEV_ERR_TABLE (the prefix is capped). */
int kv_translate_block_table(const kv_pool_t* pool, const int32_t* virt_bt_dev, int32_t n_seqs, int32_t max_pages,
                             const int32_t* seq_len_dev, const int32_t* v2p_dev, int64_t v2p_len,
                             int32_t* out_bt_dev, kv_stream_t stream);

/* Gathers that read a kernel-facing block table directly: the table
 * kv_translate_block_table writes, whose entry for a page is phys * 2L, so
 * that entry * ps + o is the kernel-facing id of the token at offset o.
 * Source: the report's read path builds this prefix-only kernel-facing page
 * table once and reads through it (关联脉络, PR #35247), over
 * translate_kv_loc_for_kernel's id form (关键源码片段
 * multi_ended_allocator.py) and build_mha_views' dense views.
 *
 * kv_gather_layer_kf: kv_gather_layer with kf_table_dev in place of a
 *   physical table: for sequence s and token j in [start_s, len_s),
 *   e = kf_table[s * max_pages + j / ps] and the token's K and V rows are
 *   those of kernel-facing id e * ps + j % ps, i.e. page e / 2L, offset
 *   j % ps. A tombstoned virtual page (entry 0) therefore reads page 0, the
 *   sink page, at the token's own offset; a negative entry (never written by
 *   kv_translate_block_table) reads the sink row (page 0, offset 0) as in
 *   kv_gather_layer. Entries past a sequence's window are never read, so the
 *   prefix-only table suffices. Arguments, output layout and the other
 *   device error bits are kv_gather_layer's. Device errors: an entry >=
 *   num_pages * 2L sets KV_DEV_ERR_ROW and one that is not a multiple of 2L
 *   sets KV_DEV_ERR_FORM; that entry's tokens are skipped (their output rows
 *   are left untouched).
 * kv_gather_plan_kf: kv_gather_plan over a kernel-facing table (entries
 *   decoded as above; an off-grid entry sets KV_DEV_ERR_FORM and is left out
 *   of the plan). The plan records its table form in flag bit 1.
 * kv_gather_layer_planned_kf: kv_gather_layer_planned over a kernel-facing
 *   table with a plan from kv_gather_plan_kf; a plan built from a physical
 *   table sets KV_DEV_ERR_TABLE and writes nothing.
 * In an MLA pool 2L reads L throughout. */
int kv_gather_layer_kf(const kv_pool_t* pool, int32_t layer, const int32_t* kf_table_dev, int32_t n_seqs,
                       int32_t max_pages, const int32_t* seq_start_dev, const int32_t* seq_len_dev,
                       const int64_t* cu_out_dev, void* out_k_dev, void* out_v_dev, int64_t out_rows,
                       kv_stream_t stream);
int kv_gather_plan_kf(const kv_pool_t* pool, const int32_t* kf_table_dev, int32_t n_seqs, int32_t max_pages,
                      const int32_t* seq_start_dev, const int32_t* seq_len_dev, void* plan_dev, int64_t plan_bytes,
                      kv_stream_t stream);
int kv_gather_layer_planned_kf(const kv_pool_t* pool, int32_t layer, const void* plan_dev, int64_t plan_bytes,
                               const int32_t* kf_table_dev, int32_t n_seqs, int32_t max_pages,
                               const int32_t* seq_start_dev, const int32_t* seq_len_dev, const int64_t* cu_out_dev,
                               void* out_k_dev, void* out_v_dev, int64_t out_rows, kv_stream_t stream);

/* Read and clear the pool's device error word. Takes the word and zeroes it
 * in one atomic exchange, ordered on `stream` (one tiny kernel), synchronizes
 * `stream`, and writes the KV_DEV_ERR_* bits raised since the last read into
 * *dev_code. Bits that work still running on other streams raises later stay
 * in the word for the next read; none is lost. Two kv_pool_last_error calls
 * on one pool must not overlap (they share the slot the taken value passes
 * through). */
int kv_pool_last_error(const kv_pool_t* pool, kv_stream_t stream, int32_t* dev_code);

/* Name of a KV_OK / KV_ERR_* code (static string). */
const char* kv_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* GATHER_TRANSLATE_KV_GB300_KV_POOL_H */
