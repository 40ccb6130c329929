/*
 * kv_oracle.c -- plain CPU oracle for the unified page-major KV-cache pool.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the checker, not the product: only
 * the test suite, the package's smoke check and the benchmark's CPU-baseline
 * leg load it. The CUDA library never links, includes or calls it, and it
 * includes nothing from the CUDA library.
 *
 * What it follows: the prhub report "PR #34602 完整报告" on sglang PR #34602,
 * "feat(unified-memory): dense KV views for uniform-row MHA/SWA models".
 * Sections used:
 *   - 实现拆解 (implementation breakdown), step 1: the page envelope
 *     [L0_K*ps | L0_V*ps | L1_K*ps | ...] is 2L equal row-blocks; layer l's K
 *     is block 2l and its V is block 2l+1.
 *   - 关键源码片段 (key source snippets), unified_memory_pool.py: the tail pad
 *     is one page envelope (page_size * entry_bytes) and the raw buffer is
 *     total_bytes + tail pad.
 *   - 关键源码片段, multi_ended_allocator.py, translate_kv_loc_for_kernel:
 *     pages/offsets split, virtual->physical lookup, stride = ps * 2L,
 *     clamp to 0 (tombstone -1 goes to the page-0 sink).
 *   - 关键源码片段, layout/page_major.py, build_mha_views: row_bytes,
 *     page_bytes, n_rows, the uniform-row assert and the last-view-end assert.
 *   - 风险与影响 (risks), item 5: kernel-facing row count < 2^31.
 *
 * How it addresses bytes. Every routine works on a host byte array M that
 * mirrors the whole raw pool buffer (anchor + pool + tail pad). A row is
 * named by the envelope decomposition
 *
 *      byte(p, b, o) = anchor + p*page_bytes + b*(ps*R) + o*R
 *
 * (physical page p, row-block b in [0, 2L), offset o in [0, ps)). The
 * kernel-facing id form appears only where the interface hands ids out
 * (translate) or in (move), and the move decodes it back into (p, o).
 *
 * Everything is integer arithmetic and memcpy; K/V bytes are opaque.
 * No blocking, no fusion, no reordering: one row at a time, in input order.
 *
 * Parity pins (the tests that hold this file to the report rather than to
 * itself): hand-computed translate values, the layout table, a brute-force
 * bijection of (slot, block) onto the envelope rows, an independently built
 * strided [page, 2L, ps, H, D] numpy reference, round trips, and planted
 * mutations that each pin must catch.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Error bits an oracle routine returns (0 = clean). They describe the same
 * conditions the CUDA library reports through its device error word; the
 * numeric values are the oracle's own. */
#define ORA_E_ROW   1  /* a page / id addressed a row outside the pool        */
#define ORA_E_V2P   2  /* a virtual page index was past the page map          */
#define ORA_E_TABLE 4  /* gather metadata inconsistent (see ora_gather)        */
#define ORA_E_FORM  8  /* a move id was not of the form p*stride + o, o < ps  */

/* Check codes of ora_check_desc (the oracle's own numbering). */
#define ORA_OK          0
#define ORA_BAD_ARG     1
#define ORA_ASYMMETRIC  2
#define ORA_ID_BOUND    3
#define ORA_TAIL_PAD    4
#define ORA_ANCHOR      5

typedef struct {
    int32_t layer_num;   /* L                                   */
    int32_t head_num;    /* H (KV heads)                        */
    int32_t head_dim;    /* D                                   */
    int32_t v_head_dim;  /* must equal D (uniform rows)         */
    int32_t itemsize;    /* bytes per element (1 fp8, 2 bf16)   */
    int32_t page_size;   /* ps, tokens per page                 */
    int64_t num_pages;   /* P                                   */
    int64_t anchor;      /* byte offset of this sub-pool in raw */
    int32_t latent_only; /* 0: MHA/SWA, K and V rows per layer  */
                         /* 1: MLA, one latent row per layer    */
    int32_t reserved_;
} ora_desc;

/* Row-blocks per page and the K block of a layer. MHA/SWA pages hold 2L
 * blocks, K of layer l in block 2l and V in 2l+1 (实现拆解 step 1); MLA
 * pages hold L blocks, layer l's latent row in block l (实现拆解 step 2:
 * blocks_per_page() returns 2 * layer_num for MHA and layer_num for MLA). */
static int64_t blocks_of(const ora_desc* d) {
    return d->latent_only ? (int64_t)d->layer_num : 2 * (int64_t)d->layer_num;
}
static int64_t k_block(const ora_desc* d, int64_t layer) {
    return d->latent_only ? layer : 2 * layer;
}

/* ---------------------------------------------------------------- sizes */

/* Layout sizes, from build_mha_views (关键源码片段, page_major.py) and the
 * tail-pad rule of MHASubPoolSpec.view_tail_pad_bytes (关键源码片段,
 * unified_memory_pool.py). entry_bytes is never defined in the report; the
 * reading used here is the bytes of one token across every layer's K and V,
 * 2L*R, so the tail pad equals one page envelope, as build_mha_views' own
 * assert message says.
 *
 *   out[0] R          = H * D * itemsize           (row_bytes)
 *   out[1] E          = B * R                      (entry_bytes)
 *   out[2] page_bytes = ps * B * R
 *   out[3] total      = P * page_bytes             (one sub-pool per pool)
 *   out[4] tail_pad   = ps * E
 *   out[5] n_rows     = P * B * ps                 (kernel-facing rows)
 *   out[6] last_view_end = anchor + (B-1)*ps*R + n_rows*R
 * with B = 2L row-blocks per page for MHA/SWA and B = L for MLA (the MLA
 * views reach past the last envelope the same way, so the same one-envelope
 * tail pad is read for them).
 */
void ora_sizes(const ora_desc* d, int64_t out[7]) {
    int64_t R = (int64_t)d->head_num * d->head_dim * d->itemsize;
    int64_t blocks = blocks_of(d);
    int64_t page_bytes = (int64_t)d->page_size * blocks * R;
    int64_t n_rows = d->num_pages * blocks * d->page_size;
    out[0] = R;
    out[1] = blocks * R;
    out[2] = page_bytes;
    out[3] = d->num_pages * page_bytes;
    out[4] = (int64_t)d->page_size * (blocks * R);
    out[5] = n_rows;
    out[6] = d->anchor + (blocks - 1) * d->page_size * R + n_rows * R;
}

/* Start-up gates, in the order the report lists them:
 *  - uniform rows: head_dim == v_head_dim (build_mha_views' first assert;
 *    风险与影响 item 4 rejects asymmetric-KV models);
 *  - the anchor is a multiple of the item size (build_mha_views);
 *  - kernel-facing row count P * 2L * ps below 2^31 (_assert_kernel_id_bound,
 *    实现拆解 step 2 and 风险与影响 item 5);
 *  - the raw buffer reaches the last view's end (build_mha_views' last
 *    assert). raw_bytes < 0 skips this check. */
int ora_check_desc(const ora_desc* d, int64_t raw_bytes) {
    if (d->layer_num < 1 || d->head_num < 1 || d->head_dim < 1 ||
        d->itemsize < 1 || d->page_size < 1 || d->num_pages < 1 || d->anchor < 0)
        return ORA_BAD_ARG;
    /* unified_memory_supported_for_model: use_mla_backend or not has_asymmetric_kv */
    if (!d->latent_only && d->head_dim != d->v_head_dim) return ORA_ASYMMETRIC;
    if (d->anchor % d->itemsize != 0) return ORA_ANCHOR;
    /* rows = P * 2L * ps, compared against 2^31 without overflowing: every
     * factor is positive, so test by successive division. */
    {
        int64_t limit = ((int64_t)1 << 31) - 1;
        int64_t blocks = blocks_of(d);
        if (d->num_pages > limit / blocks) return ORA_ID_BOUND;
        if (d->num_pages * blocks > limit / d->page_size) return ORA_ID_BOUND;
    }
    if (raw_bytes >= 0) {
        int64_t s[7];
        ora_sizes(d, s);
        if (s[6] > raw_bytes) return ORA_TAIL_PAD;
    }
    return ORA_OK;
}

/* byte(p, b, o): envelope decomposition (实现拆解 step 1). */
static int64_t env_byte(const ora_desc* d, int64_t p, int64_t b, int64_t o) {
    int64_t s[7];
    ora_sizes(d, s);
    int64_t R = s[0], page_bytes = s[2];
    return d->anchor + p * page_bytes + b * ((int64_t)d->page_size * R) + o * R;
}

/* -------------------------------------------------------------- translate */

/* Locate a token slot t in the envelope: which physical page and offset its
 * rows live at. Follows translate_kv_loc_for_kernel (关键源码片段,
 * multi_ended_allocator.py): page = t // ps, offset = t % ps, the page goes
 * through the virtual->physical map when one is given, and a negative
 * result is clamped to the page-0 sink, i.e. (page 0, offset 0).
 *
 * Readings where the report is silent: a negative slot is a tombstone and
 * needs no lookup; any negative map entry is a tombstone; a page index past
 * the map, or a physical page >= P, is an error that also lands on the sink.
 * Returns error bits; *p and *o receive the location and *sink is set
 * when the slot landed on the sink. */
static int locate_slot(const ora_desc* d, int64_t t, const int32_t* v2p,
                       int64_t v2p_len, int64_t* p, int64_t* o, int* sink) {
    *p = 0;
    *o = 0;
    *sink = 1;
    if (t < 0) return 0;                       /* tombstone -> sink */
    int64_t ps = d->page_size;
    int64_t page = t / ps;
    int64_t off = t % ps;
    int64_t phys = page;
    if (v2p != NULL) {
        if (page >= v2p_len) return ORA_E_V2P;
        phys = v2p[page];
    }
    if (phys < 0) return 0;                    /* tombstoned page -> sink */
    if (phys >= d->num_pages) return ORA_E_ROW;
    *p = phys;
    *o = off;
    *sink = 0;
    return 0;
}

/* Token slots -> kernel-facing int32 ids (translate_kv_loc_for_kernel):
 *     id = phys * (ps * 2L) + t % ps, clamped to 0 for tombstones.
 * This is the report's closed form kernel_id(t) written out as stated, with
 * kernel_page_multiplier fixed to blocks_per_page() = 2L, or L for MLA
 * (实现拆解 step 3). */
int ora_translate(const ora_desc* d, const int64_t* slots, int64_t n,
                  const int32_t* v2p, int64_t v2p_len, int32_t* ids) {
    int err = 0;
    int64_t stride = (int64_t)d->page_size * blocks_of(d);
    for (int64_t i = 0; i < n; ++i) {
        int64_t p, o;
        int sink;
        err |= locate_slot(d, slots[i], v2p, v2p_len, &p, &o, &sink);
        ids[i] = (int32_t)(p * stride + o);
    }
    return err;
}

/* Test only: translate with an explicit kernel_page_multiplier m,
 *     id = phys * (ps * m) + t % ps   (tombstones -> 0).
 * The report keeps such an override solely so tests can pin the
 * "multiplier-1 collapse" (评论区精华; 风险与影响 item 1): with m = 1 the ids
 * are physical slot ids, and a dense per-layer view then puts block b of a
 * token at view row id + b*ps, i.e. onto rows of other tokens, silently. The
 * library has no such parameter: its multiplier is always blocks_per_page(). */
int ora_translate_multiplier(const ora_desc* d, const int64_t* slots, int64_t n, int32_t m, int32_t* ids) {
    int err = 0;
    int64_t stride = (int64_t)d->page_size * m;
    for (int64_t i = 0; i < n; ++i) {
        int64_t p, o;
        int sink;
        err |= locate_slot(d, slots[i], NULL, 0, &p, &o, &sink);
        ids[i] = (int32_t)(p * stride + o);
    }
    return err;
}

/* Byte offset in M of the row of (slot, block), or -1 when the slot is a
 * tombstone or an error (both land on the sink). Used by tests that check a
 * full-size run one sampled row at a time. */
int64_t ora_slot_row_byte(const ora_desc* d, int64_t slot, const int32_t* v2p,
                          int64_t v2p_len, int32_t block) {
    int64_t p, o;
    int sink;
    int err = locate_slot(d, slot, v2p, v2p_len, &p, &o, &sink);
    if (err != 0 || sink) return -1;
    return env_byte(d, p, block, o);
}

/* ------------------------------------------------------------------ store */

/* Per-layer store: _store_kv_layer's "plain 3D assignment" (关键文件,
 * memory_pool.py / cache_move.py) through build_mha_views' views. Row i's K
 * goes to block 2l and its V to block 2l+1 of the page that slot i lives on
 * (实现拆解 step 1). K and V are [n, H, D] contiguous, R bytes per row.
 * Rows are written in input order; several tombstones all land on the sink
 * rows (page 0, offset 0), the last one written stays.
 *
 * MLA pools store one latent row per token (K only, block l); V is unused.
 *
 * With M == NULL nothing is copied: the pass records, for every row i, the
 * byte offsets it would write (kdst[i], vdst[i], -1 for MLA's absent V);
 * tests use this to check a full-size run without a host mirror of the
 * pool. */
static int store_pass(const ora_desc* d, uint8_t* M, int32_t layer, const int64_t* slots,
                      int64_t n, const int32_t* v2p, int64_t v2p_len,
                      const uint8_t* K, const uint8_t* V, int64_t* kdst, int64_t* vdst) {
    int64_t s[7];
    ora_sizes(d, s);
    int64_t R = s[0];
    int err = 0;
    if (layer < 0 || layer >= d->layer_num) return ORA_E_ROW;
    for (int64_t i = 0; i < n; ++i) {
        int64_t p, o;
        int sink;
        err |= locate_slot(d, slots[i], v2p, v2p_len, &p, &o, &sink);
        int64_t kb = env_byte(d, p, k_block(d, layer), o);
        int64_t vb = d->latent_only ? -1 : env_byte(d, p, k_block(d, layer) + 1, o);
        if (M != NULL) {
            memcpy(M + kb, K + i * R, (size_t)R);
            if (vb >= 0) memcpy(M + vb, V + i * R, (size_t)R);
        } else {
            kdst[i] = kb;
            vdst[i] = vb;
        }
    }
    return err;
}

int ora_store(const ora_desc* d, uint8_t* M, int32_t layer, const int64_t* slots,
              int64_t n, const int32_t* v2p, int64_t v2p_len,
              const uint8_t* K, const uint8_t* V) {
    if (M == NULL) return -1;
    return store_pass(d, M, layer, slots, n, v2p, v2p_len, K, V, NULL, NULL);
}

int ora_store_rows(const ora_desc* d, int32_t layer, const int64_t* slots, int64_t n,
                   const int32_t* v2p, int64_t v2p_len, int64_t* kdst, int64_t* vdst) {
    return store_pass(d, NULL, layer, slots, n, v2p, v2p_len, NULL, NULL, kdst, vdst);
}

/* All-layer store: ora_store for l = 0..L-1 with K_all[l], V_all[l]; the
 * inputs are [L, n, H, D], layer-major. */
int ora_store_all(const ora_desc* d, uint8_t* M, const int64_t* slots, int64_t n,
                  const int32_t* v2p, int64_t v2p_len,
                  const uint8_t* K_all, const uint8_t* V_all) {
    int64_t s[7];
    ora_sizes(d, s);
    int64_t R = s[0];
    int err = 0;
    for (int32_t l = 0; l < d->layer_num; ++l)
        err |= ora_store(d, M, l, slots, n, v2p, v2p_len,
                         K_all + (int64_t)l * n * R, V_all ? V_all + (int64_t)l * n * R : NULL);
    return err;
}

/* ----------------------------------------------------------------- gather */

static int decode_id(const ora_desc* d, int64_t id, int64_t* p, int64_t* o);

/* Block-table read of one layer into packed [sum, H, D] K and V outputs: the
 * read the backends do through "one contiguous tensor + one shared block
 * table" (功能与动机). The report gives no gather call, so the plainest one
 * is used: for sequence s and token j in [start_s, len_s), the page is
 * bt[s][j / ps] (a physical page; a negative entry is a tombstone and reads
 * the sink (page 0, offset 0), as translate clamps), the offset j % ps, and
 * the output row cu[s] + j - start_s.
 *
 * ORA_E_TABLE is raised, per sequence, when start_s < 0, len_s > maxp*ps,
 * cu[s] < 0, cu[s+1] < cu[s], or cu[s+1] - cu[s] < len_s - start_s; and when
 * cu[S] > out_rows. A token whose page index falls outside [0, maxp), whose
 * j is negative, or whose output row falls outside [0, out_rows) is skipped.
 * A page >= P raises ORA_E_ROW and the token is skipped. Skipped tokens leave
 * their output rows untouched. */
static int gather_pass(const ora_desc* d, const uint8_t* M, int32_t layer,
                       const int32_t* bt, int kernel_facing, int32_t n_seqs, int32_t max_pages,
                       const int32_t* seq_start, const int32_t* seq_len,
                       const int64_t* cu, uint8_t* outK, uint8_t* outV, int64_t out_rows,
                       int64_t* ksrc, int64_t* vsrc) {
    int64_t s7[7];
    ora_sizes(d, s7);
    int64_t R = s7[0];
    int64_t ps = d->page_size;
    int err = 0;
    if (layer < 0 || layer >= d->layer_num) return ORA_E_ROW;
    if (n_seqs > 0 && cu[n_seqs] > out_rows) err |= ORA_E_TABLE;
    for (int32_t s = 0; s < n_seqs; ++s) {
        int64_t st = seq_start ? seq_start[s] : 0;
        int64_t ln = seq_len[s];
        if (st < 0 || ln > (int64_t)max_pages * ps || cu[s] < 0 || cu[s + 1] < cu[s] ||
            cu[s + 1] - cu[s] < ln - st)
            err |= ORA_E_TABLE;
        for (int64_t j = st; j < ln; ++j) {
            if (j < 0) continue;
            int64_t k = j / ps;
            if (k >= max_pages) continue;
            int64_t p = bt[(int64_t)s * max_pages + k];
            int64_t o = j % ps;
            if (p < 0) { p = 0; o = 0; }
            else if (kernel_facing) {
                /* the entry is a kernel-facing page (ora_block_table_kf): the
                 * token's kernel-facing id is entry * ps + offset, decoded
                 * back into (page, offset) as a move decodes its ids */
                int e = decode_id(d, p * ps + o, &p, &o);
                if (e != 0) { err |= e; continue; }
            }
            if (p >= d->num_pages) { err |= ORA_E_ROW; continue; }
            int64_t r = cu[s] + (j - st);
            if (r < 0 || r >= out_rows) continue;
            int64_t kb = env_byte(d, p, k_block(d, layer), o);
            int64_t vb = d->latent_only ? -1 : env_byte(d, p, k_block(d, layer) + 1, o);
            if (M != NULL) {
                memcpy(outK + r * R, M + kb, (size_t)R);
                if (vb >= 0) memcpy(outV + r * R, M + vb, (size_t)R);
            } else {
                ksrc[r] = kb;
                vsrc[r] = vb;
            }
        }
    }
    return err;
}

int ora_gather(const ora_desc* d, const uint8_t* M, int32_t layer,
               const int32_t* bt, int32_t n_seqs, int32_t max_pages,
               const int32_t* seq_start, const int32_t* seq_len,
               const int64_t* cu, uint8_t* outK, uint8_t* outV, int64_t out_rows) {
    if (M == NULL) return -1;
    return gather_pass(d, M, layer, bt, 0, n_seqs, max_pages, seq_start, seq_len, cu,
                       outK, outV, out_rows, NULL, NULL);
}

/* Address mode of ora_gather: ksrc[r] / vsrc[r] receive the pool byte offset
 * output row r reads (rows no token covers are left as the caller set them). */
int ora_gather_rows(const ora_desc* d, int32_t layer, const int32_t* bt, int32_t n_seqs,
                    int32_t max_pages, const int32_t* seq_start, const int32_t* seq_len,
                    const int64_t* cu, int64_t out_rows, int64_t* ksrc, int64_t* vsrc) {
    return gather_pass(d, NULL, layer, bt, 0, n_seqs, max_pages, seq_start, seq_len, cu,
                       NULL, NULL, out_rows, ksrc, vsrc);
}

/* Gather through a kernel-facing block table, the read side of the report's
 * prefix-only kernel-facing page table (关联脉络, PR #35247; the table is
 * ora_block_table_kf's output). Reading taken: an entry e names the page
 * whose token at offset o has the kernel-facing id e * ps + o, the id
 * translate_kv_loc_for_kernel gives that token (关键源码片段
 * multi_ended_allocator.py), so the gather decodes that id into (page,
 * offset) exactly as a move decodes its ids and then reads as ora_gather.
 * Consequences: a tombstoned virtual page, which the table build turns into
 * entry 0, reads page 0 (the sink page) at the token's own offset; an entry
 * that is not a multiple of the row-blocks per page raises ORA_E_FORM and
 * an entry at or past P * 2L raises ORA_E_ROW (the token is skipped); a
 * negative entry, which the table build never writes, reads the sink row
 * (page 0, offset 0) as in ora_gather. Metadata checks are ora_gather's. */
int ora_gather_kf(const ora_desc* d, const uint8_t* M, int32_t layer,
                  const int32_t* kf_bt, int32_t n_seqs, int32_t max_pages,
                  const int32_t* seq_start, const int32_t* seq_len,
                  const int64_t* cu, uint8_t* outK, uint8_t* outV, int64_t out_rows) {
    if (M == NULL) return -1;
    return gather_pass(d, M, layer, kf_bt, 1, n_seqs, max_pages, seq_start, seq_len, cu,
                       outK, outV, out_rows, NULL, NULL);
}

/* Address mode of ora_gather_kf (see ora_gather_rows). */
int ora_gather_kf_rows(const ora_desc* d, int32_t layer, const int32_t* kf_bt, int32_t n_seqs,
                       int32_t max_pages, const int32_t* seq_start, const int32_t* seq_len,
                       const int64_t* cu, int64_t out_rows, int64_t* ksrc, int64_t* vsrc) {
    return gather_pass(d, NULL, layer, kf_bt, 1, n_seqs, max_pages, seq_start, seq_len, cu,
                       NULL, NULL, out_rows, ksrc, vsrc);
}

/* ------------------------------------------------------------------- move */

/* Decode a kernel-facing id into (page, offset): p = id / (ps*2L),
 * o = id % (ps*2L), which must be < ps for an id that translate can produce. */
static int decode_id(const ora_desc* d, int64_t id, int64_t* p, int64_t* o) {
    int64_t stride = (int64_t)d->page_size * blocks_of(d);
    int64_t n_rows = d->num_pages * stride;
    if (id < 0 || id >= n_rows) return ORA_E_ROW;
    *p = id / stride;
    *o = id % stride;
    if (*o >= d->page_size) return ORA_E_FORM;
    return 0;
}

/* move_kv_cache: copy all 2L rows (every layer's K and V) of token src_i to
 * token dst_i (关键文件, memory_pool.py _move_kv_cache_impl). The ids are
 * kernel-facing. Snapshot semantics: every source row is read before any
 * destination row is written. A pair whose src or dst id fails to decode
 * is skipped and its error bits are returned. */
int ora_move(const ora_desc* d, uint8_t* M, const int32_t* src_ids,
             const int32_t* dst_ids, int64_t m) {
    int64_t s7[7];
    ora_sizes(d, s7);
    int64_t R = s7[0];
    int64_t blocks = blocks_of(d);
    int err = 0;
    if (m <= 0) return 0;
    uint8_t* snap = (uint8_t*)malloc((size_t)(m * blocks * R));
    uint8_t* ok = (uint8_t*)malloc((size_t)m);
    if (!snap || !ok) { free(snap); free(ok); return -1; }
    for (int64_t i = 0; i < m; ++i) {
        int64_t ps_ = 0, os_ = 0, pd_ = 0, od_ = 0;
        int e = decode_id(d, src_ids[i], &ps_, &os_) | decode_id(d, dst_ids[i], &pd_, &od_);
        err |= e;
        ok[i] = (e == 0);
        if (!ok[i]) continue;
        for (int64_t b = 0; b < blocks; ++b)
            memcpy(snap + (i * blocks + b) * R, M + env_byte(d, ps_, b, os_), (size_t)R);
    }
    for (int64_t i = 0; i < m; ++i) {
        if (!ok[i]) continue;
        int64_t pd_ = 0, od_ = 0;
        decode_id(d, dst_ids[i], &pd_, &od_);
        for (int64_t b = 0; b < blocks; ++b)
            memcpy(M + env_byte(d, pd_, b, od_), snap + (i * blocks + b) * R, (size_t)R);
    }
    free(snap);
    free(ok);
    return err;
}

/* Byte offset in M of block b of the token a kernel-facing id names, or -1
 * when the id does not decode. */
int64_t ora_id_row_byte(const ora_desc* d, int64_t id, int32_t block) {
    int64_t p, o;
    if (decode_id(d, id, &p, &o) != 0) return -1;
    return env_byte(d, p, block, o);
}

/* Address mode of ora_move: for pair i and block b, src_bytes[i*2L + b] and
 * dst_bytes[i*2L + b] receive the byte offsets the move reads and writes, or
 * -1 for a skipped pair. Returns the same error bits as ora_move. */
int ora_move_rows(const ora_desc* d, const int32_t* src_ids, const int32_t* dst_ids,
                  int64_t m, int64_t* src_bytes, int64_t* dst_bytes) {
    int64_t blocks = blocks_of(d);
    int err = 0;
    for (int64_t i = 0; i < m; ++i) {
        int64_t ps_ = 0, os_ = 0, pd_ = 0, od_ = 0;
        int e = decode_id(d, src_ids[i], &ps_, &os_) | decode_id(d, dst_ids[i], &pd_, &od_);
        err |= e;
        for (int64_t b = 0; b < blocks; ++b) {
            src_bytes[i * blocks + b] = e ? -1 : env_byte(d, ps_, b, os_);
            dst_bytes[i * blocks + b] = e ? -1 : env_byte(d, pd_, b, od_);
        }
    }
    return err;
}

/* ------------------------------------------------------- block table build */

/* Kernel-facing block table, prefix only. The report moves read-path
 * translation into a "prefix-only" kernel-facing page-table build (关联脉络,
 * PR #35247; 评论区精华). Reading taken: for sequence s only the pages that
 * hold its tokens [0, len_s) -- the first ceil(len_s / ps) entries, at most
 * max_pages -- are translated; later entries are left as they are. Each
 * translated entry is the physical page scaled by the row-blocks per page,
 * phys * 2L, so that entry * ps + offset is the token's kernel-facing id, the
 * same id translate_kv_loc_for_kernel gives the slot (关键源码片段
 * multi_ended_allocator.py). A tombstone (negative virtual page or negative
 * map entry) becomes 0, the sink page. A virtual page past the map raises
 * ORA_E_V2P, a physical page >= P raises ORA_E_ROW; both write 0. len_s >
 * max_pages * ps raises ORA_E_TABLE (the prefix is capped at max_pages). */
int ora_block_table_kf(const ora_desc* d, const int32_t* virt, int32_t n_seqs, int32_t max_pages,
                       const int32_t* seq_len, const int32_t* v2p, int64_t v2p_len, int32_t* out) {
    int64_t ps = d->page_size;
    int64_t blocks = blocks_of(d);
    int err = 0;
    for (int32_t s = 0; s < n_seqs; ++s) {
        int64_t len = seq_len[s];
        int64_t np = len > 0 ? (len + ps - 1) / ps : 0;
        if (np > max_pages) {
            err |= ORA_E_TABLE;
            np = max_pages;
        }
        for (int64_t k = 0; k < np; ++k) {
            int64_t vp = virt[(int64_t)s * max_pages + k];
            int64_t phys = -1;
            if (vp >= 0) {
                if (vp >= v2p_len) err |= ORA_E_V2P;
                else phys = v2p[vp];
            }
            if (phys >= d->num_pages) {
                err |= ORA_E_ROW;
                phys = -1;
            }
            out[(int64_t)s * max_pages + k] = (int32_t)(phys < 0 ? 0 : phys * blocks);
        }
    }
    return err;
}

/* ------------------------------------------------ full -> SWA token mapping */

/* Translate through a token map first. A hybrid model keeps a full-attention
 * sub-pool and a sliding-window sub-pool in the same dense id space (实现拆解
 * step 2: init_unified_swa_pools moves into the new id space) and addresses a
 * token of an SWA layer through the full -> SWA token mapping, whose cleared
 * entries are tombstones (功能与动机 / 关联脉络: clear_full_to_swa_mapping, PR
 * #35773). Reading taken: slot t of the full pool becomes t' = tmap[t]; t < 0
 * or t' < 0 is a tombstone (id 0, the sink); t >= tmap_len raises ORA_E_V2P
 * and gives id 0; t' then goes through ora_translate's page logic (with the
 * SWA pool's optional page map). */
int ora_translate_mapped(const ora_desc* d, const int64_t* slots, int64_t n, const int64_t* tmap,
                         int64_t tmap_len, const int32_t* v2p, int64_t v2p_len, int32_t* ids) {
    int err = 0;
    int64_t stride = (int64_t)d->page_size * blocks_of(d);
    for (int64_t i = 0; i < n; ++i) {
        int64_t t = slots[i];
        int64_t mapped = -1;
        if (t >= 0) {
            if (t >= tmap_len) err |= ORA_E_V2P;
            else mapped = tmap[t];
        }
        int64_t p, o;
        int sink;
        err |= locate_slot(d, mapped, v2p, v2p_len, &p, &o, &sink);
        ids[i] = (int32_t)(p * stride + o);
    }
    return err;
}
