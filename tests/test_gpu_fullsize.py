"""GPU parity at the workloads' full sizes (8 GiB to 119 GiB pools).

No host mirror fits, so the oracle runs in address mode: for every row a call
writes or reads it names the pool byte offset (its envelope decomposition),
and the test checks on the device, with plain torch indexing, that
  * every row a store writes holds that input row at the oracle's offset,
  * every gathered row equals the content at the oracle's source offset
    (the sentinel pattern, or the row a store put there),
  * every moved row equals the source row's content,
  * no other row of the pool (nor its tail pad) changed: the set of rows
    that differ from the sentinel is exactly the set the oracle predicts.
Every output row is checked, not a sample. Tombstoned tokens go to the sink
rows, which follow the sink rule of gpu_util.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import gather_translate_kv_gb300 as gt
import oracle
import synth
from gpu_util import as_rows, dev_bits

pytestmark = pytest.mark.gpu

FILL = 31337


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gather_translate_kv_gb300 import build

    build.build()
    oracle.build()


class Full:
    """A full-size device pool filled with the sentinel, and its oracle."""

    def __init__(self, shape: synth.Shape):
        self.shape = shape
        self.o = oracle.Oracle(oracle.Geometry(shape.layer_num, shape.head_num, shape.head_dim, shape.itemsize,
                                               shape.page_size, shape.num_pages))
        self.sizes = self.o.sizes()
        self.R = self.sizes["row_bytes"]
        nbytes = self.o.raw_bytes()
        free, _ = torch.cuda.mem_get_info()
        if nbytes + (12 << 30) > free:
            pytest.skip(f"skipped: {free / 2**30:.1f} GiB free, the {shape.name} pool needs {nbytes / 2**30:.1f} GiB")
        self.raw = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        synth.fill_sentinel_torch(self.raw, FILL)
        self.rows = self.raw.view(-1, self.R)  # anchor 0: every row offset is a multiple of R
        self.pool = gt.kv_pool_create(gt.make_desc(shape.layer_num, shape.head_num, shape.head_dim, shape.itemsize,
                                                   shape.page_size, shape.num_pages), self.raw)
        self.written = []  # row indices (offset // R) the oracle says were written
        self.sinks = {self.o.slot_row_byte(0, b) // self.R for b in range(2 * shape.layer_num)}

    def close(self):
        gt.kv_pool_destroy(self.pool)
        del self.rows, self.raw
        torch.cuda.empty_cache()

    def translate(self, slots: np.ndarray) -> torch.Tensor:
        ids = torch.empty(slots.size, dtype=torch.int32, device="cuda")
        gt.kv_translate(self.pool, torch.from_numpy(slots).cuda(), ids)
        return ids

    def sentinel(self, offsets: np.ndarray) -> torch.Tensor:
        return synth.sentinel_rows_torch(FILL, torch.from_numpy(offsets).cuda(), self.R)

    def check_store(self, layer, slots, K, V, ids=None):
        """Store one layer through the C ABI and check every written row."""
        kd, vd, err = self.o.store_rows(layer, slots)
        ids = self.translate(slots) if ids is None else ids
        Kd, Vd = torch.from_numpy(as_rows(K, self.R)).cuda(), torch.from_numpy(as_rows(V, self.R)).cuda()
        gt.kv_store_layer(self.pool, layer, ids, Kd, Vd)
        assert gt.kv_pool_last_error(self.pool) == dev_bits(err) == 0
        self._check_rows(slots, kd, vd, Kd, Vd)
        return kd, vd, Kd, Vd

    def _check_rows(self, slots, kd, vd, Kd, Vd):
        live = torch.from_numpy(np.nonzero(slots >= 0)[0]).cuda()
        for off, src in ((kd, Kd), (vd, Vd)):
            idx = torch.from_numpy(off // self.R).cuda()
            got = self.rows[idx[live]]
            assert torch.equal(got, src[live]), "stored rows differ from the inputs at the oracle's offsets"
            self.written.append(idx[live])

    def check_untouched(self, chunk_rows: int = 1 << 22):
        """Rows that differ from the sentinel == rows the oracle says were
        written (sink rows aside); the tail pad never differs."""
        want = torch.unique(torch.cat(self.written)) if self.written else \
            torch.zeros(0, dtype=torch.int64, device="cuda")
        n = self.rows.shape[0]
        buf = torch.empty(min(chunk_rows, n) * self.R, dtype=torch.uint8, device="cuda")
        got = []
        for r0 in range(0, n, chunk_rows):
            r1 = min(n, r0 + chunk_rows)
            b = buf[: (r1 - r0) * self.R]
            synth.fill_sentinel_torch(b, FILL, byte_offset=r0 * self.R)
            diff = (self.rows[r0:r1] != b.view(-1, self.R)).any(dim=1)
            got.append(torch.nonzero(diff).flatten() + r0)
        got = torch.cat(got)
        if self.sinks:
            sinks = torch.tensor(sorted(self.sinks), device="cuda")
            got = got[~torch.isin(got, sinks)]
            want = want[~torch.isin(want, sinks)]
        n_pool_rows = self.sizes["total"] // self.R
        assert int((got >= n_pool_rows).sum()) == 0, "the tail pad changed"
        assert got.numel() == want.numel() and torch.equal(got, want), \
            f"{got.numel()} rows changed, the oracle predicts {want.numel()}"

    def expected_reads(self, offsets: np.ndarray, stored: list) -> torch.Tensor:
        """Content at byte offsets: the sentinel, or the row a store put there.
        `stored` = [(offsets int64[n], rows uint8[n, R] on the device)]."""
        exp = self.sentinel(offsets)
        offs_d = torch.from_numpy(offsets).cuda()
        for so, srows in stored:
            so_d = torch.from_numpy(so).cuda()
            order = torch.argsort(so_d)
            so_s = so_d[order]
            pos = torch.searchsorted(so_s, offs_d).clamp_(max=max(0, so_s.numel() - 1))
            hit = so_s[pos] == offs_d if so_s.numel() else torch.zeros_like(offs_d, dtype=torch.bool)
            exp[hit] = srows[order[pos[hit]]]
        return exp

    def check_gather(self, layer, gb: synth.GatherBatch, stored: list, planned: bool = False,
                     kernel_facing: bool = False):
        """Gather one layer (table order, or through a page-major plan) and
        compare every output row with the oracle's source offsets. With
        kernel_facing, the same physical pages are reached through a virtual
        table and a random page map: the library builds the kernel-facing
        table (checked against the oracle's) and gathers through it."""
        d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
        ok = torch.empty((gb.total, self.R), dtype=torch.uint8, device="cuda")
        ov = torch.empty_like(ok)
        ln, cu, st = d(gb.seq_len), d(gb.cu), d(gb.seq_start)
        if kernel_facing:
            P = self.shape.num_pages
            rng = np.random.default_rng(4321 + layer)
            v2p = np.zeros(P, np.int32)
            v2p[1:] = 1 + rng.permutation(P - 1)  # a bijection of pages 1..P-1
            inv = np.zeros(P, np.int32)
            inv[v2p] = np.arange(P, dtype=np.int32)
            virt = np.where(gb.block_table < 0, -1, inv[np.maximum(gb.block_table, 0)]).astype(np.int32)
            kf_ref, err = self.o.block_table_kf(virt, gb.seq_len, v2p, out=np.zeros_like(virt))
            assert err == 0
            ks, vs, err = self.o.gather_rows(layer, kf_ref, gb.seq_len, gb.cu, gb.seq_start, kernel_facing=True)
            kf = torch.zeros(virt.shape, dtype=torch.int32, device="cuda")
            gt.kv_translate_block_table(self.pool, d(virt), ln, d(v2p), kf)
            assert torch.equal(kf, d(kf_ref)), "kernel-facing table differs"
            if planned:
                plan = gt.kv_gather_plan_kf(self.pool, kf, ln, st)
                gt.kv_gather_layer_planned_kf(self.pool, layer, plan, kf, ln, cu, ok, ov, st)
            else:
                gt.kv_gather_layer_kf(self.pool, layer, kf, ln, cu, ok, ov, st)
        else:
            ks, vs, err = self.o.gather_rows(layer, gb.block_table, gb.seq_len, gb.cu, gb.seq_start)
            bt = d(gb.block_table)
            if planned:
                plan = gt.kv_gather_plan(self.pool, bt, ln, st)
                gt.kv_gather_layer_planned(self.pool, layer, plan, bt, ln, cu, ok, ov, st)
            else:
                gt.kv_gather_layer(self.pool, layer, bt, ln, cu, ok, ov, st)
        assert err == 0 and (ks >= 0).all()
        assert gt.kv_pool_last_error(self.pool) == 0
        assert torch.equal(ok, self.expected_reads(ks, stored[0])), f"gathered K of layer {layer} differs"
        assert torch.equal(ov, self.expected_reads(vs, stored[1])), f"gathered V of layer {layer} differs"


def _vals(shape, n, layer, seed_extra=0):
    return synth.kv_pair(shape, n, layer, seed=shape.seed + seed_extra)


def test_decode_llama3_8b_full():
    """Workload 2 (8 GiB pool): gathers of 256 x 4096 tokens on the fresh
    pool, the per-layer decode store for all 32 layers, gathers that read the
    new tokens (through physical and kernel-facing tables, in table and
    page-major order), and the 8192-token move."""
    sh = synth.SHAPES[2]
    F = Full(sh)
    gb = synth.gather_batch(sh)
    for layer in (0, 31):
        F.check_gather(layer, gb, ([], []))
    stored = {}
    for layer in range(sh.layer_num):
        slots = synth.store_slots(sh, layer)
        K, V = _vals(sh, slots.size, layer)
        kd, vd, Kd, Vd = F.check_store(layer, slots, K, V)
        stored[layer] = ((kd, Kd), (vd, Vd))
    for layer in (0, 17, 31):
        F.check_gather(layer, gb, ([stored[layer][0]], [stored[layer][1]]))
        F.check_gather(layer, gb, ([stored[layer][0]], [stored[layer][1]]), planned=True)
    # the same gathers read through kernel-facing tables
    F.check_gather(5, gb, ([stored[5][0]], [stored[5][1]]), kernel_facing=True)
    F.check_gather(31, gb, ([stored[31][0]], [stored[31][1]]), planned=True, kernel_facing=True)
    # move 8192 never-stored tokens to other never-stored tokens
    used = np.unique(np.concatenate([synth.store_slots(sh, l) for l in range(sh.layer_num)]))
    src, dst = synth.move_slots(sh, 8192, avoid=used)
    src = np.setdiff1d(src, used)[:8000]
    dst = dst[: src.size]
    sb, db, err = F.o.move_rows(*[F.o.translate(x)[0] for x in (src, dst)])
    assert err == 0
    gt.kv_move(F.pool, F.translate(src), F.translate(dst))
    assert gt.kv_pool_last_error(F.pool) == 0
    assert torch.equal(F.rows[torch.from_numpy(db // F.R).cuda()], F.sentinel(sb)), "moved rows differ"
    F.written.append(torch.from_numpy(db // F.R).cuda())
    F.check_untouched()
    F.close()


def test_prefill_llama3_8b_full():
    """Workload 3 (32 GiB pool): 32 per-layer stores of 32768 prefill tokens
    with 2% tombstones, then on a fresh pool the all-layer store of
    [32, 32768, 8, 128] K and V, then gathers of the 16 prefill sequences."""
    sh = synth.SHAPES[3]
    slots, pages = synth.prefill_slots(sh)
    F = Full(sh)
    for layer in range(sh.layer_num):
        K, V = _vals(sh, slots.size, layer)
        F.check_store(layer, slots, K, V)
    F.check_untouched()
    F.close()
    F = Full(sh)
    Ka, Va = synth.kv_pair_all(sh, slots.size)
    ids = F.translate(slots)
    Kd = torch.from_numpy(Ka.view(np.uint8)).cuda().view(sh.layer_num, slots.size, F.R)
    Vd = torch.from_numpy(Va.view(np.uint8)).cuda().view(sh.layer_num, slots.size, F.R)
    gt.kv_store_all_layers(F.pool, ids, Kd, Vd)
    assert gt.kv_pool_last_error(F.pool) == 0
    gb = synth.gather_batch(sh)
    for layer in range(sh.layer_num):
        kd, vd, err = F.o.store_rows(layer, slots)
        assert err == 0
        F._check_rows(slots, kd, vd, Kd[layer], Vd[layer])
        if layer in (0, 31):
            live = slots >= 0
            F.check_gather(layer, gb, ([(kd[live], Kd[layer][torch.from_numpy(live).cuda()])],
                                       [(vd[live], Vd[layer][torch.from_numpy(live).cuda()])]))
    F.check_untouched()
    F.close()


def test_swa_fp8_full():
    """Workload 4 (12 GiB fp8 pool): for each of the 24 layers, store one
    token per sequence at position c-1 and gather the 128-token window
    [c-128, c) of all 512 sequences (every third layer through a
    kernel-facing table); then the 8192-token move."""
    sh = synth.SHAPES[4]
    F = Full(sh)
    slots, gb = synth.swa_batch(sh)
    ids = F.translate(slots)
    for layer in range(sh.layer_num):
        K, V = _vals(sh, slots.size, layer)
        kd, vd, Kd, Vd = F.check_store(layer, slots, K, V, ids)
        F.check_gather(layer, gb, ([(kd, Kd)], [(vd, Vd)]), planned=layer % 2 == 1, kernel_facing=layer % 3 == 2)
    used = np.unique(gb.block_table.astype(np.int64)[:, :, None] * sh.page_size + np.arange(sh.page_size))
    src, dst = synth.move_slots(sh, 8192, avoid=used)
    src = np.setdiff1d(src, used)[:8000]
    dst = dst[: src.size]
    sb, db, err = F.o.move_rows(*[F.o.translate(x)[0] for x in (src, dst)])
    assert err == 0
    gt.kv_move(F.pool, F.translate(src), F.translate(dst))
    assert gt.kv_pool_last_error(F.pool) == 0
    assert torch.equal(F.rows[torch.from_numpy(db // F.R).cuda()], F.sentinel(sb))
    F.written.append(torch.from_numpy(db // F.R).cuda())
    F.check_untouched()
    F.close()


def test_id_bound_stress_full():
    """Workload 5 (119.2 GiB fp8 pool, 1 999 994 880 kernel rows, just under
    2^31): 1M-token stores into all 80 layers (slots include every slot of
    the last 4 pages), 1M-row gathers of layers 0 and 79, the id of the last
    slot, and the id-bound rejection one page further."""
    sh = synth.SHAPES[5]
    d_bad = gt.make_desc(sh.layer_num, sh.head_num, sh.head_dim, sh.itemsize, sh.page_size, 52429)
    with pytest.raises(gt.KVError) as e:
        gt.kv_pool_create(d_bad)  # rejected on the host, nothing allocated
    assert e.value.name == "KV_ERR_ID_BOUND"
    F = Full(sh)
    assert F.sizes["n_rows"] == 1_999_994_880
    last = np.array([sh.num_pages * sh.page_size - 1], np.int64)
    assert int(F.translate(last).item()) == 1_999_954_175
    stored = {}
    for layer in range(sh.layer_num):
        slots = synth.store_slots(sh, layer)
        assert slots.max() == sh.num_pages * sh.page_size - 1
        K, V = _vals(sh, slots.size, layer)
        kd, vd, Kd, Vd = F.check_store(layer, slots, K, V)
        if layer in (0, 79):
            stored[layer] = ((kd, Kd), (vd, Vd))
    gb = synth.gather_batch(sh)
    assert (gb.block_table == sh.num_pages - 1).any()
    for layer in (0, 79):
        F.check_gather(layer, gb, ([stored[layer][0]], [stored[layer][1]]), planned=layer == 79)
    F.check_untouched()
    F.close()


@pytest.mark.parametrize("kernel_facing", [False, True], ids=["physical_tables", "kernel_facing_tables"])
def test_bench_step_full(kernel_facing):
    """The step bench.py times, on its own inputs and in its own launch
    configuration (bench.make_step on the full 8 GiB decode pool), run twice
    as its warm-up does; also in its kernel-facing form (virtual tables and
    a page map, the table built every step, plan and gathers through it).
    Then the oracle's address mode checks every row the step wrote or read:
    the 512 translated ids, the 256-token chunk and the 256 decode tokens in
    all 32 layers, every row of the last layer's planned gather (256 x 4096
    tokens; it reads rows the stores and the previous step's move wrote), the
    64 row-blocks of the 8192 moved tokens, and that no other row of the pool
    changed."""
    import bench

    sh = bench.SHAPE
    F = Full(sh)
    inp = bench.make_inputs(0)
    st = bench.make_step(gt, F.pool, inp, torch.device("cuda", torch.cuda.current_device()),
                         torch.cuda.current_stream(), kernel_facing=kernel_facing)
    for _ in range(2):
        st.step(st.dev_in)
    torch.cuda.synchronize()
    assert gt.kv_pool_last_error(F.pool) == 0
    L, R = sh.layer_num, F.R
    if kernel_facing:
        virt, v2p = bench.virtual_tables(inp["g"], sh.num_pages)
        kf_ref, err = F.o.block_table_kf(virt, inp["g"].seq_len, v2p, out=np.zeros_like(virt))
        assert err == 0 and np.array_equal(st.kf.cpu().numpy(), kf_ref), "kernel-facing table differs"

    slots = inp["slots"]
    ids_ref, err = F.o.translate(slots)
    assert err == 0 and np.array_equal(st.ids.cpu().numpy(), ids_ref), "translated ids differ"

    dec, chunk = slots[:bench.N_DECODE], slots[bench.N_DECODE:]
    last_k, last_v = [], []
    for layer in range(L):
        for sl, kk, vv in ((chunk, inp["k_chunk"][layer], inp["v_chunk"][layer]),
                           (dec, inp["k_dec"][layer], inp["v_dec"][layer])):
            kd, vd, err = F.o.store_rows(layer, sl)
            assert err == 0
            Kd = torch.from_numpy(np.ascontiguousarray(kk)).cuda()
            Vd = torch.from_numpy(np.ascontiguousarray(vv)).cuda()
            F._check_rows(sl, kd, vd, Kd, Vd)
            if layer == L - 1:
                last_k.append((kd, Kd))
                last_v.append((vd, Vd))

    # the moved tokens' source rows were never written: they hold the sentinel
    src_ids, e1 = F.o.translate(inp["move_src"])
    dst_ids, e2 = F.o.translate(inp["move_dst"])
    assert e1 == e2 == 0
    sb, db, err = F.o.move_rows(src_ids, dst_ids)
    assert err == 0
    moved = F.sentinel(sb)
    assert torch.equal(F.rows[torch.from_numpy(db // R).cuda()], moved), "moved rows differ"
    F.written.append(torch.from_numpy(db // R).cuda())

    # the gather buffers hold the last layer's rows; the second step's gather
    # ran after the first step's move
    g = inp["g"]
    if kernel_facing:
        ks, vs, err = F.o.gather_rows(L - 1, kf_ref, g.seq_len, g.cu, g.seq_start, kernel_facing=True)
    else:
        ks, vs, err = F.o.gather_rows(L - 1, g.block_table, g.seq_len, g.cu, g.seq_start)
    assert err == 0 and (ks >= 0).all() and (vs >= 0).all()
    assert torch.equal(st.out_k, F.expected_reads(ks, last_k + [(db, moved)])), "gathered K differs"
    assert torch.equal(st.out_v, F.expected_reads(vs, last_v + [(db, moved)])), "gathered V differs"
    del st
    F.check_untouched()
    F.close()
