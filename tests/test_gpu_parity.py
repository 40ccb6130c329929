"""GPU parity: every entry point through the C ABI against the CPU oracle,
byte for byte, on pools small enough to mirror whole on the host.

The shapes keep the model geometry of each workload (rows of 32 B to 4 KiB,
page sizes 3 to 256, fp8 and bf16) on fewer pages, with token counts that
span several warps' tiles and end in a ragged tail. Inputs are seeded.
"""
from __future__ import annotations

import os

import numpy as np
import pytest
import torch

import gather_translate_kv_gb300 as gt
import oracle
import synth
from gpu_util import PoolPair, as_rows, assert_bytes_equal, assert_pool_matches, dev_bits, merge, to_dev, \
    tomb_inputs

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gather_translate_kv_gb300 import build

    build.build()
    oracle.build()


S = synth.Shape
SHAPES = [
    (synth.SHAPES[1], 0),                       # R=32, ps=4 (general row path)
    (synth.SHAPES[2].scaled(40), 0),            # R=2048, ps=16, L=32
    (synth.SHAPES[3].scaled(12), 64),           # R=2048, ps=64, anchor 64
    (synth.SHAPES[4].scaled(150), 0),           # R=512 fp8, ps=32, L=24
    (synth.SHAPES[5].scaled(20), 0),            # R=64 fp8, ps=256, L=80
    (S(0, "odd-rows", 3, 3, 16, 1, 3, 40), 16),  # R=48 (general path), ps=3
    (S(0, "wide-rows", 2, 12, 128, 1, 5, 24), 0),  # R=1536 (general path), ps=5
    (S(0, "r4096", 2, 16, 128, 2, 8, 12), 32),  # R=4096
    (S(0, "r256", 4, 2, 64, 2, 4, 30), 0),      # R=256
    (S(0, "r128", 4, 1, 64, 2, 2, 40), 0),      # R=128
    (S(0, "r1024", 2, 4, 128, 2, 16, 10), 0),   # R=1024
    (S(0, "fp32-r1024", 2, 2, 128, 4, 12, 10), 0),  # R=1024, ps=12
]
IDS = [f"{s.name}-R{s.row_bytes}-ps{s.page_size}" for s, _ in SHAPES]


def _store_pages(shape: synth.Shape) -> int:
    """Stores use pages [1, hi); pages [hi, P) stay free for move destinations."""
    return max(2, (2 * shape.num_pages) // 3)


def _tokens(shape: synth.Shape, rng, n: int, tomb: int) -> np.ndarray:
    ps = shape.page_size
    hi = _store_pages(shape)
    n = min(n, (hi - 1) * ps)
    slots = synth.distinct_slots(rng, ps, hi * ps, n)
    return synth.with_tombstones(rng, slots, min(tomb, n))


def _vals(shape, rng, lead):
    dims = tuple(lead) + (shape.head_num, shape.head_dim)
    return synth.kv_values(rng, dims, shape.itemsize), synth.kv_values(rng, dims, shape.itemsize)


def test_translate_golden():
    pp = PoolPair(synth.SHAPES[1])
    maps = {
        "none": None,
        "tomb1": np.where(np.arange(64) == 1, -1, np.arange(64)).astype(np.int32),
        "p1to9": np.where(np.arange(64) == 1, 9, np.arange(64)).astype(np.int32),
    }
    for line in open(os.path.join(GOLDEN, "translate_tiny.txt")):
        line = line.split("#", 1)[0].split()
        if not line:
            continue
        slot, case, want = int(line[0]), line[1], int(line[2])
        ids = torch.empty(1, dtype=torch.int32, device="cuda")
        v2p = None if maps[case] is None else to_dev(maps[case])
        gt.kv_translate(pp.pool, to_dev(np.array([slot], np.int64)), ids, v2p)
        assert int(ids.item()) == want, (slot, case)
    assert pp.last_error() == 0


@pytest.mark.parametrize("shape,anchor", SHAPES, ids=IDS)
def test_translate_matches_oracle(shape, anchor):
    rng = np.random.default_rng(100 + shape.row_bytes + shape.page_size)
    pp = PoolPair(shape, anchor, mirror=False)
    ps, P = shape.page_size, shape.num_pages
    n = 5000
    slots = rng.integers(-3, P * ps, size=n).astype(np.int64)
    # without a page map
    ids_ref, err = pp.o.translate(slots)
    ids = torch.empty(n, dtype=torch.int32, device="cuda")
    gt.kv_translate(pp.pool, to_dev(slots), ids)
    assert np.array_equal(ids.cpu().numpy(), ids_ref)
    assert pp.last_error() == dev_bits(err) == 0
    # with a page map: a permutation with tombstoned pages
    v2p = rng.permutation(P).astype(np.int32)
    v2p[rng.choice(P, size=max(1, P // 7), replace=False)] = -1
    ids_ref, err = pp.o.translate(slots, v2p)
    gt.kv_translate(pp.pool, to_dev(slots), ids, to_dev(v2p))
    assert np.array_equal(ids.cpu().numpy(), ids_ref)
    assert pp.last_error() == dev_bits(err) == 0
    # errors: a map shorter than the slots' pages, and pages past the pool
    short = v2p[: P // 2].copy()
    short[0] = P + 3
    ids_ref, err = pp.o.translate(slots, short)
    gt.kv_translate(pp.pool, to_dev(slots), ids, to_dev(short))
    assert np.array_equal(ids.cpu().numpy(), ids_ref)
    assert err == oracle.E_V2P | oracle.E_ROW
    assert pp.last_error() == dev_bits(err)
    pp.close()


@pytest.mark.parametrize("shape,anchor", SHAPES, ids=IDS)
def test_path_matches_oracle(shape, anchor):
    """translate -> per-layer stores -> all-layer store -> gathers -> move,
    comparing the whole pool (and every output) after each step."""
    rng = np.random.default_rng(200 + shape.row_bytes * 7 + shape.page_size)
    pp = PoolPair(shape, anchor)
    o, R, L = pp.o, pp.R, shape.layer_num
    ps, P = shape.page_size, shape.num_pages
    M0 = pp.M.copy()
    tombs: dict = {}
    stored = set()

    # per-layer stores through translate (K1 -> K2)
    for layer in sorted({0, L // 2, L - 1}):
        n = 37 * 11 if shape.cfg != 1 else 100
        slots = synth.store_slots(shape, layer) if shape.cfg == 1 else _tokens(shape, rng, n, 9)
        K, V = _vals(shape, rng, (slots.size,))
        err = o.store(pp.M, layer, slots, K, V)
        ids_ref, terr = o.translate(slots)
        ids = torch.empty(slots.size, dtype=torch.int32, device="cuda")
        gt.kv_translate(pp.pool, to_dev(slots), ids)
        assert np.array_equal(ids.cpu().numpy(), ids_ref)
        gt.kv_store_layer(pp.pool, layer, ids, to_dev(K), to_dev(V))
        assert pp.last_error() == dev_bits(err | terr) == 0
        tombs = merge(tombs, tomb_inputs(slots, K, V, layer, R))
        stored.update(int(t) for t in slots if t >= 0)
        assert_pool_matches(pp, M0, tombs)

    # all-layer store
    n = 300 if shape.cfg != 1 else 100
    slots = _tokens(shape, rng, n, 4)
    Ka, Va = _vals(shape, rng, (L, slots.size))
    err = o.store_all(pp.M, slots, Ka, Va)
    ids = torch.empty(slots.size, dtype=torch.int32, device="cuda")
    gt.kv_translate(pp.pool, to_dev(slots), ids)
    gt.kv_store_all_layers(pp.pool, ids, to_dev(Ka), to_dev(Va))
    assert pp.last_error() == dev_bits(err) == 0
    for layer in range(L):
        tombs = merge(tombs, tomb_inputs(slots, Ka[layer], Va[layer], layer, R))
    stored.update(int(t) for t in slots if t >= 0)
    assert_pool_matches(pp, M0, tombs)

    # gathers: full sequences, windows starting mid-page, an empty sequence,
    # ragged lengths, pages shared across sequences (never page 0)
    if shape.cfg == 1:
        g = synth.gather_batch(shape)
        batches = [g, synth.GatherBatch(g.block_table, np.array([3], np.int32), np.array([29], np.int32))]
    else:
        S_, maxp = 9, min(P - 1, 7)
        bt = np.stack([1 + rng.permutation(P - 1)[:maxp] for _ in range(S_)]).astype(np.int32)
        ln = rng.integers(0, maxp * ps + 1, size=S_).astype(np.int32)
        ln[2] = 0
        ln[0] = maxp * ps
        st = np.minimum(rng.integers(0, 2 * ps, size=S_), ln).astype(np.int32)
        batches = [synth.GatherBatch(bt, np.zeros(S_, np.int32), ln), synth.GatherBatch(bt, st, ln)]
    for gb in batches:
        for layer in sorted({0, L - 1}):
            rows = gb.total + 5  # a few spare rows must stay untouched
            ok = np.full((rows, R), 0x5A, np.uint8)
            ov = np.full((rows, R), 0xA5, np.uint8)
            ok, ov, err = o.gather(pp.M, layer, gb.block_table, gb.seq_len, gb.cu, gb.seq_start, rows, ok, ov)
            dk = torch.full((rows, R), 0x5A, dtype=torch.uint8, device="cuda")
            dv = torch.full((rows, R), 0xA5, dtype=torch.uint8, device="cuda")
            gt.kv_gather_layer(pp.pool, layer, to_dev(gb.block_table), to_dev(gb.seq_len), to_dev(gb.cu), dk, dv,
                               to_dev(gb.seq_start))
            assert pp.last_error() == dev_bits(err) == 0
            assert_bytes_equal(dk.cpu().numpy(), ok, f"gather K layer {layer}", R)
            assert_bytes_equal(dv.cpu().numpy(), ov, f"gather V layer {layer}", R)

    # move: stored tokens -> never-stored tokens (disjoint, distinct)
    free = np.setdiff1d(np.arange(ps, P * ps, dtype=np.int64), np.array(sorted(stored), np.int64))
    m = min(20 if shape.cfg == 1 else 150, len(stored), free.size)
    assert m >= 10, "test setup leaves too few free slots"
    src_slots = rng.choice(sorted(stored), size=m, replace=False).astype(np.int64)
    dst_slots = rng.choice(free, size=m, replace=False).astype(np.int64)
    src_ids, _ = o.translate(src_slots)
    dst_ids, _ = o.translate(dst_slots)
    err = o.move(pp.M, src_ids, dst_ids)
    gt.kv_move(pp.pool, to_dev(src_ids), to_dev(dst_ids))
    assert pp.last_error() == dev_bits(err) == 0
    assert_pool_matches(pp, M0, tombs)
    pp.close()


def test_error_paths_match_oracle():
    shape = S(0, "err", 2, 1, 64, 2, 4, 16)  # R=128
    rng = np.random.default_rng(7)
    pp = PoolPair(shape)
    o, R, ps, P = pp.o, pp.R, shape.page_size, shape.num_pages
    M0 = pp.M.copy()
    n_rows = pp.sizes["n_rows"]
    # store: ids outside [0, n_rows) are skipped and flagged
    slots = synth.distinct_slots(rng, ps, P * ps, 40)
    K, V = _vals(shape, rng, (40,))
    ids, _ = o.translate(slots)
    bad = ids.copy()
    bad[[3, 17, 39]] = [n_rows, -5, n_rows + 1000]
    keep = np.ones(40, bool)
    keep[[3, 17, 39]] = False
    o.store(pp.M, 1, slots[keep], K[keep], V[keep])
    gt.kv_store_layer(pp.pool, 1, to_dev(bad), to_dev(K), to_dev(V))
    assert pp.last_error() == gt.KV_DEV_ERR_ROW
    assert_pool_matches(pp, M0, {})
    # store: in-range ids that translate cannot produce (offset >= ps inside
    # the page envelope) are skipped too, per-layer and all-layer
    for form_bad in ([5, 21], [0, 30, 38]):
        slots2 = synth.distinct_slots(rng, ps, P * ps, 40)
        K2, V2 = _vals(shape, rng, (2, 40))
        ids2, _ = o.translate(slots2)
        bad2 = ids2.copy()
        bad2[form_bad] += ps  # same page envelope, offset in [ps, 2 ps): another row-block
        keep2 = np.ones(40, bool)
        keep2[form_bad] = False
        if len(form_bad) == 2:
            o.store(pp.M, 0, slots2[keep2], K2[0][keep2], V2[0][keep2])
            gt.kv_store_layer(pp.pool, 0, to_dev(bad2), to_dev(K2[0]), to_dev(V2[0]))
        else:
            o.store_all(pp.M, slots2[keep2], K2[:, keep2], V2[:, keep2])
            gt.kv_store_all_layers(pp.pool, to_dev(bad2), to_dev(K2), to_dev(V2))
        assert pp.last_error() == gt.KV_DEV_ERR_FORM
        assert_pool_matches(pp, M0, {})
    # move: a non-translate-form id and an out-of-range id skip their pairs
    src, _ = o.translate(slots[:6])
    free = np.setdiff1d(np.arange(ps, P * ps), slots)[:6]
    dst, _ = o.translate(free)
    src_b = src.copy()
    dst_b = dst.copy()
    src_b[1] = src[1] + ps  # offset >= ps inside its page envelope
    dst_b[4] = n_rows + 7
    err = o.move(pp.M, src_b, dst_b)
    assert err == oracle.E_FORM | oracle.E_ROW
    gt.kv_move(pp.pool, to_dev(src_b), to_dev(dst_b))
    assert pp.last_error() == dev_bits(err)
    assert_pool_matches(pp, M0, {})
    # gather: a page past the pool, a sequence whose cu span is too short, and
    # an output too small for cu[S]
    bt = np.array([[1, 2, P + 4, 3], [4, 5, 6, 7], [8, 9, 10, 11]], np.int32)
    ln = np.array([16, 16, 10], np.int32)
    st = np.array([0, 2, 1], np.int32)
    cu = np.array([0, 16, 27, 40], np.int64)  # sequence 1 needs 14 rows, gets 11
    for rows in (40, 33):
        ok = np.full((rows, R), 1, np.uint8)
        ov = np.full((rows, R), 2, np.uint8)
        ok, ov, err = o.gather(pp.M, 0, bt, ln, cu, st, rows, ok, ov)
        dk = torch.full((rows, R), 1, dtype=torch.uint8, device="cuda")
        dv = torch.full((rows, R), 2, dtype=torch.uint8, device="cuda")
        gt.kv_gather_layer(pp.pool, 0, to_dev(bt), to_dev(ln), to_dev(cu), dk, dv, to_dev(st))
        assert err == oracle.E_ROW | oracle.E_TABLE
        assert pp.last_error() == dev_bits(err)
        # rows the oracle writes and the kernel writes agree wherever the
        # metadata is consistent: sequence 0 and the rows of sequence 2 that
        # sequence 1's overlong span does not also cover (those race)
        for r0, r1 in ((0, 16), (30, min(rows, 36))):
            assert_bytes_equal(dk.cpu().numpy()[r0:r1], ok[r0:r1], "gather K", R)
            assert_bytes_equal(dv.cpu().numpy()[r0:r1], ov[r0:r1], "gather V", R)
    # host-side argument errors
    with pytest.raises(gt.KVError) as e:
        gt.kv_store_layer(pp.pool, 2, to_dev(ids), to_dev(K), to_dev(V))
    assert e.value.name == "KV_ERR_INVALID"
    with pytest.raises(gt.KVError) as e:
        kk = torch.empty(40 * R + 8, dtype=torch.uint8, device="cuda")[8:]
        gt.kv_store_layer(pp.pool, 0, to_dev(ids), kk, to_dev(V))
    assert e.value.name == "KV_ERR_ALIGN"
    pp.close()


def test_create_rejects_a_buffer_that_is_not_device_memory():
    """kv_pool_create checks where a borrowed buffer lives before any kernel
    could touch it: host memory (pageable or pinned) is refused, device
    memory of the current device is taken."""
    import ctypes

    desc = gt.make_desc(2, 2, 8, 2, 4, 64)
    total, pad = gt.kv_pool_required_bytes(desc)
    nbytes = total + pad
    pageable = np.zeros(nbytes + 16, np.uint8)
    base = pageable.ctypes.data
    pinned = torch.zeros(nbytes, dtype=torch.uint8).pin_memory()
    for ptr in (base + (-base) % 16, pinned.data_ptr()):
        h = ctypes.c_void_p()
        rc = gt.lib().kv_pool_create(ctypes.byref(desc), ctypes.c_void_p(ptr), nbytes, ctypes.byref(h))
        assert gt.STATUS[rc] == "KV_ERR_INVALID" and not h.value
    raw = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    pool = gt.kv_pool_create(desc, raw)
    assert pool.info["raw_dev"] == raw.data_ptr() and pool.info["owns_raw"] == 0
    # the refused calls left no CUDA error behind for the next launch to report
    ids = torch.zeros(4, dtype=torch.int32, device="cuda")
    gt.kv_translate(pool, torch.arange(4, 8, dtype=torch.int64, device="cuda"), ids)
    assert gt.kv_pool_last_error(pool) == 0 and ids.tolist() == [16, 17, 18, 19]
    gt.kv_pool_destroy(pool)


def test_empty_calls_are_no_ops():
    """Zero tokens, zero sequences, sequences without table entries and
    zero-length sequences: every call returns KV_OK, raises no device error
    bit, and changes no byte of the pool, of a gather output or of a block
    table."""
    shape = S(0, "empty", 2, 2, 64, 2, 4, 16)  # R=256
    pp = PoolPair(shape)
    M0 = pp.M.copy()
    R, L = pp.R, shape.layer_num
    i64 = torch.empty(0, dtype=torch.int64, device="cuda")
    i32 = torch.empty(0, dtype=torch.int32, device="cuda")
    rows0 = torch.empty((0, R), dtype=torch.uint8, device="cuda")
    all0 = torch.empty((L, 0, R), dtype=torch.uint8, device="cuda")
    gt.kv_translate(pp.pool, i64, i32)
    gt.kv_translate_mapped(pp.pool, i64, i32, torch.zeros(8, dtype=torch.int64, device="cuda"))
    gt.kv_store_layer(pp.pool, 1, i32, rows0, rows0)
    gt.kv_store_all_layers(pp.pool, i32, all0, all0)
    gt.kv_store_layer_slots(pp.pool, 0, i64, rows0, rows0)
    gt.kv_store_all_layers_slots(pp.pool, i64, all0, all0)
    gt.kv_move(pp.pool, i32, i32)
    # no sequences at all
    bt0 = torch.empty((0, 4), dtype=torch.int32, device="cuda")
    cu0 = torch.zeros(1, dtype=torch.int64, device="cuda")
    gt.kv_gather_layer(pp.pool, 0, bt0, i32, cu0, rows0, rows0)
    plan0 = gt.kv_gather_plan(pp.pool, bt0, i32)
    gt.kv_gather_layer_planned(pp.pool, 0, plan0, bt0, i32, cu0, rows0, rows0)
    assert plan0[0].item() == 0
    # three sequences with no table entries, and three zero-length sequences
    # over a real table: nothing is read, no output row is written
    zl = torch.zeros(3, dtype=torch.int32, device="cuda")
    cu = torch.zeros(4, dtype=torch.int64, device="cuda")
    gt.kv_gather_layer(pp.pool, 1, torch.empty((3, 0), dtype=torch.int32, device="cuda"), zl, cu, rows0, rows0)
    bt = torch.tensor([[1, 2], [3, 4], [5, 6]], dtype=torch.int32, device="cuda")
    ok = torch.full((5, R), 0x33, dtype=torch.uint8, device="cuda")
    ov = torch.full((5, R), 0x44, dtype=torch.uint8, device="cuda")
    gt.kv_gather_layer(pp.pool, 1, bt, zl, cu, ok, ov)
    plan = gt.kv_gather_plan(pp.pool, bt, zl)
    gt.kv_gather_layer_planned(pp.pool, 1, plan, bt, zl, cu, ok, ov)
    assert plan[0].item() == 0
    assert bool((ok == 0x33).all()) and bool((ov == 0x44).all())
    # a prefix-only table translation of zero-length sequences touches no entry
    v2p = torch.arange(16, dtype=torch.int32, device="cuda")
    out = gt.kv_translate_block_table(pp.pool, bt, zl, v2p, out_bt=torch.full_like(bt, -9))
    assert bool((out == -9).all())
    assert pp.last_error() == 0
    assert_pool_matches(pp, M0, {})
    pp.close()


def test_gather_tombstoned_table_entry_reads_sink():
    shape = S(0, "sink", 2, 2, 64, 2, 8, 10)
    pp = PoolPair(shape)
    bt = np.array([[3, -1, 5]], np.int32)
    g = synth.GatherBatch(bt, np.array([4], np.int32), np.array([22], np.int32))
    ok, ov, err = pp.o.gather(pp.M, 1, bt, g.seq_len, g.cu, g.seq_start)
    dk = torch.zeros((g.total, pp.R), dtype=torch.uint8, device="cuda")
    dv = torch.zeros_like(dk)
    gt.kv_gather_layer(pp.pool, 1, to_dev(bt), to_dev(g.seq_len), to_dev(g.cu), dk, dv, to_dev(g.seq_start))
    assert err == 0 and pp.last_error() == 0
    assert_bytes_equal(dk.cpu().numpy(), ok, "K", pp.R)
    assert_bytes_equal(dv.cpu().numpy(), ov, "V", pp.R)
    sink_k = pp.M[pp.o.slot_row_byte(0, 2): pp.o.slot_row_byte(0, 2) + pp.R]
    assert np.array_equal(ok[8 - 4], sink_k)  # token 8 sits on the tombstoned page


def test_calls_capture_in_a_cuda_graph():
    """translate -> store -> gather, and plan -> planned gather, captured once,
    replayed on new inputs. The pages hold 64 KiB of K and V per layer and the
    table has more entries than the pool has pages, so both gathers run their
    fan-out form (bulk copies through 64 KiB of shared memory) inside the graph."""
    shape = synth.SHAPES[2].scaled(24)
    pp = PoolPair(shape)
    o, R, ps, P = pp.o, pp.R, shape.page_size, shape.num_pages
    M0 = pp.M.copy()
    n = 64
    slots_d = torch.zeros(n, dtype=torch.int64, device="cuda")
    ids_d = torch.zeros(n, dtype=torch.int32, device="cuda")
    k_d = torch.zeros((n, R), dtype=torch.uint8, device="cuda")
    v_d = torch.zeros_like(k_d)
    bt = np.stack([1 + np.arange(8) + 2 * s for s in range(4)]).astype(np.int32)  # 14 pages, 32 entries: page-major
    assert bt.size >= P and 2 * ps * R == 65536
    g = synth.GatherBatch(bt, np.zeros(4, np.int32), np.full(4, 8 * ps, np.int32))
    bt_d, ln_d, cu_d = to_dev(bt), to_dev(g.seq_len), to_dev(g.cu)
    ok_d = torch.zeros((g.total, R), dtype=torch.uint8, device="cuda")
    ov_d = torch.zeros_like(ok_d)
    pk_d = torch.zeros_like(ok_d)
    pv_d = torch.zeros_like(ok_d)
    plan_d = torch.zeros(gt.kv_gather_plan_bytes(pp.pool, *bt.shape) // 4, dtype=torch.int32, device="cuda")

    def step():
        gt.kv_translate(pp.pool, slots_d, ids_d)
        gt.kv_store_layer(pp.pool, 3, ids_d, k_d, v_d)
        gt.kv_gather_layer(pp.pool, 3, bt_d, ln_d, cu_d, ok_d, ov_d)
        gt.kv_gather_plan(pp.pool, bt_d, ln_d, plan=plan_d)
        gt.kv_gather_layer_planned(pp.pool, 3, plan_d, bt_d, ln_d, cu_d, pk_d, pv_d)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # warm-up outside capture
        step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    # restore the pool and the mirror to the sentinel before the replays
    synth.fill_sentinel_torch(pp.raw, pp.fill_seed)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    rng = np.random.default_rng(9)
    for rep in range(2):
        slots = synth.distinct_slots(rng, ps, 17 * ps, n)  # pages the gather reads
        K, V = _vals(shape, rng, (n,))
        slots_d.copy_(to_dev(slots))
        k_d.copy_(to_dev(as_rows(K, R)))
        v_d.copy_(to_dev(as_rows(V, R)))
        o.store(pp.M, 3, slots, K, V)
        graph.replay()
        torch.cuda.synchronize()
        rk, rv, _ = o.gather(pp.M, 3, bt, g.seq_len, g.cu)
        assert_bytes_equal(ok_d.cpu().numpy(), rk, "graph gather K", R)
        assert_bytes_equal(ov_d.cpu().numpy(), rv, "graph gather V", R)
        assert_bytes_equal(pk_d.cpu().numpy(), rk, "graph planned gather K", R)
        assert_bytes_equal(pv_d.cpu().numpy(), rv, "graph planned gather V", R)
        assert_pool_matches(pp, M0, {})
    assert pp.last_error() == 0
    pp.close()


def test_remaining_calls_capture_in_a_cuda_graph():
    """The calls the graph test above leaves out, captured once with a page
    map and replayed twice on new inputs: fused translate + all-layer store,
    fused translate + per-layer store, translate of move ids, the move (of
    tokens the same replay stored), the prefix-only kernel-facing block table
    and the full -> SWA token map."""
    shape = S(0, "graph2", 4, 2, 64, 2, 8, 40)  # R=256, L=4, ps=8
    pp = PoolPair(shape)
    o, R, L, ps, P = pp.o, pp.R, shape.layer_num, shape.page_size, shape.num_pages
    M0 = pp.M.copy()
    rng = np.random.default_rng(77)
    v2p = np.zeros(P, np.int32)
    v2p[1:] = 1 + rng.permutation(P - 1)  # a bijection of pages 1..P-1; page 0 stays the sink
    na, nb, nm, S_, mp, nf, tlen = 48, 40, 16, 3, 4, 20, 300
    z = lambda shp, dt: torch.zeros(shp, dtype=dt, device="cuda")  # noqa: E731
    sa_d, sb_d = z(na, torch.int64), z(nb, torch.int64)
    ka_d, va_d = z((L, na, R), torch.uint8), z((L, na, R), torch.uint8)
    kb_d, vb_d = z((nb, R), torch.uint8), z((nb, R), torch.uint8)
    ms_d, md_d = z(nm, torch.int64), z(nm, torch.int64)
    src_d, dst_d = z(nm, torch.int32), z(nm, torch.int32)
    vbt_d, ln_d, obt_d = z((S_, mp), torch.int32), z(S_, torch.int32), z((S_, mp), torch.int32)
    fs_d, mid_d, tmap_d = z(nf, torch.int64), z(nf, torch.int32), z(tlen, torch.int64)
    v2p_d = to_dev(v2p)

    def step():
        gt.kv_store_all_layers_slots(pp.pool, sa_d, ka_d, va_d, v2p=v2p_d)
        gt.kv_store_layer_slots(pp.pool, 2, sb_d, kb_d, vb_d, v2p=v2p_d)
        gt.kv_translate(pp.pool, ms_d, src_d, v2p_d)
        gt.kv_translate(pp.pool, md_d, dst_d, v2p_d)
        gt.kv_move(pp.pool, src_d, dst_d)
        gt.kv_translate_block_table(pp.pool, vbt_d, ln_d, v2p_d, out_bt=obt_d)
        gt.kv_translate_mapped(pp.pool, fs_d, mid_d, tmap_d, v2p=v2p_d)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # warm-up outside capture (all inputs zero: page-0 sink rows only)
        step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    synth.fill_sentinel_torch(pp.raw, pp.fill_seed)
    assert pp.last_error() == 0
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for rep in range(2):
        sa = synth.distinct_slots(rng, ps, 13 * ps, na)           # virtual pages 1..12
        sb = synth.distinct_slots(rng, 13 * ps, 20 * ps, nb)      # virtual pages 13..19
        ms = rng.choice(sa, size=nm, replace=False)              # move tokens stored this replay
        md = synth.distinct_slots(rng, 20 * ps, 30 * ps, nm)      # to virtual pages 20..29
        Ka, Va = _vals(shape, rng, (L, na))
        Kb, Vb = _vals(shape, rng, (nb,))
        vbt = rng.integers(-1, P, size=(S_, mp)).astype(np.int32)
        ln = rng.integers(0, mp * ps + 1, size=S_).astype(np.int32)
        tmap = rng.integers(-1, P * ps, size=tlen).astype(np.int64)
        fs = rng.integers(-2, tlen, size=nf).astype(np.int64)
        for d, h in ((sa_d, sa), (sb_d, sb), (ms_d, ms), (md_d, md), (vbt_d, vbt), (ln_d, ln), (tmap_d, tmap),
                     (fs_d, fs)):
            d.copy_(to_dev(h))
        ka_d.copy_(to_dev(as_rows(Ka, R).reshape(L, na, R)))
        va_d.copy_(to_dev(as_rows(Va, R).reshape(L, na, R)))
        kb_d.copy_(to_dev(as_rows(Kb, R)))
        vb_d.copy_(to_dev(as_rows(Vb, R)))
        obt_d.fill_(-7)
        assert o.store_all(pp.M, sa, Ka, Va, v2p) == 0
        assert o.store(pp.M, 2, sb, Kb, Vb, v2p) == 0
        src, e1 = o.translate(ms, v2p)
        dst, e2 = o.translate(md, v2p)
        assert e1 == e2 == 0 and o.move(pp.M, src, dst) == 0
        bt_ref, e3 = o.block_table_kf(vbt, ln, v2p)
        mid_ref, e4 = o.translate_mapped(fs, tmap, v2p)
        assert e3 == e4 == 0
        graph.replay()
        torch.cuda.synchronize()
        assert pp.last_error() == 0
        assert np.array_equal(src_d.cpu().numpy(), src) and np.array_equal(dst_d.cpu().numpy(), dst)
        assert np.array_equal(obt_d.cpu().numpy(), bt_ref), "graph block table"
        assert np.array_equal(mid_d.cpu().numpy(), mid_ref), "graph token-mapped ids"
        assert_pool_matches(pp, M0, {})
    pp.close()


def test_two_streams_share_one_pool():
    """Two streams store and gather different layers of one pool at the same
    time; one of them also stores a batch with an out-of-range id. Both
    streams' results match the oracle and the error bit reaches the pool's
    shared error word."""
    shape = S(0, "streams", 4, 2, 64, 2, 8, 40)  # R=256, L=4, ps=8
    pp = PoolPair(shape)
    o, R, ps, P = pp.o, pp.R, shape.page_size, shape.num_pages
    M0 = pp.M.copy()
    rng = np.random.default_rng(78)
    work = []
    for layer, lo, hi in ((1, 1, 20), (3, 20, 40)):
        slots = synth.distinct_slots(rng, lo * ps, hi * ps, 96)
        K, V = _vals(shape, rng, (96,))
        ids, _ = o.translate(slots)
        bt = rng.integers(1, P, size=(6, 5)).astype(np.int32)
        g = synth.GatherBatch(bt, np.zeros(6, np.int32), rng.integers(1, 5 * ps + 1, size=6).astype(np.int32))
        work.append((layer, slots, K, V, ids, g))
    bad = work[1][4].copy()
    bad[7] = pp.sizes["n_rows"] + 3
    dev = [dict(ids=to_dev(ids), K=to_dev(as_rows(K, R)), V=to_dev(as_rows(V, R)), bt=to_dev(g.block_table),
                ln=to_dev(g.seq_len), cu=to_dev(g.cu), ok=torch.zeros((g.total, R), dtype=torch.uint8, device="cuda"),
                ov=torch.zeros((g.total, R), dtype=torch.uint8, device="cuda"))
           for (_, _, K, V, ids, g) in work]
    bad_d = to_dev(bad)
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for st in streams:
        st.wait_stream(torch.cuda.current_stream())
    for (layer, *_), d, st in zip(work, dev, streams):
        gt.kv_store_layer(pp.pool, layer, d["ids"], d["K"], d["V"], stream=st)
        gt.kv_gather_layer(pp.pool, layer, d["bt"], d["ln"], d["cu"], d["ok"], d["ov"], stream=st)
    # stream 2 then stores layer 0 with one id past the pool: that row is skipped
    gt.kv_store_layer(pp.pool, 0, bad_d, dev[1]["K"], dev[1]["V"], stream=streams[1])
    torch.cuda.synchronize()
    assert pp.last_error() == gt.KV_DEV_ERR_ROW
    for (layer, slots, K, V, ids, g), d in zip(work, dev):
        assert o.store(pp.M, layer, slots, K, V) == 0
        rk, rv, err = o.gather(pp.M, layer, g.block_table, g.seq_len, g.cu)
        assert err == 0
        assert_bytes_equal(d["ok"].cpu().numpy(), rk, f"stream gather K, layer {layer}", R)
        assert_bytes_equal(d["ov"].cpu().numpy(), rv, f"stream gather V, layer {layer}", R)
    keep = np.ones(96, bool)
    keep[7] = False
    _, slots1, K1, V1, _, _ = work[1]
    assert o.store(pp.M, 0, slots1[keep], K1[keep], V1[keep]) == 0
    assert_pool_matches(pp, M0, {})
    pp.close()


@pytest.mark.parametrize("shape,anchor", SHAPES[:6], ids=IDS[:6])
def test_fused_translate_store_matches_oracle(shape, anchor):
    """kv_store_layer_slots / kv_store_all_layers_slots (translate fused into
    the store) against the oracle's store, which takes slots natively; with a
    page map that tombstones some pages, and with a map too short (errors)."""
    rng = np.random.default_rng(300 + shape.row_bytes + shape.page_size)
    pp = PoolPair(shape, anchor)
    o, R, L = pp.o, pp.R, shape.layer_num
    ps, P = shape.page_size, shape.num_pages
    M0 = pp.M.copy()
    hi = _store_pages(shape)
    v2p = np.arange(P, dtype=np.int32)
    v2p[1:hi] = (1 + rng.permutation(hi - 1)).astype(np.int32)  # virtual pages 1..hi-1 shuffled
    v2p[rng.choice(np.arange(1, hi), size=max(1, hi // 6), replace=False)] = -1
    tombs: dict = {}
    for layer in sorted({0, L - 1}):
        slots = _tokens(shape, rng, 257, 6)
        K, V = _vals(shape, rng, (slots.size,))
        err = o.store(pp.M, layer, slots, K, V, v2p)
        gt.kv_store_layer_slots(pp.pool, layer, to_dev(slots), to_dev(K), to_dev(V), to_dev(v2p))
        assert pp.last_error() == dev_bits(err) == 0
        # tombstoned slots and slots on tombstoned pages both land on the sink
        sunk = (slots < 0) | (v2p[np.maximum(slots, 0) // ps] < 0)
        tombs = merge(tombs, tomb_inputs(np.where(sunk, -1, slots), K, V, layer, R))
        assert_pool_matches(pp, M0, tombs)
    slots = _tokens(shape, rng, 190, 3)
    Ka, Va = _vals(shape, rng, (L, slots.size))
    err = o.store_all(pp.M, slots, Ka, Va, v2p)
    gt.kv_store_all_layers_slots(pp.pool, to_dev(slots), to_dev(Ka), to_dev(Va), to_dev(v2p))
    assert pp.last_error() == dev_bits(err) == 0
    sunk = (slots < 0) | (v2p[np.maximum(slots, 0) // ps] < 0)
    for layer in range(L):
        tombs = merge(tombs, tomb_inputs(np.where(sunk, -1, slots), Ka[layer], Va[layer], layer, R))
    assert_pool_matches(pp, M0, tombs)
    # a page map shorter than the pages used: those tokens go to the sink with V2P set
    short = v2p[: max(2, hi // 2)].copy()
    slots = _tokens(shape, rng, 100, 0)
    K, V = _vals(shape, rng, (slots.size,))
    err = o.store(pp.M, 0, slots, K, V, short)
    gt.kv_store_layer_slots(pp.pool, 0, to_dev(slots), to_dev(K), to_dev(V), to_dev(short))
    assert err & oracle.E_V2P and pp.last_error() == dev_bits(err)
    vp_ = np.maximum(slots, 0) // ps
    sunk = (slots < 0) | (vp_ >= short.size) | (short[np.minimum(vp_, short.size - 1)] < 0)
    tombs = merge(tombs, tomb_inputs(np.where(sunk, -1, slots), K, V, 0, R))
    assert_pool_matches(pp, M0, tombs)
    pp.close()


@pytest.mark.parametrize("shape", [synth.SHAPES[1], synth.SHAPES[2].scaled(300), synth.SHAPES[5].scaled(64),
                                   S(0, "odd", 3, 1, 16, 1, 3, 90)], ids=lambda s: s.name)
def test_block_table_matches_oracle(shape):
    """kv_translate_block_table against the oracle (entries, untouched tails,
    error bits), in place and out of place, and entry*ps + o equal to
    kv_translate's id of the same virtual slot."""
    rng = np.random.default_rng(400 + shape.page_size)
    pp = PoolPair(shape, mirror=False)
    ps, P = shape.page_size, shape.num_pages
    S_, maxp = 37, 9
    V = P + 5  # virtual page space, a few past the physical pages
    v2p = rng.permutation(V).astype(np.int32) % P
    v2p[rng.choice(V, size=V // 8, replace=False)] = -1
    virt = rng.integers(-1, V, size=(S_, maxp)).astype(np.int32)
    ln = rng.integers(0, maxp * ps + 1, size=S_).astype(np.int32)
    want, err = pp.o.block_table_kf(virt, ln, v2p, out=np.full(virt.shape, -7, np.int32))
    assert err == 0
    out = torch.full(virt.shape, -7, dtype=torch.int32, device="cuda")
    gt.kv_translate_block_table(pp.pool, to_dev(virt), to_dev(ln), to_dev(v2p), out)
    assert pp.last_error() == 0
    assert np.array_equal(out.cpu().numpy(), want)
    # in place; a short map and an overlong sequence raise their bits
    short = v2p[: V // 2].copy()
    ln2 = ln.copy()
    ln2[3] = maxp * ps + 2
    pre = np.where(np.arange(maxp)[None, :] < -(-ln2[:, None] // ps), virt, -7).astype(np.int32)
    want2, err2 = pp.o.block_table_kf(virt, ln2, short, out=pre.copy())
    vt = to_dev(pre.copy())
    vt.copy_(to_dev(virt))
    gt.kv_translate_block_table(pp.pool, vt, to_dev(ln2), to_dev(short))  # out_bt = virt_bt
    assert pp.last_error() == dev_bits(err2) and err2 & oracle.E_TABLE
    got2 = vt.cpu().numpy()
    mask = np.arange(maxp)[None, :] < np.minimum(-(-ln2[:, None] // ps), maxp)
    assert np.array_equal(got2[mask], want2[mask]) and np.array_equal(got2[~mask], virt[~mask])
    # consistency with kv_translate on the same virtual slots
    kk = np.nonzero(mask & (want > 0))
    offs = rng.integers(0, ps, size=kk[0].size)
    slots = virt[kk].astype(np.int64) * ps + offs
    ids = torch.empty(slots.size, dtype=torch.int32, device="cuda")
    gt.kv_translate(pp.pool, to_dev(slots), ids, to_dev(v2p))
    assert np.array_equal(ids.cpu().numpy(), want[kk].astype(np.int64) * ps + offs)
    pp.close()


MLA_SHAPES = [
    (S(0, "mla-deepseek-like", 6, 1, 576, 2, 64, 10), 0),  # latent 512+64 bf16: R=1152 (general row path)
    (S(0, "mla-r512", 5, 1, 256, 2, 16, 30), 32),          # R=512
    (S(0, "mla-fp8-r64", 9, 1, 64, 1, 32, 24), 0),          # R=64
]


@pytest.mark.parametrize("shape,anchor", MLA_SHAPES, ids=[s.name for s, _ in MLA_SHAPES])
def test_mla_path_matches_oracle(shape, anchor):
    """MLA pools (one latent row per layer, L blocks per page, no V): translate,
    per-layer and all-layer stores (id and fused forms), gathers and a move,
    each against the oracle on the whole pool."""
    rng = np.random.default_rng(500 + shape.row_bytes)
    pp = PoolPair(shape, anchor, latent=True)
    o, R, L = pp.o, pp.R, shape.layer_num
    ps, P = shape.page_size, shape.num_pages
    assert pp.pool.info["blocks_per_page"] == L and pp.pool.info["latent_only"] == 1
    M0 = pp.M.copy()
    tombs: dict = {}
    stored = set()
    for layer in sorted({0, L // 2, L - 1}):
        slots = _tokens(shape, rng, 150, 5)
        K = synth.kv_values(rng, (slots.size, shape.head_num, shape.head_dim), shape.itemsize)
        err = o.store(pp.M, layer, slots, K, None)
        ids_ref, _ = o.translate(slots)
        ids = torch.empty(slots.size, dtype=torch.int32, device="cuda")
        gt.kv_translate(pp.pool, to_dev(slots), ids)
        assert np.array_equal(ids.cpu().numpy(), ids_ref)
        if layer == 0:
            gt.kv_store_layer_slots(pp.pool, layer, to_dev(slots), to_dev(K), None)
        else:
            gt.kv_store_layer(pp.pool, layer, ids, to_dev(K), None)
        assert pp.last_error() == dev_bits(err) == 0
        tombs = merge(tombs, tomb_inputs(slots, K, None, layer, R))
        stored.update(int(t) for t in slots if t >= 0)
        assert_pool_matches(pp, M0, tombs)
    slots = _tokens(shape, rng, 120, 2)
    Ka = synth.kv_values(rng, (L, slots.size, shape.head_num, shape.head_dim), shape.itemsize)
    err = o.store_all(pp.M, slots, Ka, None)
    ids = torch.empty(slots.size, dtype=torch.int32, device="cuda")
    gt.kv_translate(pp.pool, to_dev(slots), ids)
    gt.kv_store_all_layers(pp.pool, ids, to_dev(Ka), None)
    assert pp.last_error() == dev_bits(err) == 0
    for layer in range(L):
        tombs = merge(tombs, tomb_inputs(slots, Ka[layer], None, layer, R))
    stored.update(int(t) for t in slots if t >= 0)
    assert_pool_matches(pp, M0, tombs)
    # gathers: latent rows only
    S_, maxp = 7, min(P - 1, 5)
    bt = np.stack([1 + rng.permutation(P - 1)[:maxp] for _ in range(S_)]).astype(np.int32)
    ln = rng.integers(0, maxp * ps + 1, size=S_).astype(np.int32)
    st = np.minimum(rng.integers(0, ps + 3, size=S_), ln).astype(np.int32)
    gb = synth.GatherBatch(bt, st, ln)
    for layer in sorted({0, L - 1}):
        rows = gb.total + 3
        ok = np.full((rows, R), 0x33, np.uint8)
        ok, ov, err = o.gather(pp.M, layer, bt, ln, gb.cu, st, rows, ok, None)
        dk = torch.full((rows, R), 0x33, dtype=torch.uint8, device="cuda")
        gt.kv_gather_layer(pp.pool, layer, to_dev(bt), to_dev(ln), to_dev(gb.cu), dk, None, to_dev(st))
        assert err == 0 and pp.last_error() == 0
        assert_bytes_equal(dk.cpu().numpy(), ok, f"MLA gather layer {layer}", R)
    # move: all L latent rows of stored tokens to free tokens
    free = np.setdiff1d(np.arange(ps, P * ps, dtype=np.int64), np.array(sorted(stored), np.int64))
    m = min(40, len(stored), free.size)
    src_slots = rng.choice(sorted(stored), size=m, replace=False).astype(np.int64)
    dst_slots = rng.choice(free, size=m, replace=False).astype(np.int64)
    si, _ = o.translate(src_slots)
    di, _ = o.translate(dst_slots)
    err = o.move(pp.M, si, di)
    gt.kv_move(pp.pool, to_dev(si), to_dev(di))
    assert err == 0 and pp.last_error() == 0
    assert_pool_matches(pp, M0, tombs)
    # an MHA-only argument error stays an error on an MHA pool
    mha = PoolPair(synth.SHAPES[1], mirror=False)
    with pytest.raises(gt.KVError):
        gt.kv_store_layer(mha.pool, 0, ids[:4], to_dev(np.zeros((4, mha.R), np.uint8)), None)
    mha.close()
    pp.close()


def test_failed_create_leaves_no_pending_error():
    """A pool the device cannot hold (2 TB of 64 KiB rows): kv_pool_create
    returns KV_ERR_CUDA, allocates nothing, and the failed allocation does not
    surface as the status of the next launch on another pool."""
    huge = gt.make_desc(1, 64, 256, 4, 16, 1 << 20)  # n_rows = 2^25 < 2^31, 64 KiB rows
    total, _ = gt.kv_pool_required_bytes(huge)
    assert total >= 1 << 41
    with pytest.raises(gt.KVError) as e:
        gt.kv_pool_create(huge)
    assert e.value.name == "KV_ERR_CUDA"
    pool = gt.kv_pool_create(gt.make_desc(2, 2, 8, 2, 4, 8))
    ids = torch.empty(2, dtype=torch.int32, device="cuda")
    gt.kv_translate(pool, torch.tensor([5, -1], dtype=torch.int64, device="cuda"), ids)
    assert ids.cpu().tolist() == [1 * 16 + 1, 0] and gt.kv_pool_last_error(pool) == 0
    gt.kv_pool_destroy(pool)


def test_library_owned_buffer_round_trip():
    """kv_pool_create without a buffer: the library allocates anchor + total +
    tail pad bytes itself; a store then a gather returns the stored rows, and
    kv_pool_destroy frees it."""
    shape = synth.SHAPES[2].scaled(20)
    ps, P = shape.page_size, shape.num_pages
    desc = gt.make_desc(shape.layer_num, shape.head_num, shape.head_dim, shape.itemsize, ps, P, anchor_bytes=256)
    pool = gt.kv_pool_create(desc)
    info = pool.info
    total, pad = gt.kv_pool_required_bytes(desc)
    assert info["owns_raw"] == 1 and info["raw_dev"] and info["raw_bytes"] == 256 + total + pad
    rng = np.random.default_rng(21)
    pages = (1 + rng.permutation(P - 1)[:4]).astype(np.int32)
    slots = (pages.astype(np.int64)[:, None] * ps + np.arange(ps)).reshape(-1)
    K, V = _vals(shape, rng, (slots.size,))
    ids = torch.empty(slots.size, dtype=torch.int32, device="cuda")
    gt.kv_translate(pool, to_dev(slots), ids)
    gt.kv_store_layer(pool, 5, ids, to_dev(K), to_dev(V))
    g = synth.GatherBatch(pages[None, :], np.zeros(1, np.int32), np.array([slots.size], np.int32))
    dk = torch.empty((g.total, shape.row_bytes), dtype=torch.uint8, device="cuda")
    dv = torch.empty_like(dk)
    gt.kv_gather_layer(pool, 5, to_dev(g.block_table), to_dev(g.seq_len), to_dev(g.cu), dk, dv)
    assert gt.kv_pool_last_error(pool) == 0
    assert np.array_equal(dk.cpu().numpy(), as_rows(K, shape.row_bytes))
    assert np.array_equal(dv.cpu().numpy(), as_rows(V, shape.row_bytes))
    gt.kv_pool_destroy(pool)


@pytest.mark.parametrize("shape,anchor,latent", [(s, a, False) for s, a in SHAPES[:8]] + [(MLA_SHAPES[0][0], 0, True)],
                         ids=IDS[:8] + [MLA_SHAPES[0][0].name])
def test_planned_gather_matches_oracle(shape, anchor, latent):
    """kv_gather_plan + kv_gather_layer_planned: the plan holds every entry
    that has tokens in its sequence's window exactly once, grouped by page,
    and the planned gather writes exactly what the oracle's gather writes."""
    rng = np.random.default_rng(600 + shape.row_bytes + shape.page_size)
    pp = PoolPair(shape, anchor, latent=latent)
    o, R, L, ps, P = pp.o, pp.R, shape.layer_num, shape.page_size, shape.num_pages
    S_, maxp = 23, min(P - 1, 6)
    # heavily shared pages: every sequence draws from a few pages
    bt = rng.integers(1, min(P, 5), size=(S_, maxp)).astype(np.int32)
    bt[3, 1] = -1  # a tombstoned entry reads the sink
    ln = rng.integers(0, maxp * ps + 1, size=S_).astype(np.int32)
    ln[0], ln[5] = maxp * ps, 0
    st = np.minimum(rng.integers(0, 2 * ps, size=S_), ln).astype(np.int32)
    g = synth.GatherBatch(bt, st, ln)
    plan = gt.kv_gather_plan(pp.pool, to_dev(bt), to_dev(ln), to_dev(st))
    assert pp.last_error() == 0
    h = plan.cpu().numpy()
    n_valid, entries = int(h[0]), h[4 + P + 1:]
    want = [s * maxp + k for s in range(S_) for k in range(maxp) if k * ps < ln[s] and (k + 1) * ps > st[s]]
    assert (h[1], h[2]) == (S_, maxp) and n_valid == len(want)
    assert h[3] == 1, "pages this shared should be walked page by page"
    assert sorted(entries[:n_valid].tolist()) == sorted(want)
    pages = np.maximum(bt.reshape(-1)[entries[:n_valid]], 0)
    assert np.all(np.diff(pages) >= 0), "plan entries are not grouped by page"
    for layer in sorted({0, L - 1}):
        rows = g.total + 2
        ok = np.full((rows, R), 0x11, np.uint8)
        ov = None if latent else np.full((rows, R), 0x22, np.uint8)
        ok, ov, err = o.gather(pp.M, layer, bt, ln, g.cu, st, rows, ok, ov)
        dk = torch.full((rows, R), 0x11, dtype=torch.uint8, device="cuda")
        dv = None if latent else torch.full((rows, R), 0x22, dtype=torch.uint8, device="cuda")
        gt.kv_gather_layer_planned(pp.pool, layer, plan, to_dev(bt), to_dev(ln), to_dev(g.cu), dk, dv, to_dev(st))
        assert err == 0 and pp.last_error() == 0
        assert_bytes_equal(dk.cpu().numpy(), ok, f"planned gather K layer {layer}", R)
        if not latent:
            assert_bytes_equal(dv.cpu().numpy(), ov, f"planned gather V layer {layer}", R)
    # distinct pages: the plan says to keep the table's order, and the planned
    # gather still matches the oracle
    if P - 1 >= S_ * maxp:
        btd = (1 + rng.permutation(P - 1)[: S_ * maxp]).reshape(S_, maxp).astype(np.int32)
        pd = gt.kv_gather_plan(pp.pool, to_dev(btd), to_dev(ln), to_dev(st))
        assert int(pd.cpu()[3]) == 0
        ok, ov, err = o.gather(pp.M, 0, btd, ln, g.cu, st, g.total)
        dk = torch.zeros((g.total, R), dtype=torch.uint8, device="cuda")
        dv = None if latent else torch.zeros((g.total, R), dtype=torch.uint8, device="cuda")
        gt.kv_gather_layer_planned(pp.pool, 0, pd, to_dev(btd), to_dev(ln), to_dev(g.cu), dk, dv, to_dev(st))
        assert err == 0 and pp.last_error() == 0
        assert_bytes_equal(dk.cpu().numpy(), ok, "planned gather, table order", R)
    # a plan built for another table shape: a buffer too small for this table
    # is refused on the host, a large enough one on the device; nothing written
    dk = torch.full((g.total, R), 0x33, dtype=torch.uint8, device="cuda")
    dv = None if latent else torch.full((g.total, R), 0x33, dtype=torch.uint8, device="cuda")
    small = gt.kv_gather_plan(pp.pool, to_dev(bt[:, :-1]), to_dev(np.minimum(ln, (maxp - 1) * ps)))
    with pytest.raises(gt.KVError) as e:
        gt.kv_gather_layer_planned(pp.pool, 0, small, to_dev(bt), to_dev(ln), to_dev(g.cu), dk, dv, to_dev(st))
    assert e.value.name == "KV_ERR_INVALID"
    other = gt.kv_gather_plan(pp.pool, to_dev(np.concatenate([bt, bt])), to_dev(np.concatenate([ln, ln])))
    gt.kv_gather_layer_planned(pp.pool, 0, other, to_dev(bt), to_dev(ln), to_dev(g.cu), dk, dv, to_dev(st))
    assert pp.last_error() == gt.KV_DEV_ERR_TABLE
    assert bool((dk == 0x33).all())
    pp.close()


@pytest.mark.parametrize("shape,anchor,latent", [(synth.SHAPES[2].scaled(40), 0, False), (SHAPES[5][0], 16, False),
                                                 (synth.SHAPES[5].scaled(20), 0, False),
                                                 (MLA_SHAPES[0][0], 0, True),
                                                 (S(0, "mla-r1152-ps128", 3, 1, 576, 2, 128, 12), 0, True),
                                                 (S(0, "mla-r512-ps256", 2, 1, 256, 2, 256, 10), 16, True),
                                                 (S(0, "r2048-ps64", 2, 8, 128, 2, 64, 12), 0, False)],
                         ids=["R2048-ps16", "odd-rows", "R64-ps256", "mla-r1152", "mla-r1152-ps128-vector",
                              "mla-r512-ps256-vector", "R2048-ps64-vector"])
def test_planned_gather_both_forms(shape, anchor, latent):
    """Where a page holds at most 72 KiB per layer (the first four shapes)
    the gathers stage pages in shared memory and bulk-copy them to their
    readers, with two plan positions per block for tables of at least
    num_pages entries and one below that; larger pages (the last three,
    including the 1152-byte latent rows' own vector rounds) are copied by warps
    through registers. The same pool read through a table on each side of the
    table-size rule, with shared pages, tombstoned entries, windows starting
    mid-page and gaps between the output spans, must equal the oracle's
    gather, in both table forms, planned and not."""
    rng = np.random.default_rng(700 + shape.row_bytes)
    pp = PoolPair(shape, anchor, latent=latent)
    o, R, L, ps, P = pp.o, pp.R, shape.layer_num, shape.page_size, shape.num_pages
    B = pp.pool.info["blocks_per_page"]
    staged = (2 - latent) * ps * R <= 73728
    maxp = min(P - 1, 6)
    for S_ in (-(-P // maxp) + 3, max(1, (P - 1) // maxp)):  # n_seqs * max_pages >= P, then < P
        fan = S_ * maxp >= P
        bt = np.where(rng.random((S_, maxp)) < 0.7, rng.integers(1, min(P, 6), size=(S_, maxp)),
                      rng.integers(1, P, size=(S_, maxp))).astype(np.int32)
        bt[rng.random((S_, maxp)) < 0.05] = -1
        ln = rng.integers(0, maxp * ps + 1, size=S_).astype(np.int32)
        ln[0] = maxp * ps
        st = np.minimum(rng.integers(0, 2 * ps, size=S_), ln).astype(np.int32)
        cu = np.zeros(S_ + 1, np.int64)
        cu[1:] = np.cumsum(ln - st + rng.integers(0, 3, size=S_))  # gaps between the spans stay untouched
        rows = int(cu[-1]) + 2
        kf = np.where(bt >= 0, bt * B, bt).astype(np.int32)
        for form, table in (("physical", bt), ("kernel-facing", kf)):
            plan = (gt.kv_gather_plan_kf if form == "kernel-facing" else gt.kv_gather_plan)(
                pp.pool, to_dev(table), to_dev(ln), to_dev(st))
            assert pp.last_error() == 0
            for layer in sorted({0, L - 1}):
                ok = np.full((rows, R), 0x11, np.uint8)
                ov = None if latent else np.full((rows, R), 0x22, np.uint8)
                ok, ov, err = o.gather(pp.M, layer, bt, ln, cu, st, rows, ok, ov)
                assert err == 0
                dk = torch.full((rows, R), 0x11, dtype=torch.uint8, device="cuda")
                dv = None if latent else torch.full((rows, R), 0x22, dtype=torch.uint8, device="cuda")
                fn = gt.kv_gather_layer_planned_kf if form == "kernel-facing" else gt.kv_gather_layer_planned
                fn(pp.pool, layer, plan, to_dev(table), to_dev(ln), to_dev(cu), dk, dv, to_dev(st))
                assert pp.last_error() == 0
                what = (f"planned gather ({2 if fan else 1} positions per block), " if staged else
                        "planned gather (vector kernel), ") + f"{form} table, layer {layer}"
                assert_bytes_equal(dk.cpu().numpy(), ok, what + " K", R)
                if not latent:
                    assert_bytes_equal(dv.cpu().numpy(), ov, what + " V", R)
                dk.fill_(0x11)
                if not latent:
                    dv.fill_(0x22)
                fn = gt.kv_gather_layer_kf if form == "kernel-facing" else gt.kv_gather_layer
                fn(pp.pool, layer, to_dev(table), to_dev(ln), to_dev(cu), dk, dv, to_dev(st))
                assert pp.last_error() == 0
                assert_bytes_equal(dk.cpu().numpy(), ok, f"gather without a plan, {form} table, layer {layer} K", R)
                if not latent:
                    assert_bytes_equal(dv.cpu().numpy(), ov, f"gather without a plan, {form} table, layer {layer} V",
                                       R)
    pp.close()
