"""Randomised geometries on GPU against the oracle: row sizes from 16 bytes to
4 KiB (and the generic whole-warp path), page sizes that chunks do not divide,
anchors, MLA pools, shared and tombstoned block-table entries, partial windows,
empty sequences. Each case runs translate (with a page map), per-layer and
all-layer stores, the table-order, planned and allocation-free-planned gathers,
the kernel-facing table build and both gathers that read it, and a move, and
compares every byte of the pool and of the outputs."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import gather_translate_kv_gb300 as gt
import oracle
import synth
from gpu_util import PoolPair, assert_bytes_equal, assert_pool_matches, dev_bits, merge, to_dev, tomb_inputs

pytestmark = pytest.mark.gpu

ROWS = (16, 32, 48, 64, 96, 128, 192, 256, 512, 1024, 1152, 1536, 2048, 4096)
PAGE_SIZES = (1, 2, 3, 5, 7, 8, 16, 33, 64)


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gather_translate_kv_gb300 import build

    build.build()
    oracle.build()


def _geometry(rng: np.random.Generator):
    while True:
        R = int(rng.choice(ROWS))
        itemsize = int(rng.choice((1, 2)))
        H = int(rng.choice((1, 2, 3, 4, 8)))
        if R % (H * itemsize):
            continue
        D = R // (H * itemsize)
        ps = int(rng.choice(PAGE_SIZES))
        L = int(rng.integers(1, 7))
        P = int(rng.integers(12, 160))
        latent = bool(rng.random() < 0.2)
        if P * ps * (L if latent else 2 * L) * R > (48 << 20):  # keep the pool small
            continue
        anchor = 16 * int(rng.integers(0, 40)) if rng.random() < 0.4 else 0
        return synth.Shape(0, f"fuzz-R{R}-ps{ps}", L, H, D, itemsize, ps, P, latent), anchor


@pytest.mark.parametrize("seed", range(160))
def test_random_geometry_matches_oracle(seed):
    rng = np.random.default_rng(7000 + seed)
    shape, anchor = _geometry(rng)
    latent = shape.latent
    pp = PoolPair(shape, anchor, fill_seed=11 + seed, latent=latent)
    o, R, L, ps, P = pp.o, pp.R, shape.layer_num, shape.page_size, shape.num_pages
    M0 = pp.M.copy()
    tomb = {}

    # translate through a page map with a few unmapped pages
    v2p = rng.permutation(P).astype(np.int32)
    v2p[rng.choice(P, size=2, replace=False)] = -1
    slots = rng.integers(-3, P * ps, size=int(rng.integers(1, 300))).astype(np.int64)
    ids_ref, err = o.translate(slots, v2p)
    ids = torch.empty(slots.size, dtype=torch.int32, device="cuda")
    gt.kv_translate(pp.pool, to_dev(slots), ids, to_dev(v2p))
    assert np.array_equal(ids.cpu().numpy(), ids_ref)
    assert pp.last_error() == dev_bits(err)

    # stores: distinct slots outside page 0, some tombstoned, into random layers
    n = int(rng.integers(1, min(400, (P - 1) * ps) + 1))
    st_slots = synth.with_tombstones(rng, synth.distinct_slots(rng, ps, P * ps, n), min(n, int(rng.integers(0, 4))))
    ids_d = torch.empty(n, dtype=torch.int32, device="cuda")
    gt.kv_translate(pp.pool, to_dev(st_slots), ids_d)
    for layer in sorted(set(rng.integers(0, L, size=2).tolist())):
        K = synth.kv_values(rng, (n, shape.head_num, shape.head_dim), shape.itemsize)
        V = None if latent else synth.kv_values(rng, (n, shape.head_num, shape.head_dim), shape.itemsize)
        assert o.store(pp.M, layer, st_slots, K, V) == 0
        gt.kv_store_layer(pp.pool, layer, ids_d, to_dev(K), None if V is None else to_dev(V))
        tomb = merge(tomb, tomb_inputs(st_slots, K, V, layer, R))
    Ka = synth.kv_values(rng, (L, n, shape.head_num, shape.head_dim), shape.itemsize)
    Va = None if latent else synth.kv_values(rng, (L, n, shape.head_num, shape.head_dim), shape.itemsize)
    assert o.store_all(pp.M, st_slots, Ka, Va) == 0
    gt.kv_store_all_layers(pp.pool, ids_d, to_dev(Ka), None if Va is None else to_dev(Va))
    for layer in range(L):
        tomb = merge(tomb, tomb_inputs(st_slots, Ka[layer], None if Va is None else Va[layer], layer, R))
    assert pp.last_error() == 0
    assert_pool_matches(pp, M0, tomb)
    # the sink rows hold words of racing tombstone writers (checked just above):
    # take the device's bytes into the mirror so gathers of tombstoned entries
    # read the same sink on both sides
    got = pp.raw.cpu().numpy()
    for sb in pp.sink_bytes():
        pp.M[sb:sb + R] = got[sb:sb + R]

    # gathers: shared pages, tombstoned entries, partial windows, empty sequences
    S = int(rng.integers(1, 40))
    maxp = int(rng.integers(1, 12))
    hot = rng.integers(1, P, size=max(1, P // 8))
    bt = np.where(rng.random((S, maxp)) < 0.5, rng.choice(hot, size=(S, maxp)),
                  rng.integers(1, P, size=(S, maxp))).astype(np.int32)
    bt[rng.random((S, maxp)) < 0.03] = -1
    ln = rng.integers(0, maxp * ps + 1, size=S).astype(np.int32)
    st = np.minimum(rng.integers(0, 2 * ps + 1, size=S), ln).astype(np.int32)
    g = synth.GatherBatch(bt, st, ln)
    rows = g.total
    plan = gt.kv_gather_plan(pp.pool, to_dev(bt), to_dev(ln), to_dev(st))
    plan_na = torch.full_like(plan, -5)
    gt.kv_gather_plan_noalloc(pp.pool, to_dev(bt), to_dev(ln), plan_na, to_dev(st))
    assert pp.last_error() == 0
    for layer in sorted(set(rng.integers(0, L, size=2).tolist())):
        ok, ov, err = o.gather(pp.M, layer, bt, ln, g.cu, st, rows)
        assert err == 0
        for how in ("table", "plan", "plan_noalloc"):
            dk = torch.full((rows, R), 0x6B, dtype=torch.uint8, device="cuda")
            dv = None if latent else torch.full((rows, R), 0x6B, dtype=torch.uint8, device="cuda")
            if how == "table":
                gt.kv_gather_layer(pp.pool, layer, to_dev(bt), to_dev(ln), to_dev(g.cu), dk, dv, to_dev(st))
            else:
                gt.kv_gather_layer_planned(pp.pool, layer, plan if how == "plan" else plan_na, to_dev(bt),
                                           to_dev(ln), to_dev(g.cu), dk, dv, to_dev(st))
            assert pp.last_error() == 0
            assert_bytes_equal(dk.cpu().numpy(), ok, f"{shape.name} gather K ({how}) layer {layer}", R)
            if not latent:
                assert_bytes_equal(dv.cpu().numpy(), ov, f"{shape.name} gather V ({how}) layer {layer}", R)

    # the read path through a kernel-facing table: the same table read as
    # virtual pages through the page map, prefix-only build, then both
    # kernel-facing gathers
    kf_ref, err = o.block_table_kf(bt, ln, v2p, out=np.full(bt.shape, -7, np.int32))
    kf_d = torch.full(bt.shape, -7, dtype=torch.int32, device="cuda")
    gt.kv_translate_block_table(pp.pool, to_dev(bt), to_dev(ln), to_dev(v2p), kf_d)
    assert pp.last_error() == dev_bits(err)
    assert np.array_equal(kf_d.cpu().numpy(), kf_ref)
    plan_kf = gt.kv_gather_plan_kf(pp.pool, kf_d, to_dev(ln), to_dev(st))
    assert pp.last_error() == 0
    for layer in sorted(set(rng.integers(0, L, size=2).tolist())):
        ok, ov, err = o.gather_kf(pp.M, layer, kf_ref, ln, g.cu, st, rows)
        assert err == 0
        for how in ("kf", "kf_plan"):
            dk = torch.full((rows, R), 0x6B, dtype=torch.uint8, device="cuda")
            dv = None if latent else torch.full((rows, R), 0x6B, dtype=torch.uint8, device="cuda")
            if how == "kf":
                gt.kv_gather_layer_kf(pp.pool, layer, kf_d, to_dev(ln), to_dev(g.cu), dk, dv, to_dev(st))
            else:
                gt.kv_gather_layer_planned_kf(pp.pool, layer, plan_kf, kf_d, to_dev(ln), to_dev(g.cu), dk, dv,
                                              to_dev(st))
            assert pp.last_error() == 0
            assert_bytes_equal(dk.cpu().numpy(), ok, f"{shape.name} gather K ({how}) layer {layer}", R)
            if not latent:
                assert_bytes_equal(dv.cpu().numpy(), ov, f"{shape.name} gather V ({how}) layer {layer}", R)

    # move: disjoint src (stored slots) and dst (fresh slots) sets
    live = st_slots[st_slots >= 0]
    free = np.setdiff1d(np.arange(ps, P * ps, dtype=np.int64), live)
    m = int(rng.integers(0, min(live.size, free.size, 64) + 1))
    src = rng.choice(live, size=m, replace=False) if m else np.zeros(0, np.int64)
    dst = rng.choice(free, size=m, replace=False) if m else np.zeros(0, np.int64)
    src_ids, _ = o.translate(src)
    dst_ids, _ = o.translate(dst)
    assert o.move(pp.M, src_ids, dst_ids) == 0
    if m:
        gt.kv_move(pp.pool, to_dev(src_ids), to_dev(dst_ids))
    assert pp.last_error() == 0
    assert_pool_matches(pp, M0, tomb)
    pp.close()
