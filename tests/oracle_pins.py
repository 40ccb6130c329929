"""Pins that hold the CPU oracle to the report, not to itself.

Each ``pin_*`` function takes the path of a compiled oracle library and
raises AssertionError when the oracle disagrees with something fixed
independently of it:

  * hand-computed values of the report's closed forms (tests/golden/),
  * an independently built [page, 2L, ps, H, D] reference (strided_ref),
  * the dense per-layer view arithmetic of build_mha_views (view base
    anchor + b*ps*R plus id*R) against the oracle's envelope offsets,
  * brute-force invariants on tiny pools (bijection, exact tiling),
  * round trips (store then gather, move then gather).

Run as a script (``python oracle_pins.py <lib.so>``) it executes every pin
and exits 1 at the first failure; the mutation test uses that to show each
planted mistake is caught. Source of every rule: the prhub report on sglang
PR #34602, "feat(unified-memory): dense KV views for uniform-row MHA/SWA
models".
"""
from __future__ import annotations

import ctypes
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
for p in (ROOT, HERE):
    if p not in sys.path:
        sys.path.insert(0, p)

import oracle  # noqa: E402
import strided_ref  # noqa: E402
import synth  # noqa: E402

GOLDEN = os.path.join(HERE, "golden")


def _rows(path):
    out = []
    with open(path) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                out.append(line.split())
    return out


def _geom(L, H, D, it, ps, P, anchor=0, Dv=None, latent=False):
    return oracle.Geometry(L, H, D, it, ps, P, anchor, Dv, latent)


def _mk(so, g):
    return oracle.Oracle(g, so)


def _fresh(o: oracle.Oracle, seed=7):
    n = o.raw_bytes()
    return synth.sentinel_bytes(seed, 0, n)


# ----------------------------------------------------------------- pins

def pin_translate_golden(so):
    """Hand-computed kernel ids for the tiny pool (tests/golden/translate_tiny.txt)."""
    o = _mk(so, _geom(2, 2, 8, 2, 4, 64))
    maps = {
        "none": None,
        "tomb1": np.where(np.arange(64) == 1, -1, np.arange(64)).astype(np.int32),
        "p1to9": np.where(np.arange(64) == 1, 9, np.arange(64)).astype(np.int32),
    }
    for slot, case, want in _rows(os.path.join(GOLDEN, "translate_tiny.txt")):
        ids, err = o.translate(np.array([int(slot)]), maps[case])
        assert err == 0, (slot, case, err)
        assert int(ids[0]) == int(want), (slot, case, int(ids[0]), want)


def pin_layout_table(so):
    """Per-workload layout numbers (tests/golden/layout_table.txt)."""
    for r in _rows(os.path.join(GOLDEN, "layout_table.txt")):
        L, H, D, it, ps, P = map(int, r[:6])
        R, pb, tot, tp, nr, lve = map(int, r[7:])
        s = _mk(so, _geom(L, H, D, it, ps, P)).sizes()
        got = (s["row_bytes"], s["page_bytes"], s["total"], s["tail_pad"], s["n_rows"], s["last_view_end"])
        assert got == (R, pb, tot, tp, nr, lve), (r, got)


def pin_gates(so):
    """Start-up gates: uniform rows, anchor alignment, id bound, tail pad."""
    g = {k: int(v) for k, v in _rows(os.path.join(GOLDEN, "id_bound.txt"))}
    ok = _mk(so, _geom(80, 1, 64, 1, 256, g["max_pages_ok"]))
    assert ok.check() == "ok"
    bad = _mk(so, _geom(80, 1, 64, 1, 256, g["first_pages_rejected"]))
    assert bad.check() == "id_bound"
    st = _mk(so, _geom(80, 1, 64, 1, 256, 48828))
    assert st.sizes()["n_rows"] == g["stress_n_rows"]
    ids, err = st.translate(np.array([g["stress_last_slot"]]))
    assert err == 0 and int(ids[0]) == g["stress_last_slot_id"], int(ids[0])
    # the view-space row of that slot in block 159 is the last row of the view
    assert int(ids[0]) + 159 * 256 == g["stress_last_row_b159"] == g["stress_n_rows"] - 1
    assert _mk(so, _geom(1, 1, 16, 1, 2, g["edge_pages_rejected"])).check() == "id_bound"
    assert _mk(so, _geom(1, 1, 16, 1, 2, g["edge_pages_ok"])).check() == "ok"
    assert _mk(so, _geom(2, 2, 8, 2, 4, 64, Dv=16)).check() == "asymmetric"
    assert _mk(so, _geom(2, 2, 8, 2, 4, 64, anchor=3)).check() == "anchor"
    assert _mk(so, _geom(2, 2, 8, 2, 4, 64, anchor=4)).check() == "ok"
    t = _mk(so, _geom(2, 2, 8, 2, 4, 64))
    lve = t.sizes()["last_view_end"]
    # build_mha_views: the last view ends exactly (2L-1)*ps rows past the pool
    assert lve == 32768 + 3 * 4 * 32
    assert t.check(lve) == "ok" and t.check(lve - 1) == "tail_pad"
    # the pool's own allocation, total + one page envelope, always suffices
    assert t.check(t.raw_bytes()) == "ok"


def pin_bijection(so):
    """Brute force on tiny pools: (slot, block) -> row is a bijection that tiles
    the pool exactly, and the oracle's envelope offset of (slot, block) equals
    the dense view of build_mha_views at row kernel_id(slot): view base
    anchor + b*ps*R plus kernel_id*R."""
    for (L, H, D, it, ps, P, anchor) in [
        (1, 1, 8, 2, 1, 5, 0), (2, 2, 8, 2, 4, 6, 32), (3, 1, 16, 1, 2, 7, 16),
        (1, 2, 4, 4, 8, 3, 0), (4, 1, 32, 1, 3, 5, 64),
    ]:
        o = _mk(so, _geom(L, H, D, it, ps, P, anchor))
        s = o.sizes()
        R = s["row_bytes"]
        slots = np.arange(P * ps, dtype=np.int64)
        ids, err = o.translate(slots)
        assert err == 0
        seen_rows, seen_bytes = [], []
        for t, kid in zip(slots, ids):
            for b in range(2 * L):
                byte = o.slot_row_byte(int(t), b)
                assert byte == anchor + b * ps * R + int(kid) * R, (t, b, byte)
                seen_rows.append(int(kid) + b * ps)
                seen_bytes.append(byte)
        assert sorted(seen_rows) == list(range(P * 2 * L * ps))
        assert sorted(seen_bytes) == [anchor + R * k for k in range(s["n_rows"])]
        assert anchor + R * s["n_rows"] == anchor + s["total"]
        # ids decode back to the same bytes (the move's decoding)
        for kid in ids[:: max(1, len(ids) // 17)]:
            for b in (0, 2 * L - 1):
                assert o.id_row_byte(int(kid), b) == anchor + b * ps * R + int(kid) * R


def _random_case(rng, L, H, D, it, ps, P, anchor, n, tomb):
    slots = rng.permutation(np.arange(ps, P * ps))[:n].astype(np.int64)
    if tomb:
        slots[rng.choice(n, size=tomb, replace=False)] = -1
    K = synth.kv_values(rng, (n, H, D), it)
    V = synth.kv_values(rng, (n, H, D), it)
    return slots, K, V


def pin_store_vs_strided(so):
    """Per-layer and all-layer stores equal the [page, 2L, ps, H, D] reference
    byte for byte (tombstones included: both write in input order)."""
    rng = np.random.default_rng(11)
    for (L, H, D, it, ps, P, anchor, n, tomb) in [
        (2, 2, 8, 2, 4, 64, 0, 100, 5), (3, 2, 4, 1, 8, 9, 16, 40, 3),
        (1, 1, 16, 2, 2, 11, 0, 18, 0), (24, 1, 16, 1, 32, 3, 32, 50, 4),
    ]:
        o = _mk(so, _geom(L, H, D, it, ps, P, anchor))
        M = _fresh(o)
        T = M.copy()
        env = strided_ref.envelope(T, L, H, D, it, ps, P, anchor)
        for layer in range(L):
            slots, K, V = _random_case(rng, L, H, D, it, ps, P, anchor, n, tomb)
            assert o.store(M, layer, slots, K, V) == 0
            strided_ref.store(env, layer, slots, K, V)
            assert np.array_equal(M, T), ("store", L, layer)
        slots, K, V = _random_case(rng, L, H, D, it, ps, P, anchor, n, tomb)
        Ka = np.stack([synth.kv_values(rng, (n, H, D), it) for _ in range(L)])
        Va = np.stack([synth.kv_values(rng, (n, H, D), it) for _ in range(L)])
        assert o.store_all(M, slots, Ka, Va) == 0
        for layer in range(L):
            strided_ref.store(env, layer, slots, Ka[layer], Va[layer])
        assert np.array_equal(M, T), ("store_all", L)


def pin_v2p_store(so):
    """Virtual->physical page map: store through the map equals the reference
    store through the same map; tombstoned pages land on the sink."""
    rng = np.random.default_rng(12)
    L, H, D, it, ps, P = 2, 2, 8, 2, 4, 16
    o = _mk(so, _geom(L, H, D, it, ps, P))
    v2p = (1 + rng.permutation(P - 1)).astype(np.int32)[: P - 1]
    v2p = np.concatenate([[-1], v2p]).astype(np.int32)  # virtual page 0 -> tombstone
    v2p[5] = -1
    slots = rng.permutation(np.arange(0, P * ps))[:30].astype(np.int64)
    K = synth.kv_values(rng, (30, H, D), it)
    V = synth.kv_values(rng, (30, H, D), it)
    M = _fresh(o)
    T = M.copy()
    env = strided_ref.envelope(T, L, H, D, it, ps, P)
    assert o.store(M, 1, slots, K, V, v2p) == 0
    strided_ref.store(env, 1, slots, K, V, v2p)
    assert np.array_equal(M, T)
    ids, err = o.translate(slots, v2p)
    assert err == 0
    for t, kid in zip(slots, ids):
        vp, off = divmod(int(t), ps)
        if v2p[vp] < 0:
            assert kid == 0
        else:
            assert o.slot_row_byte(int(t), 2, v2p) == (int(kid) + 2 * ps) * H * D * it
    # a page index past the map is an error and lands on the sink
    ids, err = o.translate(np.array([P * ps + 1], np.int64), v2p[: P // 2])
    assert err == oracle.E_V2P and ids[0] == 0


def pin_gather_vs_strided(so):
    """Gather equals the reference read, for full windows, windows starting
    mid-page, empty sequences and tombstoned (negative) table entries."""
    rng = np.random.default_rng(13)
    for (L, H, D, it, ps, P, anchor) in [(2, 2, 8, 2, 4, 64, 0), (3, 1, 32, 1, 8, 13, 48)]:
        o = _mk(so, _geom(L, H, D, it, ps, P, anchor))
        M = _fresh(o, seed=99)
        env = strided_ref.envelope(M, L, H, D, it, ps, P, anchor)
        S, maxp = 5, 6
        bt = rng.integers(1, P, size=(S, maxp)).astype(np.int32)
        bt[2, 1] = -1
        ln = np.array([maxp * ps, 3, 0, maxp * ps - 5, 2 * ps + 1], np.int32)
        st = np.array([0, 1, 0, ps + 2, 2 * ps], np.int32)
        g = synth.GatherBatch(bt, st, ln)
        for layer in range(L):
            k, v, err = o.gather(M, layer, bt, ln, g.cu, st)
            assert err == 0
            rk, rv = strided_ref.gather(env, layer, bt, st, ln)
            assert np.array_equal(k, rk.reshape(len(rk), -1).view(np.uint8).reshape(k.shape))
            assert np.array_equal(v, rv.reshape(len(rv), -1).view(np.uint8).reshape(v.shape))


def pin_roundtrip(so):
    """Store then gather returns the stored rows; move then gather at the
    destination returns the source rows, and nothing else changes."""
    rng = np.random.default_rng(14)
    L, H, D, it, ps, P = 3, 2, 8, 2, 4, 20
    o = _mk(so, _geom(L, H, D, it, ps, P))
    R = o.sizes()["row_bytes"]
    M = _fresh(o)
    pages = (1 + rng.permutation(P - 1)[:6]).astype(np.int32)
    bt = pages[None, :]
    slots = (pages.astype(np.int64)[:, None] * ps + np.arange(ps)).reshape(-1)
    n = slots.size
    for layer in range(L):
        K = synth.kv_values(rng, (n, H, D), it)
        V = synth.kv_values(rng, (n, H, D), it)
        assert o.store(M, layer, slots, K, V) == 0
        g = synth.GatherBatch(bt, np.zeros(1, np.int32), np.array([n], np.int32))
        k, v, err = o.gather(M, layer, bt, g.seq_len, g.cu, g.seq_start)
        assert err == 0
        assert np.array_equal(k, K.reshape(n, -1).view(np.uint8).reshape(n, R))
        assert np.array_equal(v, V.reshape(n, -1).view(np.uint8).reshape(n, R))
    # move: tokens of the first two pages -> two fresh pages
    free = np.setdiff1d(np.arange(1, P), pages)[:2].astype(np.int64)
    src_slots = slots[: 2 * ps]
    dst_slots = (free[:, None] * ps + np.arange(ps)).reshape(-1)
    src_ids, e1 = o.translate(src_slots)
    dst_ids, e2 = o.translate(dst_slots)
    before = M.copy()
    assert o.move(M, src_ids, dst_ids) == 0
    T = before.copy()
    strided_ref.move(strided_ref.envelope(T, L, H, D, it, ps, P), src_slots, dst_slots)
    assert np.array_equal(M, T)
    btd = free.astype(np.int32)[None, :]
    bts = pages[:2][None, :]
    for layer in range(L):
        g = synth.GatherBatch(btd, np.zeros(1, np.int32), np.array([2 * ps], np.int32))
        kd, vd, _ = o.gather(M, layer, btd, g.seq_len, g.cu, g.seq_start)
        ks, vs, _ = o.gather(before, layer, bts, g.seq_len, g.cu, g.seq_start)
        assert np.array_equal(kd, ks) and np.array_equal(vd, vs)
    changed = np.nonzero(M != before)[0]
    dst_bytes = {o.slot_row_byte(int(t), b) for t in dst_slots for b in range(2 * L)}
    assert all(any(d <= c < d + R for d in dst_bytes) for c in changed[:: max(1, len(changed) // 200)])


def pin_tail_untouched(so):
    """Writing every slot of every layer never touches the anchor prefix or
    the tail pad (the tail pad exists only so the last view stays in bounds)."""
    rng = np.random.default_rng(15)
    L, H, D, it, ps, P, anchor = 2, 1, 16, 2, 4, 5, 64
    o = _mk(so, _geom(L, H, D, it, ps, P, anchor))
    s = o.sizes()
    M = _fresh(o)
    before = M.copy()
    slots = np.arange(P * ps, dtype=np.int64)
    Ka = synth.kv_values(rng, (L, slots.size, H, D), it)
    Va = synth.kv_values(rng, (L, slots.size, H, D), it)
    assert o.store_all(M, slots, Ka, Va) == 0
    assert np.array_equal(M[:anchor], before[:anchor])
    assert np.array_equal(M[anchor + s["total"] :], before[anchor + s["total"] :])
    assert np.count_nonzero(M[anchor : anchor + s["total"]] != before[anchor : anchor + s["total"]]) > 0


def pin_errors(so):
    """Error reporting: ids past the pool, ids not in translate form, gather
    metadata that does not fit the output, and pages past the pool."""
    L, H, D, it, ps, P = 2, 1, 16, 1, 4, 8
    o = _mk(so, _geom(L, H, D, it, ps, P))
    M = _fresh(o)
    before = M.copy()
    stride = ps * 2 * L
    assert o.move(M, np.array([P * stride], np.int32), np.array([stride], np.int32)) == oracle.E_ROW
    assert o.move(M, np.array([stride + ps], np.int32), np.array([2 * stride], np.int32)) == oracle.E_FORM
    assert np.array_equal(M, before)
    ids, err = o.translate(np.array([P * ps], np.int64))
    assert err == oracle.E_ROW and ids[0] == 0
    bt = np.array([[1, P]], np.int32)
    k, v, err = o.gather(M, 0, bt, np.array([2 * ps], np.int32), np.array([0, 2 * ps], np.int64))
    assert err == oracle.E_ROW
    k, v, err = o.gather(M, 0, bt[:, :1], np.array([ps], np.int32), np.array([0, ps - 1], np.int64),
                         out_rows=ps - 1)
    assert err == oracle.E_TABLE


def pin_address_mode(so):
    """The address-mode routines (used to check full-size runs) name exactly
    the bytes the copying routines move."""
    rng = np.random.default_rng(16)
    L, H, D, it, ps, P = 3, 1, 16, 2, 4, 12
    o = _mk(so, _geom(L, H, D, it, ps, P))
    R = o.sizes()["row_bytes"]
    slots = rng.permutation(np.arange(ps, P * ps))[:20].astype(np.int64)
    K = synth.kv_values(rng, (20, H, D), it)
    V = synth.kv_values(rng, (20, H, D), it)
    M = _fresh(o)
    T = M.copy()
    assert o.store(M, 2, slots, K, V) == 0
    kd, vd, err = o.store_rows(2, slots)
    assert err == 0
    Kb, Vb = K.reshape(20, -1).view(np.uint8), V.reshape(20, -1).view(np.uint8)
    for i in range(20):
        T[kd[i]:kd[i] + R] = Kb[i]
        T[vd[i]:vd[i] + R] = Vb[i]
    assert np.array_equal(M, T)
    bt = rng.integers(1, P, size=(3, 4)).astype(np.int32)
    g = synth.GatherBatch(bt, np.array([0, 2, 5], np.int32), np.array([16, 9, 5], np.int32))
    k, v, err = o.gather(M, 1, bt, g.seq_len, g.cu, g.seq_start)
    ks, vs, err2 = o.gather_rows(1, bt, g.seq_len, g.cu, g.seq_start)
    assert err == err2 == 0
    for r in range(g.total):
        assert np.array_equal(k[r], M[ks[r]:ks[r] + R]) and np.array_equal(v[r], M[vs[r]:vs[r] + R])
    src, _ = o.translate(slots[:5])
    dst, _ = o.translate(np.setdiff1d(np.arange(ps, P * ps), slots)[:5])
    sb, db, err = o.move_rows(src, dst)
    before = M.copy()
    assert err == 0 and o.move(M, src, dst) == 0
    for a, b in zip(sb, db):
        assert np.array_equal(M[b:b + R], before[a:a + R])


def pin_block_table_kf(so):
    """Prefix-only kernel-facing block table: hand-computed entries
    (tests/golden/block_table_tiny.txt), untouched entries past each prefix,
    and every entry*ps + o equal to translate's id of the same virtual slot."""
    o = _mk(so, _geom(2, 2, 8, 2, 4, 64))
    v2p = np.arange(41, dtype=np.int32) + 10
    v2p[7] = -1
    v2p[9] = 70
    rows = [r for r in _rows(os.path.join(GOLDEN, "block_table_tiny.txt"))]
    ln = np.array([int(r[0]) for r in rows], np.int32)
    virt = np.array([[int(x) for x in r[2:7]] for r in rows], np.int32)
    want = np.array([[int(x) for x in r[8:13]] for r in rows], np.int32)
    got, err = o.block_table_kf(virt, ln, v2p)
    assert err == 0 and np.array_equal(got, want), got
    for s_ in range(len(rows)):
        np_ = -(-int(ln[s_]) // 4)
        for k in range(np_):
            for off in range(4):
                slot = int(virt[s_, k]) * 4 + off
                ids, _ = o.translate(np.array([slot], np.int64), v2p)
                assert int(ids[0]) == (int(got[s_, k]) * 4 + off if got[s_, k] else int(ids[0]))
                if got[s_, k]:
                    assert int(ids[0]) == int(got[s_, k]) * 4 + off
    # errors: a virtual page past the map, a physical page past the pool, an overlong sequence
    bad, err = o.block_table_kf(np.array([[41, 9, 1]], np.int32), np.array([12], np.int32), v2p)
    assert err == oracle.E_V2P | oracle.E_ROW and list(bad[0]) == [0, 0, 44]
    _, err = o.block_table_kf(np.array([[1, 2]], np.int32), np.array([9], np.int32), v2p)
    assert err == oracle.E_TABLE


def pin_gather_kf(so):
    """Gather through a prefix-only kernel-facing block table
    (tests/golden/gather_kf_tiny.txt, hand-computed): the table build gives
    the listed entries, and every output row holds the K and V rows of the
    listed (page, offset), read from the [P, 2L, ps, H, D] reference. Then:
    on tables without tombstones the result equals the physical-page gather
    of entry / 2L; an entry off the 2L grid raises E_FORM and one past the
    pool E_ROW (rows untouched); a negative entry reads the sink row."""
    L, H, D, it, ps, P = 2, 2, 8, 2, 4, 64
    o = _mk(so, _geom(L, H, D, it, ps, P))
    R = o.sizes()["row_bytes"]
    v2p = np.arange(41, dtype=np.int32) + 10
    v2p[7] = -1
    rows = _rows(os.path.join(GOLDEN, "gather_kf_tiny.txt"))
    trows = [r for r in rows if r[0] == "T"]
    st = np.array([int(r[2]) for r in trows], np.int32)
    ln = np.array([int(r[3]) for r in trows], np.int32)
    virt = np.array([[int(x) for x in r[5:8]] for r in trows], np.int32)
    want_kf = np.array([[int(x) for x in r[9:12]] for r in trows], np.int32)
    kf, err = o.block_table_kf(virt, ln, v2p)
    assert err == 0 and np.array_equal(kf, want_kf), kf
    M = _fresh(o, seed=23)
    env = strided_ref.envelope(M, L, H, D, it, ps, P)
    g = synth.GatherBatch(kf, st, ln)
    k, v, err = o.gather_kf(M, 1, kf, ln, g.cu, st)
    rrows = [tuple(map(int, r[1:4])) for r in rows if r[0] == "R"]
    assert err == 0 and k.shape[0] == len(rrows) == g.total
    for r, page, off in rrows:
        assert np.array_equal(k[r], env[page, 2, off].reshape(-1).view(np.uint8)), (r, page, off)
        assert np.array_equal(v[r], env[page, 3, off].reshape(-1).view(np.uint8)), (r, page, off)
    ks, vs, err = o.gather_rows(1, kf, ln, g.cu, st, kernel_facing=True)
    assert err == 0
    for r, page, off in rrows:
        assert ks[r] == o.slot_row_byte(page * ps + off, 2) and vs[r] == o.slot_row_byte(page * ps + off, 3)
    # without tombstones, the same rows as the physical gather of entry / 2L
    rng = np.random.default_rng(21)
    phys = rng.integers(1, P, size=(4, 5)).astype(np.int32)
    gb = synth.GatherBatch(phys, np.array([0, 3, 7, 1], np.int32), np.array([20, 17, 9, 2], np.int32))
    for layer in range(L):
        k1, v1, e1 = o.gather_kf(M, layer, phys * (2 * L), gb.seq_len, gb.cu, gb.seq_start)
        k2, v2, e2 = o.gather(M, layer, phys, gb.seq_len, gb.cu, gb.seq_start)
        assert e1 == e2 == 0 and np.array_equal(k1, k2) and np.array_equal(v1, v2)
    # errors: off the grid (E_FORM), past the pool (E_ROW); those rows stay as they were
    for entry, bit in ((5 * 2 * L + 1, oracle.E_FORM), (P * 2 * L, oracle.E_ROW)):
        bt = np.array([[3 * 2 * L, entry]], np.int32)
        gk = synth.GatherBatch(bt, np.zeros(1, np.int32), np.array([2 * ps], np.int32))
        k, v, err = o.gather_kf(M, 0, bt, gk.seq_len, gk.cu, gk.seq_start)
        assert err == bit, (entry, err)
        assert np.array_equal(k[0], env[3, 0, 0].reshape(-1).view(np.uint8))
        assert not k[ps:].any() and not v[ps:].any()
    # a negative entry reads the sink row (page 0, offset 0) for every token
    bt = np.array([[-1]], np.int32)
    k, v, err = o.gather_kf(M, 1, bt, np.array([ps], np.int32), np.array([0, ps], np.int64))
    assert err == 0 and all(np.array_equal(k[i], env[0, 2, 0].reshape(-1).view(np.uint8)) for i in range(ps))
    assert all(np.array_equal(v[i], env[0, 3, 0].reshape(-1).view(np.uint8)) for i in range(ps))
    assert R == 32


def pin_mla(so):
    """MLA pools (one latent row per layer, blocks_per_page = L): hand-computed
    layout and ids (tests/golden/mla_tiny.txt), the id bound, the uniform-row
    gate not applying, a brute-force bijection, and store / gather / move
    against the [P, L, ps, H, D] reference."""
    g = {k: int(v) for k, v in _rows(os.path.join(GOLDEN, "mla_tiny.txt"))}
    o = _mk(so, _geom(2, 1, 16, 2, 4, 64, latent=True))
    sz = o.sizes()
    assert (sz["row_bytes"], sz["page_bytes"], sz["total"], sz["tail_pad"], sz["n_rows"], sz["last_view_end"]) == \
        (g["row_bytes"], g["page_bytes"], g["total"], g["tail_pad"], g["n_rows"], g["last_view_end"])
    for t in (0, 5, 255, -1):
        ids, err = o.translate(np.array([t], np.int64))
        assert err == 0 and int(ids[0]) == g[f"id_{t}"], (t, int(ids[0]))
    big = _mk(so, _geom(61, 1, 576, 2, 64, 1000, latent=True)).sizes()
    assert (big["page_bytes"], big["n_rows"], big["last_view_end"]) == \
        (g["big_page_bytes"], g["big_n_rows"], g["big_last_view_end"])
    assert _mk(so, _geom(61, 1, 576, 2, 64, g["big_max_pages_ok"], latent=True)).check() == "ok"
    assert _mk(so, _geom(61, 1, 576, 2, 64, g["big_max_pages_ok"] + 1, latent=True)).check() == "id_bound"
    # MLA has no V: the report admits it whatever v_head_dim says
    assert _mk(so, _geom(2, 1, 16, 2, 4, 64, Dv=128, latent=True)).check() == "ok"
    # bijection on a tiny MLA pool
    L, ps, P = 3, 4, 5
    t_ = _mk(so, _geom(L, 1, 16, 1, ps, P, anchor=32, latent=True))
    R = t_.sizes()["row_bytes"]
    ids, _ = t_.translate(np.arange(P * ps, dtype=np.int64))
    seen = sorted(t_.slot_row_byte(int(t), b) for t in range(P * ps) for b in range(L))
    assert seen == [32 + R * k for k in range(P * L * ps)]
    for t, kid in zip(range(P * ps), ids):
        assert t_.slot_row_byte(t, 1) == 32 + (int(kid) + 1 * ps) * R
    # store / gather / move against the reference
    rng = np.random.default_rng(17)
    L, H, D, it, ps, P = 4, 1, 32, 2, 8, 9
    o = _mk(so, _geom(L, H, D, it, ps, P, latent=True))
    M = _fresh(o)
    T = M.copy()
    env = strided_ref.envelope(T, L, H, D, it, ps, P, latent=True)
    for layer in range(L):
        slots = rng.permutation(np.arange(ps, P * ps))[:30].astype(np.int64)
        slots[3] = -1
        K = synth.kv_values(rng, (30, H, D), it)
        assert o.store(M, layer, slots, K, None) == 0
        strided_ref.store(env, layer, slots, K, None, latent=True)
        assert np.array_equal(M, T)
    Ka = synth.kv_values(rng, (L, 20, H, D), it)
    slots = rng.permutation(np.arange(ps, P * ps))[:20].astype(np.int64)
    assert o.store_all(M, slots, Ka, None) == 0
    for layer in range(L):
        strided_ref.store(env, layer, slots, Ka[layer], None, latent=True)
    assert np.array_equal(M, T)
    bt = rng.integers(1, P, size=(3, 4)).astype(np.int32)
    gb = synth.GatherBatch(bt, np.array([0, 3, 9], np.int32), np.array([32, 20, 12], np.int32))
    for layer in range(L):
        k, v, err = o.gather(M, layer, bt, gb.seq_len, gb.cu, gb.seq_start)
        rk, _ = strided_ref.gather(env, layer, bt, gb.seq_start, gb.seq_len, latent=True)
        assert err == 0 and v is None
        assert np.array_equal(k, rk.reshape(len(rk), -1).view(np.uint8).reshape(k.shape))
    src = slots[:6]
    dst = np.setdiff1d(np.arange(ps, P * ps), slots)[:6]
    si, _ = o.translate(src)
    di, _ = o.translate(dst)
    assert o.move(M, si, di) == 0
    strided_ref.move(env, src, dst)
    assert np.array_equal(M, T)


def pin_mla_address_mode(so):
    """MLA pools in address mode (the form the full-size checks use): store,
    gather and move name exactly the bytes their copying twins move, report
    no V row, and a move names L rows per pair, one per layer (blocks_per_page()
    returns layer_num for MLA, 实现拆解 step 2)."""
    rng = np.random.default_rng(19)
    L, H, D, it, ps, P = 4, 1, 32, 2, 8, 9
    o = _mk(so, _geom(L, H, D, it, ps, P, latent=True))
    R = o.sizes()["row_bytes"]
    M = _fresh(o)
    used = rng.permutation(np.arange(ps, P * ps))
    slots = used[:20].astype(np.int64)
    K = synth.kv_values(rng, (20, H, D), it)
    T = M.copy()
    assert o.store(M, 3, slots, K, None) == 0
    kd, vd, err = o.store_rows(3, slots)
    assert err == 0 and kd.size == 20 and np.all(vd == -1)
    Kb = K.reshape(20, -1).view(np.uint8)
    for i in range(20):
        T[kd[i]:kd[i] + R] = Kb[i]
    assert np.array_equal(M, T)
    bt = rng.integers(1, P, size=(3, 4)).astype(np.int32)
    gb = synth.GatherBatch(bt, np.array([0, 3, 9], np.int32), np.array([32, 20, 12], np.int32))
    k, v, err = o.gather(M, 2, bt, gb.seq_len, gb.cu, gb.seq_start)
    ks, vs, err2 = o.gather_rows(2, bt, gb.seq_len, gb.cu, gb.seq_start)
    assert err == err2 == 0 and v is None and np.all(vs == -1)
    for r in range(gb.total):
        assert np.array_equal(k[r], M[ks[r]:ks[r] + R])
    m = 6
    src_slots, dst_slots = used[:m], used[20:20 + m]
    src, _ = o.translate(src_slots)
    dst, _ = o.translate(dst_slots)
    # the raw routine first, into buffers twice the size it may write: it must
    # fill exactly m * L entries and leave the rest alone
    sb_raw = np.full(2 * m * L, -7, np.int64)
    db_raw = np.full(2 * m * L, -7, np.int64)
    err = o._L.ora_move_rows(ctypes.byref(o._d), src.ctypes.data, dst.ctypes.data, m, sb_raw.ctypes.data,
                             db_raw.ctypes.data)
    assert err == 0 and np.all(sb_raw[m * L:] == -7) and np.all(db_raw[m * L:] == -7)
    sb, db, err = o.move_rows(src, dst)
    assert err == 0 and sb.size == db.size == m * L
    assert np.array_equal(sb, sb_raw[:m * L]) and np.array_equal(db, db_raw[:m * L])
    # pair i, layer b names block b of the token, found by slot (not by id)
    for i in range(m):
        for b in range(L):
            assert sb[i * L + b] == o.slot_row_byte(int(src_slots[i]), b)
            assert db[i * L + b] == o.slot_row_byte(int(dst_slots[i]), b)
    before = M.copy()
    assert o.move(M, src, dst) == 0
    T = before.copy()
    for a, b in zip(sb, db):
        T[b:b + R] = before[a:a + R]
    assert np.array_equal(M, T)


def pin_swa_token_map(so):
    """Full -> SWA token mapping (tests/golden/swa_map_tiny.txt), a slot past
    the map, and translate_mapped(t) = translate(map[t]) on random maps."""
    o = _mk(so, _geom(2, 1, 16, 1, 4, 16))
    tmap = np.array([-1, 5, 6, -1, 17, 18, 19, 40, 63, 0, -1, 22], np.int64)
    rows = _rows(os.path.join(GOLDEN, "swa_map_tiny.txt"))
    slots = np.array([int(r[0]) for r in rows], np.int64)
    want = np.array([int(r[1]) for r in rows], np.int32)
    ids, err = o.translate_mapped(slots, tmap)
    assert err == 0 and np.array_equal(ids, want), ids
    ids, err = o.translate_mapped(np.array([12, 1], np.int64), tmap)
    assert err == oracle.E_V2P and list(ids) == [0, 17]
    rng = np.random.default_rng(18)
    tm = rng.integers(-1, 64, size=200).astype(np.int64)
    sl = rng.integers(-2, 200, size=500).astype(np.int64)
    v2p = rng.permutation(16).astype(np.int32)
    ids, err = o.translate_mapped(sl, tm, v2p)
    ref, err2 = o.translate(np.where(sl < 0, -1, tm[np.clip(sl, 0, 199)]), v2p)
    assert err == err2 == 0 and np.array_equal(ids, ref)


def pin_multiplier_one_collapse(so):
    """The "multiplier-1 collapse" the report's review pins with a test-only
    override (评论区精华; 风险与影响 item 1): ids translated with
    kernel_page_multiplier = 1 are physical slot ids, and the dense per-layer
    views (block b of id at view row id + b*ps) then land block b >= 1 of a
    token on rows of other tokens. With the multiplier blocks_per_page() = 2L
    the ids are translate()'s and the rows tile the pool once."""
    L, H, D, it, ps, P = 2, 2, 8, 2, 4, 8
    o = _mk(so, _geom(L, H, D, it, ps, P, 0))
    slots = np.arange(P * ps, dtype=np.int64)
    good, err = o.translate_multiplier(slots, 2 * L)
    ref, err2 = o.translate(slots)
    assert err == err2 == 0 and np.array_equal(good, ref)
    rows = [int(k) + b * ps for k in good for b in range(2 * L)]
    assert sorted(rows) == list(range(P * 2 * L * ps))  # a bijection onto the pool's rows
    bad, err = o.translate_multiplier(slots, 1)
    assert err == 0 and np.array_equal(bad, slots)  # physical slot ids
    rows1 = [int(k) + b * ps for k in bad for b in range(2 * L)]
    assert len(set(rows1)) < len(rows1)  # rows alias
    # the first token of page 1, layer 0 K (block 0), lands on page 0's first
    # token's layer 0 V row (block 1): a store of one overwrites the other
    assert int(bad[ps]) + 0 * ps == int(bad[0]) + 1 * ps
    # and every row of the multiplier-1 id space stays inside the first
    # P*ps + (2L-1)*ps rows: the upper pages of the pool are never addressed
    assert max(rows1) == P * ps - 1 + (2 * L - 1) * ps < P * 2 * L * ps - 1


PINS = [
    pin_translate_golden, pin_layout_table, pin_gates, pin_bijection, pin_store_vs_strided,
    pin_v2p_store, pin_gather_vs_strided, pin_roundtrip, pin_tail_untouched, pin_errors, pin_address_mode,
    pin_block_table_kf, pin_gather_kf, pin_mla, pin_mla_address_mode, pin_swa_token_map, pin_multiplier_one_collapse,
]


def main(argv):
    so = argv[1]
    for pin in PINS:
        try:
            pin(so)
        except AssertionError as e:  # a caught mistake
            print(f"FAILED {pin.__name__}: {e!r}"[:400])
            return 1
    print("all pins hold")
    return 0


if __name__ == "__main__":
    sys.exit(main(sys.argv))
