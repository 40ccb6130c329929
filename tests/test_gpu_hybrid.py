"""Hybrid full-attention + sliding-window model on GPU: two sub-pools packed in
one raw buffer (full pool at anchor 0, SWA pool right after it, one shared
tail pad), SWA layers addressed through a full -> SWA token map with cleared
(evicted) entries, checked against the oracle on the whole buffer."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import gather_translate_kv_gb300 as gt
import oracle
import synth
from gpu_util import as_rows, assert_bytes_equal, dev_bits, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gather_translate_kv_gb300 import build

    build.build()
    oracle.build()


def test_translate_mapped_matches_oracle():
    shape = synth.SHAPES[4].scaled(64)
    g = oracle.Geometry(shape.layer_num, shape.head_num, shape.head_dim, shape.itemsize, shape.page_size,
                        shape.num_pages)
    o = oracle.Oracle(g)
    raw = torch.empty(o.raw_bytes(), dtype=torch.uint8, device="cuda")
    pool = gt.kv_pool_create(gt.make_desc(shape.layer_num, shape.head_num, shape.head_dim, shape.itemsize,
                                          shape.page_size, shape.num_pages), raw)
    rng = np.random.default_rng(31)
    n_full = 5000
    tmap = rng.integers(-1, shape.num_pages * shape.page_size, size=n_full).astype(np.int64)
    slots = rng.integers(-2, n_full + 40, size=3000).astype(np.int64)  # some past the map
    v2p = rng.permutation(shape.num_pages).astype(np.int32)
    v2p[5] = -1
    ids_ref, err = o.translate_mapped(slots, tmap, v2p)
    ids = torch.empty(slots.size, dtype=torch.int32, device="cuda")
    gt.kv_translate_mapped(pool, to_dev(slots), ids, to_dev(tmap), to_dev(v2p))
    assert err == oracle.E_V2P
    assert gt.kv_pool_last_error(pool) == dev_bits(err)
    assert np.array_equal(ids.cpu().numpy(), ids_ref)
    gt.kv_pool_destroy(pool)


def test_full_and_swa_subpools_in_one_buffer():
    Lf, Ls, H, D, it, ps = 3, 2, 2, 64, 2, 16
    Pf, Ps = 40, 12
    gf = oracle.Geometry(Lf, H, D, it, ps, Pf, 0)
    of = oracle.Oracle(gf)
    anchor_s = (of.sizes()["total"] + 255) // 256 * 256  # the SWA pool right after the full pool's envelopes
    gs = oracle.Geometry(Ls, H, D, it, ps, Ps, anchor_s)
    osw = oracle.Oracle(gs)
    R = of.sizes()["row_bytes"]
    # UnifiedKVPool.__init__: one buffer, total bytes + the largest tail pad of its sub-pools
    nbytes = anchor_s + osw.sizes()["total"] + max(of.sizes()["tail_pad"], osw.sizes()["tail_pad"])
    raw = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    synth.fill_sentinel_torch(raw, 77)
    M = synth.sentinel_bytes(77, 0, nbytes)
    M0 = M.copy()
    pf = gt.kv_pool_create(gt.make_desc(Lf, H, D, it, ps, Pf, 0), raw, nbytes)
    psw = gt.kv_pool_create(gt.make_desc(Ls, H, D, it, ps, Ps, anchor_s), raw, nbytes)

    rng = np.random.default_rng(32)
    # 3 sequences of 60 tokens in the full pool (4 pages each); the SWA pool
    # keeps each sequence's last 2 pages (window 32 tokens), older tokens evicted
    pages_f = (1 + rng.permutation(Pf - 1)[:12]).reshape(3, 4).astype(np.int32)
    pages_s = (1 + rng.permutation(Ps - 1)[:6]).reshape(3, 2).astype(np.int32)
    n_tok = 60
    full_slots = np.concatenate([pages_f[s][np.arange(n_tok) // ps] * ps + np.arange(n_tok) % ps
                                 for s in range(3)]).astype(np.int64)
    tmap = np.full(Pf * ps, -1, np.int64)
    swa_of_token = []
    for s in range(3):
        for j in range(n_tok):
            k = j // ps
            t_full = int(pages_f[s][k]) * ps + j % ps
            if k >= 2:  # in the window: the SWA pool's page 0/1 of this sequence
                sw = int(pages_s[s][k - 2]) * ps + j % ps
                tmap[t_full] = sw
            swa_of_token.append(tmap[t_full])
    swa_slots = np.array(swa_of_token, np.int64)

    ids_f = torch.empty(full_slots.size, dtype=torch.int32, device="cuda")
    ids_s = torch.empty(full_slots.size, dtype=torch.int32, device="cuda")
    gt.kv_translate(pf, to_dev(full_slots), ids_f)
    gt.kv_translate_mapped(psw, to_dev(full_slots), ids_s, to_dev(tmap))
    ref_s, err = osw.translate_mapped(full_slots, tmap)
    assert err == 0 and np.array_equal(ids_s.cpu().numpy(), ref_s)
    tomb = {}
    for layer in range(max(Lf, Ls)):
        K = synth.kv_values(rng, (full_slots.size, H, D), it)
        V = synth.kv_values(rng, (full_slots.size, H, D), it)
        if layer < Lf:
            assert of.store(M, layer, full_slots, K, V) == 0
            gt.kv_store_layer(pf, layer, ids_f, to_dev(K), to_dev(V))
        if layer < Ls:
            assert osw.store(M, layer, swa_slots, K, V) == 0
            gt.kv_store_layer(psw, layer, ids_s, to_dev(K), to_dev(V))
            ev = np.nonzero(swa_slots < 0)[0]
            tomb.setdefault(2 * layer, []).extend(as_rows(K, R)[ev])
            tomb.setdefault(2 * layer + 1, []).extend(as_rows(V, R)[ev])
    assert gt.kv_pool_last_error(pf) == 0 and gt.kv_pool_last_error(psw) == 0

    got = raw.cpu().numpy()
    mask = np.ones(nbytes, bool)
    sinks_s = [osw.slot_row_byte(0, b) for b in range(2 * Ls)]
    for sb in sinks_s:
        mask[sb:sb + R] = False
    assert_bytes_equal(got[mask], M[mask], "hybrid buffer (outside the sink rows)")
    for b, sb in enumerate(sinks_s):  # evicted tokens were written to the SWA sink
        row = got[sb:sb + R].view(np.uint32)
        ok = row == M0[sb:sb + R].view(np.uint32)
        for t in tomb.get(b, []):
            ok |= row == np.ascontiguousarray(t).view(np.uint32)
        assert ok.all()

    # full layer: the whole context; SWA layer: the 32-token window, through each pool's own table
    gfb = synth.GatherBatch(pages_f, np.zeros(3, np.int32), np.full(3, n_tok, np.int32))
    gsb = synth.GatherBatch(pages_s, np.zeros(3, np.int32), np.full(3, n_tok - 2 * ps, np.int32))
    for pool, o, gb, layer in ((pf, of, gfb, Lf - 1), (psw, osw, gsb, Ls - 1)):
        ok_, ov_, err = o.gather(M, layer, gb.block_table, gb.seq_len, gb.cu, gb.seq_start)
        dk = torch.empty((gb.total, R), dtype=torch.uint8, device="cuda")
        dv = torch.empty_like(dk)
        gt.kv_gather_layer(pool, layer, to_dev(gb.block_table), to_dev(gb.seq_len), to_dev(gb.cu), dk, dv)
        assert err == 0 and gt.kv_pool_last_error(pool) == 0
        assert_bytes_equal(dk.cpu().numpy(), ok_, "hybrid gather K", R)
        assert_bytes_equal(dv.cpu().numpy(), ov_, "hybrid gather V", R)
    # layer 0 was stored into both pools with the same rows: the SWA window of
    # each sequence equals the full pool's tokens [32, 60), read on the GPU
    win = synth.GatherBatch(pages_f, np.full(3, 2 * ps, np.int32), np.full(3, n_tok, np.int32))
    fk = torch.empty((win.total, R), dtype=torch.uint8, device="cuda")
    fv = torch.empty_like(fk)
    gt.kv_gather_layer(pf, 0, to_dev(win.block_table), to_dev(win.seq_len), to_dev(win.cu), fk, fv,
                       to_dev(win.seq_start))
    sk = torch.empty((gsb.total, R), dtype=torch.uint8, device="cuda")
    sv = torch.empty_like(sk)
    gt.kv_gather_layer(psw, 0, to_dev(gsb.block_table), to_dev(gsb.seq_len), to_dev(gsb.cu), sk, sv)
    assert torch.equal(fk, sk) and torch.equal(fv, sv)
    assert gt.kv_pool_last_error(pf) == 0 and gt.kv_pool_last_error(psw) == 0
    gt.kv_pool_destroy(pf)
    gt.kv_pool_destroy(psw)
