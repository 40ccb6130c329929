"""GPU parity of the gathers that read a kernel-facing block table directly
(kv_gather_layer_kf, kv_gather_plan_kf + kv_gather_layer_planned_kf), composed
with the prefix-only table build (kv_translate_block_table), against the
oracle's composition (block_table_kf, then gather_kf).

The read path of the prhub report on sglang PR #34602 (关联脉络, PR #35247)
builds the kernel-facing page table once per batch, translating only the
prefix a sequence uses, and reads the pool through it.
"""
from __future__ import annotations

import os

import numpy as np
import pytest
import torch

import gather_translate_kv_gb300 as gt
import oracle
import synth
from gpu_util import PoolPair, assert_bytes_equal, dev_bits, to_dev

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
S = synth.Shape


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gather_translate_kv_gb300 import build

    build.build()
    oracle.build()


def _golden_rows():
    out = []
    with open(os.path.join(GOLDEN, "gather_kf_tiny.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                out.append(line.split())
    return out


def _gpu_gathers(pp, layer, kf_d, ln, cu, st, rows, latent, plan_d=None):
    """(k, v) from the table-order and the planned kernel-facing gathers, each
    into outputs pre-filled with a marker (rows no token covers must keep it)."""
    R = pp.R
    outs = []
    for planned in (False, True):
        dk = torch.full((rows, R), 0x5A, dtype=torch.uint8, device="cuda")
        dv = None if latent else torch.full((rows, R), 0x5A, dtype=torch.uint8, device="cuda")
        if planned:
            gt.kv_gather_layer_planned_kf(pp.pool, layer, plan_d, kf_d, to_dev(ln), to_dev(cu), dk, dv,
                                          None if st is None else to_dev(st))
        else:
            gt.kv_gather_layer_kf(pp.pool, layer, kf_d, to_dev(ln), to_dev(cu), dk, dv,
                                  None if st is None else to_dev(st))
        outs.append((dk.cpu().numpy(), None if dv is None else dv.cpu().numpy()))
    return outs


def test_kf_gather_golden():
    """The hand-computed case of tests/golden/gather_kf_tiny.txt: the table the
    GPU builds, and every output row of the GPU gathers (table order and
    planned), equal the golden entries and the rows of the listed (page,
    offset), and the oracle's composition."""
    shape = synth.SHAPES[1]  # L=2, H=2, D=8, bf16, ps=4, P=64
    pp = PoolPair(shape)
    o, R, ps = pp.o, pp.R, shape.page_size
    rows = _golden_rows()
    trows = [r for r in rows if r[0] == "T"]
    st = np.array([int(r[2]) for r in trows], np.int32)
    ln = np.array([int(r[3]) for r in trows], np.int32)
    virt = np.array([[int(x) for x in r[5:8]] for r in trows], np.int32)
    want_kf = np.array([[int(x) for x in r[9:12]] for r in trows], np.int32)
    v2p = np.arange(41, dtype=np.int32) + 10
    v2p[7] = -1
    kf_d = torch.full(virt.shape, -7, dtype=torch.int32, device="cuda")
    gt.kv_translate_block_table(pp.pool, to_dev(virt), to_dev(ln), to_dev(v2p), kf_d)
    assert pp.last_error() == 0
    assert np.array_equal(kf_d.cpu().numpy(), want_kf)
    g = synth.GatherBatch(want_kf, st, ln)
    plan_d = gt.kv_gather_plan_kf(pp.pool, kf_d, to_dev(ln), to_dev(st))
    assert pp.last_error() == 0
    assert int(plan_d.cpu()[3]) & 2, "a kernel-facing plan records its form"
    ok, ov, err = o.gather_kf(pp.M, 1, want_kf, ln, g.cu, st)
    assert err == 0
    for dk, dv in _gpu_gathers(pp, 1, kf_d, ln, g.cu, st, g.total, False, plan_d):
        assert pp.last_error() == 0
        assert_bytes_equal(dk, ok, "golden kf gather K", R)
        assert_bytes_equal(dv, ov, "golden kf gather V", R)
        for out_row, page, off in ([int(x) for x in row[1:4]] for row in rows if row[0] == "R"):
            kb = o.slot_row_byte(page * ps + off, 2)
            vb = o.slot_row_byte(page * ps + off, 3)
            assert np.array_equal(dk[out_row], pp.M[kb:kb + R]), out_row
            assert np.array_equal(dv[out_row], pp.M[vb:vb + R]), out_row
    pp.close()


KF_SHAPES = [
    (synth.SHAPES[1], 0, False),                      # R=32, ps=4
    (synth.SHAPES[2].scaled(40), 0, False),           # R=2048, ps=16, L=32
    (synth.SHAPES[4].scaled(150), 32, False),         # R=512 fp8, ps=32, L=24
    (synth.SHAPES[5].scaled(20), 0, False),           # R=64 fp8, ps=256, L=80
    (S(0, "odd-rows", 3, 3, 16, 1, 3, 40), 16, False),  # R=48 (general path), ps=3
    (S(0, "mla-r1152", 6, 1, 576, 2, 64, 10), 0, True),  # MLA latent rows
    (S(0, "mla-r512", 5, 1, 256, 2, 16, 30), 32, True),
    (S(0, "mla-one-layer", 1, 1, 2048, 2, 16, 40), 0, True),  # 1 block per page: entries equal pages
]


@pytest.mark.parametrize("shape,anchor,latent", KF_SHAPES,
                         ids=[f"{s.name}-R{s.row_bytes}-ps{s.page_size}" for s, _, _ in KF_SHAPES])
def test_kf_gather_matches_oracle(shape, anchor, latent):
    """Virtual tables with tombstoned pages (map entries -1 and -1 table
    entries), shared pages, windows starting mid-page and empty sequences:
    the GPU table build then both kernel-facing gathers equal the oracle's
    block_table_kf then gather_kf, on the first and last layer."""
    rng = np.random.default_rng(900 + shape.row_bytes + shape.page_size)
    pp = PoolPair(shape, anchor, latent=latent)
    o, R, L, ps, P = pp.o, pp.R, shape.layer_num, shape.page_size, shape.num_pages
    S_, maxp = 29, min(7, P - 1)
    V = P + 3
    v2p = np.zeros(V, np.int32)
    v2p[:P] = rng.permutation(P)
    v2p[P:] = rng.integers(1, P, size=V - P)
    v2p[rng.choice(V, size=max(1, V // 10), replace=False)] = -1
    hot = rng.integers(0, V, size=4)
    virt = np.where(rng.random((S_, maxp)) < 0.6, rng.choice(hot, size=(S_, maxp)),
                    rng.integers(0, V, size=(S_, maxp))).astype(np.int32)
    virt[rng.random((S_, maxp)) < 0.05] = -1
    ln = rng.integers(0, maxp * ps + 1, size=S_).astype(np.int32)
    ln[0], ln[4] = maxp * ps, 0
    st = np.minimum(rng.integers(0, 2 * ps + 1, size=S_), ln).astype(np.int32)
    kf_ref, err = o.block_table_kf(virt, ln, v2p, out=np.full(virt.shape, -7, np.int32))
    assert err == 0
    kf_d = torch.full(virt.shape, -7, dtype=torch.int32, device="cuda")
    gt.kv_translate_block_table(pp.pool, to_dev(virt), to_dev(ln), to_dev(v2p), kf_d)
    assert pp.last_error() == 0
    assert np.array_equal(kf_d.cpu().numpy(), kf_ref)
    g = synth.GatherBatch(kf_ref, st, ln)
    plan_d = gt.kv_gather_plan_kf(pp.pool, kf_d, to_dev(ln), to_dev(st))
    assert pp.last_error() == 0
    for layer in sorted({0, L - 1}):
        rows = g.total + 3
        ok = np.full((rows, R), 0x5A, np.uint8)
        ov = None if latent else np.full((rows, R), 0x5A, np.uint8)
        ok, ov, err = o.gather_kf(pp.M, layer, kf_ref, ln, g.cu, st, rows, ok, ov)
        assert err == 0
        for how, (dk, dv) in zip(("table", "planned"), _gpu_gathers(pp, layer, kf_d, ln, g.cu, st, rows, latent,
                                                                   plan_d)):
            assert pp.last_error() == 0
            assert_bytes_equal(dk, ok, f"kf gather K ({how}) layer {layer}", R)
            if not latent:
                assert_bytes_equal(dv, ov, f"kf gather V ({how}) layer {layer}", R)
    # in place: past each sequence's prefix the table keeps its virtual pages
    # (off the 2L grid unless 2L divides them); the gathers never read there,
    # so they raise no bit and give the same rows
    ip_d = to_dev(virt.copy())
    gt.kv_translate_block_table(pp.pool, ip_d, to_dev(ln), to_dev(v2p))
    assert pp.last_error() == 0
    ip = ip_d.cpu().numpy()
    pre = np.arange(maxp)[None, :] < -(-ln[:, None] // ps)
    assert np.array_equal(ip[pre], kf_ref[pre]) and np.array_equal(ip[~pre], virt[~pre])
    plan_ip = gt.kv_gather_plan_kf(pp.pool, ip_d, to_dev(ln), to_dev(st))
    assert pp.last_error() == 0
    rows = g.total + 3
    ok = np.full((rows, R), 0x5A, np.uint8)
    ov = None if latent else np.full((rows, R), 0x5A, np.uint8)
    ok, ov, err = o.gather_kf(pp.M, L - 1, kf_ref, ln, g.cu, st, rows, ok, ov)
    for how, (dk, dv) in zip(("table", "planned"), _gpu_gathers(pp, L - 1, ip_d, ln, g.cu, st, rows, latent,
                                                               plan_ip)):
        assert pp.last_error() == 0
        assert_bytes_equal(dk, ok, f"kf gather K over an in-place table ({how})", R)
        if not latent:
            assert_bytes_equal(dv, ov, f"kf gather V over an in-place table ({how})", R)
    pp.close()


def test_kf_gather_errors_match_oracle():
    """Entries off the 2L grid (KV_DEV_ERR_FORM) and past the pool
    (KV_DEV_ERR_ROW) are skipped with the oracle's error bits and leave their
    output rows untouched; a negative entry reads the sink row; a plan of the
    other table form is refused on the device and writes nothing."""
    shape = S(0, "kf-err", 3, 2, 64, 2, 8, 30)  # R=256, L=3 (2L=6), ps=8
    pp = PoolPair(shape)
    o, R, L, ps, P = pp.o, pp.R, shape.layer_num, shape.page_size, shape.num_pages
    B = 2 * L
    kf = np.array([[5 * B, 5 * B + 1, 7 * B],       # an entry off the grid
                   [P * B, 2 * B, 3 * B],           # an entry past the pool
                   [-1, 4 * B, (P - 1) * B],        # a negative entry: the sink row
                   [P * B + 3, 6 * B, 0]], np.int32)  # past the pool and off the grid: a row error
    ln = np.full(4, 3 * ps, np.int32)
    st = np.array([0, 2, 1, 0], np.int32)
    g = synth.GatherBatch(kf, st, ln)
    ok, ov, err = o.gather_kf(pp.M, 2, kf, ln, g.cu, st, g.total, np.full((g.total, R), 0x5A, np.uint8),
                              np.full((g.total, R), 0x5A, np.uint8))
    assert err == oracle.E_FORM | oracle.E_ROW
    kf_d = to_dev(kf)
    dk = torch.full((g.total, R), 0x5A, dtype=torch.uint8, device="cuda")
    dv = torch.full((g.total, R), 0x5A, dtype=torch.uint8, device="cuda")
    gt.kv_gather_layer_kf(pp.pool, 2, kf_d, to_dev(ln), to_dev(g.cu), dk, dv, to_dev(st))
    assert pp.last_error() == dev_bits(err)
    assert_bytes_equal(dk.cpu().numpy(), ok, "kf gather K with bad entries", R)
    assert_bytes_equal(dv.cpu().numpy(), ov, "kf gather V with bad entries", R)
    plan_d = gt.kv_gather_plan_kf(pp.pool, kf_d, to_dev(ln), to_dev(st))
    assert pp.last_error() == dev_bits(err)  # the plan leaves the bad entries out, with the same bits
    dk.fill_(0x5A)
    dv.fill_(0x5A)
    gt.kv_gather_layer_planned_kf(pp.pool, 2, plan_d, kf_d, to_dev(ln), to_dev(g.cu), dk, dv, to_dev(st))
    assert pp.last_error() == dev_bits(err)
    assert_bytes_equal(dk.cpu().numpy(), ok, "planned kf gather K with bad entries", R)
    assert_bytes_equal(dv.cpu().numpy(), ov, "planned kf gather V with bad entries", R)
    # plans of the other form: nothing written, KV_DEV_ERR_TABLE
    phys = np.maximum(kf, 0) // B % P
    plan_phys = gt.kv_gather_plan(pp.pool, to_dev(phys.astype(np.int32)), to_dev(ln), to_dev(st))
    assert pp.last_error() == 0
    dk.fill_(0x33)
    gt.kv_gather_layer_planned_kf(pp.pool, 2, plan_phys, kf_d, to_dev(ln), to_dev(g.cu), dk, dv, to_dev(st))
    assert pp.last_error() == gt.KV_DEV_ERR_TABLE and bool((dk == 0x33).all())
    gt.kv_gather_layer_planned(pp.pool, 2, plan_d, to_dev(phys.astype(np.int32)), to_dev(ln), to_dev(g.cu), dk,
                               dv, to_dev(st))
    assert pp.last_error() == gt.KV_DEV_ERR_TABLE and bool((dk == 0x33).all())
    pp.close()


def test_kf_read_path_captures_in_a_cuda_graph():
    """Table build -> kernel-facing plan -> both kernel-facing gathers,
    captured once and replayed on new virtual tables, page maps and windows."""
    shape = S(0, "kf-graph", 4, 2, 64, 2, 8, 40)  # R=256, L=4, ps=8
    pp = PoolPair(shape)
    o, R, L, ps, P = pp.o, pp.R, shape.layer_num, shape.page_size, shape.num_pages
    S_, maxp = 5, 6
    z = lambda shp, dt: torch.zeros(shp, dtype=dt, device="cuda")  # noqa: E731
    virt_d, ln_d, st_d, v2p_d = z((S_, maxp), torch.int32), z(S_, torch.int32), z(S_, torch.int32), z(P, torch.int32)
    cu_d = z(S_ + 1, torch.int64)
    kf_d = z((S_, maxp), torch.int32)
    rows = S_ * maxp * ps
    outs = [z((rows, R), torch.uint8) for _ in range(4)]
    plan_d = z(gt.kv_gather_plan_bytes(pp.pool, S_, maxp) // 4, torch.int32)

    def step():
        gt.kv_translate_block_table(pp.pool, virt_d, ln_d, v2p_d, out_bt=kf_d)
        gt.kv_gather_plan_kf(pp.pool, kf_d, ln_d, st_d, plan=plan_d)
        gt.kv_gather_layer_kf(pp.pool, 3, kf_d, ln_d, cu_d, outs[0], outs[1], st_d)
        gt.kv_gather_layer_planned_kf(pp.pool, 3, plan_d, kf_d, ln_d, cu_d, outs[2], outs[3], st_d)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # warm-up outside capture (all zero: empty sequences)
        step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    assert pp.last_error() == 0
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    rng = np.random.default_rng(31)
    for rep in range(2):
        v2p = rng.permutation(P).astype(np.int32)
        v2p[rng.choice(P, size=3, replace=False)] = -1
        virt = rng.integers(0, P, size=(S_, maxp)).astype(np.int32)
        ln = rng.integers(1, maxp * ps + 1, size=S_).astype(np.int32)
        st = np.minimum(rng.integers(0, ps + 1, size=S_), ln).astype(np.int32)
        g = synth.GatherBatch(virt, st, ln)
        for d, h in ((virt_d, virt), (ln_d, ln), (st_d, st), (v2p_d, v2p), (cu_d, g.cu)):
            d.copy_(to_dev(h))
        for t in outs:
            t.fill_(0x5A)
        graph.replay()
        torch.cuda.synchronize()
        assert pp.last_error() == 0
        kf_ref, err = o.block_table_kf(virt, ln, v2p, out=virt.copy())
        assert err == 0
        got_kf = kf_d.cpu().numpy()
        np_ = -(-ln // ps)
        mask = np.arange(maxp)[None, :] < np_[:, None]
        assert np.array_equal(got_kf[mask], kf_ref[mask])
        ok, ov, err = o.gather_kf(pp.M, 3, kf_ref, ln, g.cu, st, rows, np.full((rows, R), 0x5A, np.uint8),
                                  np.full((rows, R), 0x5A, np.uint8))
        assert err == 0
        for i, what in ((0, "table"), (2, "planned")):
            assert_bytes_equal(outs[i].cpu().numpy(), ok, f"graph kf gather K ({what})", R)
            assert_bytes_equal(outs[i + 1].cpu().numpy(), ov, f"graph kf gather V ({what})", R)
    pp.close()
