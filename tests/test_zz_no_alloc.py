"""kv_gather_plan_noalloc against kv_gather_plan, through the C ABI.

kv_gather_plan_noalloc is for callers that cannot allocate device memory (a
framework's allocator owns it, or allocation must stay out of a serving loop):
its sort counters live in a fixed array inside the library instead of the
caller's plan buffer. The plan it writes must be kv_gather_plan's, up to the
order of entries within one page (atomics decide that order in both), and
gathers through either plan must write identical bytes. The array keeps the
last call's contents, so the check runs on two different tables in a row.

This file is collected last on purpose: a run that stops at its first failure
has then already run every other test."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import gather_translate_kv_gb300 as gt
import synth

pytestmark = pytest.mark.gpu

HEADER = 4  # entries, n_seqs, max_pages, page-major flag


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gather_translate_kv_gb300 import build

    build.build()


def _dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _noalloc_plan(pool, bt, ln, st, nbytes) -> torch.Tensor:
    plan = torch.full((nbytes // 4,), -7, dtype=torch.int32, device="cuda")  # nothing left from a clean buffer
    rc = gt.lib().kv_gather_plan_noalloc(
        pool.handle, gt._dev(bt, "block_table", torch.int32), bt.shape[0], bt.shape[1],
        gt._dev(st, "seq_start", torch.int32), gt._dev(ln, "seq_len", torch.int32),
        gt._dev(plan, "plan", torch.int32), nbytes, None)
    assert rc == gt.KV_OK, gt.kv_status_string(rc)
    return plan


def _assert_same_plan(ref: np.ndarray, got: np.ndarray, bt: np.ndarray, P: int):
    # header and per-page end offsets are fully determined
    assert np.array_equal(got[:HEADER + P + 1], ref[:HEADER + P + 1])
    n = int(ref[0])
    ea, eb = ref[HEADER + P + 1:][:n], got[HEADER + P + 1:][:n]
    pa, pb = np.maximum(bt.reshape(-1)[ea], 0), np.maximum(bt.reshape(-1)[eb], 0)
    assert np.array_equal(pa, pb), "entries are grouped into different pages"
    assert np.all(np.diff(pb) >= 0)
    # within one page the order is free: compare each page's set of entries
    assert np.array_equal(ea[np.lexsort((ea, pa))], eb[np.lexsort((eb, pb))])


def _tables(P: int, ps: int):
    rng = np.random.default_rng(4242)
    # first call: 48 sequences over a few heavily shared pages (page-major order)
    S1, m1 = 48, 24
    bt1 = rng.integers(1, 40, size=(S1, m1)).astype(np.int32)
    bt1[2, 3] = -1  # tombstone: read through the page-0 sink
    ln1 = rng.integers(0, m1 * ps + 1, size=S1).astype(np.int32)
    ln1[0] = m1 * ps
    st1 = np.minimum(rng.integers(0, 3 * ps, size=S1), ln1).astype(np.int32)
    # second call: another shape and mostly distinct pages (the table's order)
    S2, m2 = 20, 9
    bt2 = (1 + rng.permutation(P - 1)[: S2 * m2]).reshape(S2, m2).astype(np.int32)
    ln2 = rng.integers(1, m2 * ps + 1, size=S2).astype(np.int32)
    st2 = np.zeros(S2, np.int32)
    return [(bt1, ln1, st1, 1), (bt2, ln2, st2, 0)]


def test_noalloc_plan_matches_kv_gather_plan_on_two_calls_in_a_row():
    L, H, D, it, ps, P = 4, 8, 128, 2, 16, 512
    pool = gt.kv_pool_create(gt.make_desc(L, H, D, it, ps, P))
    R = pool.row_bytes
    # deterministic, distinct pool contents: every layer stores its own rows
    all_slots = np.arange(P * ps, dtype=np.int64)
    ids = torch.empty(all_slots.size, dtype=torch.int32, device="cuda")
    gt.kv_translate(pool, _dev(all_slots), ids)
    for layer in range(L):
        k = torch.from_numpy(synth.sentinel_bytes(900 + layer, 0, all_slots.size * R)).cuda()
        v = torch.from_numpy(synth.sentinel_bytes(950 + layer, 0, all_slots.size * R)).cuda()
        gt.kv_store_layer(pool, layer, ids, k.view(all_slots.size, H, D * it), v.view(all_slots.size, H, D * it))
    assert gt.kv_pool_last_error(pool) == 0

    for call, (bt, ln, st, mode) in enumerate(_tables(P, ps)):
        nbytes = gt.kv_gather_plan_bytes(pool, *bt.shape)
        ref = gt.kv_gather_plan(pool, _dev(bt), _dev(ln), _dev(st))
        got = _noalloc_plan(pool, _dev(bt), _dev(ln), _dev(st), nbytes)
        torch.cuda.synchronize()
        assert gt.kv_pool_last_error(pool) == 0
        r, g = ref.cpu().numpy(), got.cpu().numpy()
        assert int(g[3]) == mode, f"call {call}: page-major flag"
        _assert_same_plan(r, g, bt, P)

        cu = np.zeros(bt.shape[0] + 1, np.int64)
        cu[1:] = np.cumsum(np.maximum(ln - st, 0))
        rows = int(cu[-1])
        for layer in (0, L - 1):
            outs = []
            for plan in (ref, got):
                dk = torch.full((rows, R), 0x5A, dtype=torch.uint8, device="cuda")
                dv = torch.full((rows, R), 0xA5, dtype=torch.uint8, device="cuda")
                gt.kv_gather_layer_planned(pool, layer, plan, _dev(bt), _dev(ln), _dev(cu), dk, dv, _dev(st))
                outs.append((dk, dv))
            assert gt.kv_pool_last_error(pool) == 0
            assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1]), \
                f"call {call}, layer {layer}: gathers through the two plans differ"
    gt.kv_pool_destroy(pool)


def test_noalloc_plan_limit_and_argument_errors():
    # the largest pool the fixed array serves, and one page more
    ok = gt.kv_pool_create(gt.make_desc(1, 1, 8, 2, 1, 65536))
    big = gt.kv_pool_create(gt.make_desc(1, 1, 8, 2, 1, 65537))
    bt = _dev(np.array([[65535, 0, 7]], np.int32))
    ln = _dev(np.array([3], np.int32))
    nbytes = gt.kv_gather_plan_bytes(ok, 1, 3)
    got = _noalloc_plan(ok, bt, ln, None, nbytes)
    ref = gt.kv_gather_plan(ok, bt, ln)
    _assert_same_plan(ref.cpu().numpy(), got.cpu().numpy(), np.array([[65535, 0, 7]], np.int32), 65536)

    plan = torch.zeros(gt.kv_gather_plan_bytes(big, 1, 3) // 4, dtype=torch.int32, device="cuda")
    with pytest.raises(gt.KVError) as e:
        gt.kv_gather_plan_noalloc(big, bt, ln, plan)
    assert e.value.name == "KV_ERR_CAPACITY"
    assert gt.kv_status_string(-8) == "KV_ERR_CAPACITY"
    assert bool((plan == 0).all()), "a rejected call must enqueue nothing"
    short = torch.zeros(nbytes // 4 - 1, dtype=torch.int32, device="cuda")
    with pytest.raises(gt.KVError) as e:
        gt.kv_gather_plan_noalloc(ok, bt, ln, short)
    assert e.value.name == "KV_ERR_INVALID"
    assert gt.kv_pool_last_error(ok) == 0 and gt.kv_pool_last_error(big) == 0
    gt.kv_pool_destroy(ok)
    gt.kv_pool_destroy(big)
