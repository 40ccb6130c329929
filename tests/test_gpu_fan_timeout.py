"""The bounded waits of the bulk-copy kernels, made to run out on purpose.

The fan-out form of kv_gather_layer_planned and kv_gather_layer, and the
bulk-copy form of kv_move, stage rows in shared memory with bulk copies whose
completion they count on an mbarrier, polling at most a fixed number of times
(about a second). A build with GTKV_TEST_EXTRA_TX=16 makes every such barrier
expect 16 bytes more than its loads deliver, so the loads land but the barrier
never completes: every block must give up after its bounded waits, raise
KV_DEV_ERR_TIMEOUT, write none of its rows and return, leaving the context
usable. Nothing faults, traps or hangs; the library itself is never built
with that flag.
"""
from __future__ import annotations

import ctypes
import os
import time

import pytest
import torch

import gather_translate_kv_gb300 as gt
from gather_translate_kv_gb300 import build

pytestmark = pytest.mark.gpu

VARIANT_DIR = os.path.join(build.BUILD, "fan_timeout_test")
VARIANT_LIB = os.path.join(VARIANT_DIR, "libgtkv_fan_timeout_test.so")


@pytest.fixture(scope="module")
def variant():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    path = build.build(force=True, extra_flags=["-DGTKV_TEST_EXTRA_TX=16"], lib=VARIANT_LIB,
                       build_dir=VARIANT_DIR)
    return gt.load(path)


def _ok(rc):
    assert rc == gt.KV_OK, gt.STATUS.get(rc, rc)


def test_fan_gather_wait_runs_out_cleanly(variant):
    L = variant
    torch.cuda.init()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    # L=2, H=2, D=64 bf16 (R=256), ps=8, 4 pages; 2 sequences x 2 entries >= 4 pages: the fan-out form
    desc = gt.make_desc(2, 2, 64, 2, 8, 4)
    total, pad = ctypes.c_int64(), ctypes.c_int64()
    _ok(L.kv_pool_required_bytes(ctypes.byref(desc), ctypes.byref(total), ctypes.byref(pad)))
    nbytes = total.value + pad.value  # anchor 0
    raw = torch.randint(0, 256, (nbytes,), dtype=torch.uint8, device="cuda")
    pool = ctypes.c_void_p()
    _ok(L.kv_pool_create(ctypes.byref(desc), ctypes.c_void_p(raw.data_ptr()), nbytes, ctypes.byref(pool)))
    try:
        R, ps = 256, 8
        bt = torch.tensor([[1, 2], [3, 1]], dtype=torch.int32, device="cuda")
        ln = torch.full((2,), 2 * ps, dtype=torch.int32, device="cuda")
        cu = torch.tensor([0, 2 * ps, 4 * ps], dtype=torch.int64, device="cuda")
        need = ctypes.c_int64()
        _ok(L.kv_gather_plan_bytes(pool, 2, 2, ctypes.byref(need)))
        plan = torch.zeros(need.value // 4, dtype=torch.int32, device="cuda")
        p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
        _ok(L.kv_gather_plan(pool, p(bt), 2, 2, None, p(ln), p(plan), need.value, stream))
        out_k = torch.full((4 * ps, R), 0x5A, dtype=torch.uint8, device="cuda")
        out_v = torch.full((4 * ps, R), 0x5A, dtype=torch.uint8, device="cuda")
        err = ctypes.c_int32()
        _ok(L.kv_pool_last_error(pool, stream, ctypes.byref(err)))
        assert err.value == 0
        t0 = time.time()
        _ok(L.kv_gather_layer_planned(pool, 1, p(plan), need.value, p(bt), 2, 2, None, p(ln), p(cu), p(out_k),
                                      p(out_v), 4 * ps, stream))
        torch.cuda.synchronize()
        waited = time.time() - t0
        _ok(L.kv_pool_last_error(pool, stream, ctypes.byref(err)))
        assert err.value == gt.KV_DEV_ERR_TIMEOUT
        assert bool((out_k == 0x5A).all()) and bool((out_v == 0x5A).all())  # no block wrote a row
        assert waited < 60
        # the gather without a plan (table order, one entry per block) takes the same wait
        _ok(L.kv_gather_layer(pool, 0, p(bt), 2, 2, None, p(ln), p(cu), p(out_k), p(out_v), 4 * ps, stream))
        torch.cuda.synchronize()
        _ok(L.kv_pool_last_error(pool, stream, ctypes.byref(err)))
        assert err.value == gt.KV_DEV_ERR_TIMEOUT
        assert bool((out_k == 0x5A).all()) and bool((out_v == 0x5A).all())
        # the move of 1 KiB pairs (4 rows of 256 bytes) takes its bulk-copy form: no row moves
        before = raw.clone()
        src = torch.tensor([1 * 32 + 3, 2 * 32 + 5], dtype=torch.int32, device="cuda")
        dst = torch.tensor([3 * 32 + 3, 1 * 32 + 7], dtype=torch.int32, device="cuda")
        _ok(L.kv_move(pool, p(src), p(dst), 2, stream))
        torch.cuda.synchronize()
        _ok(L.kv_pool_last_error(pool, stream, ctypes.byref(err)))
        assert err.value == gt.KV_DEV_ERR_TIMEOUT
        assert torch.equal(raw, before)
        # the context is still usable: a translate on the same pool and stream
        slots = torch.tensor([9, 17, -1], dtype=torch.int64, device="cuda")
        ids = torch.empty(3, dtype=torch.int32, device="cuda")
        _ok(L.kv_translate(pool, p(slots), 3, None, 0, p(ids), stream))
        torch.cuda.synchronize()
        stride = ps * 2 * 2
        assert ids.cpu().tolist() == [1 * stride + 1, 2 * stride + 1, 0]
        _ok(L.kv_pool_last_error(pool, stream, ctypes.byref(err)))
        assert err.value == 0
    finally:
        _ok(L.kv_pool_destroy(pool))
