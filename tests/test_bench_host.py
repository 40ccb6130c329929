"""Host-side accounting of bench.py (no GPU): the method bytes of a gather
launch against a brute-force count, and the decode step's totals against
values worked out by hand."""
from __future__ import annotations

import numpy as np

import bench
import synth


def _brute(g: synth.GatherBatch, ps: int, R: int, kv_rows: int = 2):
    tokens, rows, entries = set(), 0, set()
    for s in range(g.block_table.shape[0]):
        for j in range(int(g.seq_start[s]), int(g.seq_len[s])):
            page = int(g.block_table[s, j // ps])
            tokens.add(-1 if page < 0 else page * ps + j % ps)
            entries.add((s, j // ps))
            rows += 1
    S = g.block_table.shape[0]
    method = len(tokens) * kv_rows * R + rows * kv_rows * R + len(entries) * 4 + S * 16
    return method, rows, len(tokens), len(entries)


def test_gather_method_bytes_match_brute_force():
    rng = np.random.default_rng(5)
    for ps, kv_rows in ((4, 2), (16, 2), (3, 1)):
        bt = rng.integers(1, 9, size=(7, 5)).astype(np.int32)
        bt[2, 1] = -1
        bt[4, 0] = -1
        ln = rng.integers(0, 5 * ps + 1, size=7).astype(np.int32)
        st = np.minimum(rng.integers(0, 2 * ps, size=7), ln).astype(np.int32)
        g = synth.GatherBatch(bt, st, ln)
        got = bench.gather_bytes(g, ps, 64, kv_rows)
        method, rows, distinct, entries = _brute(g, ps, 64, kv_rows)
        assert (got["method"], got["rows"], got["distinct_source_rows"], got["table_entries"]) == \
            (method, rows, distinct, entries)
        assert got["per_reader"] == rows * 2 * kv_rows * 64 + rows * 4 // ps


def test_decode_step_bytes_by_hand():
    """256 sequences x 4096 tokens over tables that are heads of permutations
    of pages 1..4095: all 4095 pages are read, 16 rows each, K and V of 2 KiB."""
    inp = bench.make_inputs(0)
    by_kernel, gb = bench.step_bytes(inp["g"])
    assert gb["rows"] == 256 * 4096 and gb["table_entries"] == 256 * 256
    assert gb["distinct_source_rows"] == 4095 * 16
    assert gb["method"] == 4095 * 16 * 4096 + 256 * 4096 * 4096 + 256 * 256 * 4 + 256 * 16
    assert gb["per_reader"] == 256 * 4096 * 8192 + 256 * 4096 * 4 // 16
    assert by_kernel["gather"] == 32 * gb["method"]
    assert by_kernel["move"] == 8192 * (64 * 2048 * 2 + 8)
    assert by_kernel["store_layer"] == 32 * 256 * (4 * 2048 + 4)
    assert by_kernel["store_all_layers"] == 256 * (64 * 2048 * 2 + 4)
    # the method bytes never count a source row twice: at most the per-reader figure
    assert gb["method"] < gb["per_reader"]


def test_cpu_table_cases_fit_their_pools():
    for cfg in bench.CPU_TABLE:
        c = bench._cpu_cases(cfg)
        sh = c["sh"]
        assert c["slots"].min() >= sh.page_size and c["slots"].max() < sh.num_pages * sh.page_size
        assert c["g"].block_table.max() < sh.num_pages and c["g"].block_table.min() >= 1
        assert len(set(c["slots"].tolist())) == c["n"]
