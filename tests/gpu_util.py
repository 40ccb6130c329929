"""Helpers for the GPU parity tests: a sentinel-filled device pool next to its
host mirror, and byte comparisons with the sink rule.

Sink rule. Tombstoned tokens all clamp to id 0, the page-0 sink (the report:
"tombstone -1 clamped to 0 (page-0 sink)"), so one store may write the sink
rows (page 0, offset 0, every block) several times at once. The oracle writes
them in input order; on the GPU the writers race. So the sink rows are not
compared byte for byte: each aligned 4-byte word of a sink row must equal the
word at the same position of the row's prior content or of one of the
tombstoned inputs written to that block (a 4-byte word is the unit a 16-byte
vector store writes atomically). Every other byte is compared exactly.
"""
from __future__ import annotations

import numpy as np
import torch

import gather_translate_kv_gb300 as gt
import oracle
import synth

DEV_BITS = {oracle.E_ROW: gt.KV_DEV_ERR_ROW, oracle.E_V2P: gt.KV_DEV_ERR_V2P,
            oracle.E_TABLE: gt.KV_DEV_ERR_TABLE, oracle.E_FORM: gt.KV_DEV_ERR_FORM}


def dev_bits(oracle_err: int) -> int:
    out = 0
    for ob, gb in DEV_BITS.items():
        if oracle_err & ob:
            out |= gb
    return out


class PoolPair:
    """A device pool (borrowed sentinel-filled torch buffer) and, optionally,
    a host mirror of the same bytes for the oracle."""

    def __init__(self, shape: synth.Shape, anchor: int = 0, fill_seed: int = 4242, mirror: bool = True,
                 device: str = "cuda", latent: bool = False):
        self.shape = shape
        self.latent = latent
        self.geom = oracle.Geometry(shape.layer_num, shape.head_num, shape.head_dim, shape.itemsize,
                                    shape.page_size, shape.num_pages, anchor, latent_only=latent)
        self.o = oracle.Oracle(self.geom)
        self.sizes = self.o.sizes()
        self.R = self.sizes["row_bytes"]
        self.nbytes = self.o.raw_bytes()
        self.fill_seed = fill_seed
        self.raw = torch.empty(self.nbytes, dtype=torch.uint8, device=device)
        synth.fill_sentinel_torch(self.raw, fill_seed)
        self.M = synth.sentinel_bytes(fill_seed, 0, self.nbytes) if mirror else None
        self.desc = gt.make_desc(shape.layer_num, shape.head_num, shape.head_dim, shape.itemsize,
                                 shape.page_size, shape.num_pages, anchor, latent_only=latent)
        self.pool = gt.kv_pool_create(self.desc, self.raw)
        self.anchor = anchor

    def sink_bytes(self) -> list[int]:
        return [self.o.slot_row_byte(0, b) for b in range(self.geom.blocks)]

    def last_error(self) -> int:
        return gt.kv_pool_last_error(self.pool)

    def close(self):
        gt.kv_pool_destroy(self.pool)
        del self.raw


def to_dev(a: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def as_rows(a: np.ndarray, R: int) -> np.ndarray:
    b = np.ascontiguousarray(a).view(np.uint8)
    return b.reshape(-1, R)


def assert_bytes_equal(got: np.ndarray, want: np.ndarray, what: str, R: int | None = None):
    if np.array_equal(got, want):
        return
    bad = np.nonzero(got != want)[0]
    first = int(bad[0])
    msg = f"{what}: {bad.size} bytes differ, first at byte {first}"
    if R:
        msg += f" (row {first // R}, byte {first % R})"
    raise AssertionError(msg)


def assert_pool_matches(pp: PoolPair, M_prior: np.ndarray, tomb_rows: dict[int, list[np.ndarray]] | None = None):
    """Device pool == pp.M everywhere but the sink rows, which follow the sink rule."""
    got = pp.raw.cpu().numpy()
    want = pp.M
    R = pp.R
    mask = np.ones(got.size, dtype=bool)
    sinks = pp.sink_bytes()
    for s in sinks:
        mask[s:s + R] = False
    assert_bytes_equal(got[mask], want[mask], "pool (outside the sink rows)")
    tomb_rows = tomb_rows or {}
    for b, s in enumerate(sinks):
        row = got[s:s + R].view(np.uint32)
        cands = [M_prior[s:s + R].view(np.uint32)] + [np.ascontiguousarray(t).view(np.uint32)
                                                       for t in tomb_rows.get(b, [])]
        ok = np.zeros(row.size, dtype=bool)
        for c in cands:
            ok |= row == c
        assert ok.all(), f"sink row of block {b} holds words from no candidate"


def tomb_inputs(slots: np.ndarray, K: np.ndarray, V: np.ndarray | None, layer: int, R: int) -> dict:
    """Rows written to the sink by tombstoned tokens, keyed by block (an MLA
    pool, V None, has one latent block per layer)."""
    idx = np.nonzero(np.asarray(slots) < 0)[0]
    Kr = as_rows(K, R)
    if V is None:
        return {layer: [Kr[i] for i in idx]}
    Vr = as_rows(V, R)
    return {2 * layer: [Kr[i] for i in idx], 2 * layer + 1: [Vr[i] for i in idx]}


def merge(a: dict, b: dict) -> dict:
    out = {k: list(v) for k, v in a.items()}
    for k, v in b.items():
        out.setdefault(k, []).extend(v)
    return out
