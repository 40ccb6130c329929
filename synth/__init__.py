"""Seeded synthetic inputs for the unified page-major KV-cache pool.

This module is shared by the CPU oracle side and the CUDA side of every test
and of the benchmark, and it holds none of the pool's arithmetic: no slot
decomposition, no kernel-facing ids, no row addressing. It only draws token
slots, block tables, sequence lengths and opaque K/V bytes, and it defines
the sentinel pattern a fresh pool is filled with.

Randomness: numpy PCG64. Every (workload seed, stream, layer) triple has its
own generator, seeded with ``SeedSequence([seed, stream, layer])``, so any
layer's inputs can be drawn without drawing the others. Workload seeds are
``1000 + cfg``.

Value distributions:
  * bf16 K/V: float32 standard normal, rounded to bf16 (round to nearest,
    ties to even) by bit manipulation.
  * fp8 (e4m3fn) K/V: uniform over the 254 byte codes that are not NaN
    (0x7F and 0xFF excluded).

Sentinel fill: the 8-byte word at byte offset 8*w of the raw pool buffer is
``splitmix64(fill_seed ^ w)``, stored little-endian. splitmix64 is Vigna's
published mixer (increment 0x9E3779B97F4A7C15, multipliers
0xBF58476D1CE4E5B9 and 0x94D049BB133111EB, shifts 30/27/31). Every row of a
filled pool is then distinct, so reading a row never written in a run still
has well-defined expected bytes. A numpy version serves the host side and a
torch version fills device buffers in place; tests check they agree.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

# streams
S_SLOTS, S_TOMB, S_TABLE, S_VALS, S_MOVE, S_MISC = range(6)


def rng_for(seed: int, stream: int, layer: int = 0) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([int(seed), int(stream), int(layer)]))


# --------------------------------------------------------------------- values

def bf16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest, ties to even."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = (u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_normal(rng: np.random.Generator, shape) -> np.ndarray:
    return bf16_bits_from_f32(rng.standard_normal(shape, dtype=np.float32))


def fp8_e4m3_bytes(rng: np.random.Generator, shape) -> np.ndarray:
    """Uniform over the 254 non-NaN e4m3fn codes (skip 0x7F and 0xFF)."""
    x = rng.integers(0, 254, size=shape, dtype=np.uint16)
    x = x + (x >= 0x7F).astype(np.uint16)
    return x.astype(np.uint8)


def kv_values(rng: np.random.Generator, shape, itemsize: int) -> np.ndarray:
    """K or V payload with the dtype's distribution; returned as raw bytes
    (uint16 for bf16, uint8 for fp8)."""
    if itemsize == 2:
        return bf16_normal(rng, shape)
    if itemsize == 1:
        return fp8_e4m3_bytes(rng, shape)
    if itemsize == 4:
        return rng.standard_normal(shape, dtype=np.float32).view(np.uint32)
    raise ValueError(f"itemsize {itemsize}")


# ------------------------------------------------------------------- sentinel

_SM_INC = np.uint64(0x9E3779B97F4A7C15)
_SM_M1 = np.uint64(0xBF58476D1CE4E5B9)
_SM_M2 = np.uint64(0x94D049BB133111EB)


def splitmix64_np(x: np.ndarray) -> np.ndarray:
    z = np.asarray(x, dtype=np.uint64) + _SM_INC
    z = (z ^ (z >> np.uint64(30))) * _SM_M1
    z = (z ^ (z >> np.uint64(27))) * _SM_M2
    return z ^ (z >> np.uint64(31))


def sentinel_bytes(fill_seed: int, offset: int, nbytes: int) -> np.ndarray:
    """Bytes [offset, offset+nbytes) of the sentinel pattern."""
    if nbytes <= 0:
        return np.zeros(0, dtype=np.uint8)
    w0 = offset // 8
    w1 = (offset + nbytes + 7) // 8
    words = np.arange(w0, w1, dtype=np.uint64) ^ np.uint64(fill_seed)
    b = splitmix64_np(words).astype("<u8").view(np.uint8)
    s = offset - 8 * w0
    return b[s : s + nbytes].copy()


def sentinel_rows(fill_seed: int, byte_offsets: np.ndarray, row_bytes: int) -> np.ndarray:
    """Sentinel content of many rows at once: [len(byte_offsets), row_bytes]."""
    offs = np.asarray(byte_offsets, dtype=np.int64)
    out = np.empty((offs.size, row_bytes), dtype=np.uint8)
    if offs.size == 0:
        return out
    aligned = np.all(offs % 8 == 0) and row_bytes % 8 == 0
    if aligned:
        nw = row_bytes // 8
        w = (offs // 8)[:, None] + np.arange(nw, dtype=np.int64)[None, :]
        words = splitmix64_np(w.astype(np.uint64) ^ np.uint64(fill_seed))
        return words.astype("<u8").view(np.uint8).reshape(offs.size, row_bytes)
    for i, o in enumerate(offs):
        out[i] = sentinel_bytes(fill_seed, int(o), row_bytes)
    return out


def _i64(v: int) -> int:
    v &= (1 << 64) - 1
    return v - (1 << 64) if v >= (1 << 63) else v


def fill_sentinel_torch(buf, fill_seed: int, chunk_words: int = 1 << 26, byte_offset: int = 0) -> None:
    """Fill a uint8 torch tensor (any device, contiguous, length % 8 == 0)
    with the sentinel pattern, in place, chunk by chunk. ``byte_offset``
    (a multiple of 8) is the pattern offset of buf[0]."""
    import torch

    assert buf.dtype == torch.uint8 and buf.is_contiguous() and buf.numel() % 8 == 0 and byte_offset % 8 == 0
    words = buf.view(torch.int64)
    n = words.numel()
    inc, m1, m2 = _i64(0x9E3779B97F4A7C15), _i64(0xBF58476D1CE4E5B9), _i64(0x94D049BB133111EB)
    mask = {k: (1 << (64 - k)) - 1 for k in (30, 27, 31)}
    for w0 in range(0, n, chunk_words):
        w1 = min(n, w0 + chunk_words)
        z = torch.arange(w0 + byte_offset // 8, w1 + byte_offset // 8, dtype=torch.int64, device=buf.device)
        z.bitwise_xor_(int(fill_seed))
        z.add_(inc)
        z.bitwise_xor_(torch.bitwise_right_shift(z, 30).bitwise_and_(mask[30])).mul_(m1)
        z.bitwise_xor_(torch.bitwise_right_shift(z, 27).bitwise_and_(mask[27])).mul_(m2)
        z.bitwise_xor_(torch.bitwise_right_shift(z, 31).bitwise_and_(mask[31]))
        words[w0:w1].copy_(z)
        del z


# ------------------------------------------------------------------ workloads

@dataclass(frozen=True)
class Shape:
    """Model / pool shape of one workload, in the report's notation."""

    cfg: int
    name: str
    layer_num: int
    head_num: int
    head_dim: int
    itemsize: int
    page_size: int
    num_pages: int
    latent: bool = False  # MLA pool: one latent row (head_num * head_dim) per layer per token

    @property
    def seed(self) -> int:
        return 1000 + self.cfg

    @property
    def row_bytes(self) -> int:
        return self.head_num * self.head_dim * self.itemsize

    @property
    def n_slots(self) -> int:
        return self.page_size * self.num_pages

    def scaled(self, num_pages: int) -> "Shape":
        """Same model shape on a smaller pool (for element-by-element tests)."""
        return Shape(self.cfg, self.name + f"@P{num_pages}", self.layer_num, self.head_num,
                     self.head_dim, self.itemsize, self.page_size, num_pages, self.latent)


SHAPES = {
    1: Shape(1, "tiny", 2, 2, 8, 2, 4, 64),
    2: Shape(2, "llama3-8b-decode", 32, 8, 128, 2, 16, 4096),
    3: Shape(3, "llama3-8b-prefill", 32, 8, 128, 2, 64, 4096),
    4: Shape(4, "swa-fp8", 24, 8, 64, 1, 32, 16384),
    5: Shape(5, "id-bound-stress-fp8", 80, 1, 64, 1, 256, 48828),
    # MLA pool (DeepSeek-like latent 512 + 64 rope, bf16, 61 layers), ~8 GiB
    6: Shape(6, "mla-deepseek-like", 61, 1, 576, 2, 64, 1820, latent=True),
}


@dataclass
class GatherBatch:
    """Block-table read of one layer: physical pages per sequence, token
    window [seq_start, seq_len), packed output offsets cu (len n_seqs+1)."""

    block_table: np.ndarray  # int32 [S, max_pages]
    seq_start: np.ndarray    # int32 [S]
    seq_len: np.ndarray      # int32 [S]
    cu: np.ndarray = field(default=None)  # int64 [S+1]

    def __post_init__(self):
        if self.cu is None:
            cnt = np.maximum(self.seq_len.astype(np.int64) - self.seq_start.astype(np.int64), 0)
            self.cu = np.concatenate([[0], np.cumsum(cnt)]).astype(np.int64)

    @property
    def total(self) -> int:
        return int(self.cu[-1])


def kv_pair(shape: Shape, n: int, layer: int, seed: int | None = None, stream: int = S_VALS):
    """K and V payload rows [n, H, D] (raw bits) for one layer."""
    rng = rng_for(shape.seed if seed is None else seed, stream, layer)
    dims = (n, shape.head_num, shape.head_dim)
    return kv_values(rng, dims, shape.itemsize), kv_values(rng, dims, shape.itemsize)


def kv_pair_all(shape: Shape, n: int, seed: int | None = None, stream: int = S_VALS):
    """K_all and V_all [L, n, H, D], layer-major."""
    ks, vs = [], []
    for l in range(shape.layer_num):
        k, v = kv_pair(shape, n, l, seed, stream + 100)
        ks.append(k)
        vs.append(v)
    return np.stack(ks), np.stack(vs)


def distinct_slots(rng, lo: int, hi: int, n: int) -> np.ndarray:
    """n distinct slots drawn uniformly from [lo, hi)."""
    span = hi - lo
    assert 0 <= n <= span
    if n * 8 < span:
        picked = np.unique(rng.integers(lo, hi, size=int(n * 1.1) + 16, dtype=np.int64))
        while picked.size < n:
            more = rng.integers(lo, hi, size=n, dtype=np.int64)
            picked = np.unique(np.concatenate([picked, more]))
        return rng.permutation(rng.choice(picked, size=n, replace=False))
    return lo + rng.permutation(span)[:n].astype(np.int64)


def with_tombstones(rng, slots: np.ndarray, count: int) -> np.ndarray:
    out = slots.copy()
    if count > 0:
        out[rng.choice(out.size, size=count, replace=False)] = -1
    return out


# -- per-config generators (sizes follow the workload table of the build plan)

def store_slots(shape: Shape, layer: int, n: int | None = None) -> np.ndarray:
    """Token slots for one layer's store call of this workload."""
    ps, P = shape.page_size, shape.num_pages
    rng = rng_for(shape.seed, S_SLOTS, layer)
    if shape.cfg == 1:
        n = 100 if n is None else n
        s = rng.permutation(np.arange(ps, 256 if P == 64 else P * ps, dtype=np.int64))[:n]
        return with_tombstones(rng_for(shape.seed, S_TOMB, layer), s, max(1, n // 20))
    if shape.cfg in (2, 6):
        n = 256 if n is None else n
        return distinct_slots(rng, ps, P * ps, n)
    if shape.cfg == 3:
        return prefill_slots(shape)[0]
    if shape.cfg == 4:
        return swa_batch(shape)[0]
    if shape.cfg == 5:
        n = (1 << 20) if n is None else n
        last4 = np.arange(max(1, P - 4) * ps, P * ps, dtype=np.int64)
        n_forced = min(n, last4.size)
        rest = distinct_slots(rng, ps, max(1, P - 4) * ps, n - n_forced)
        s = np.concatenate([last4[-n_forced:], rest])
        return rng.permutation(s)
    raise ValueError(shape.cfg)


def prefill_slots(shape: Shape, n_seqs: int = 16, pages_per_seq: int = 32):
    """Prefill layout: pages 1..P-1 cut into runs of U{1..8} pages, runs
    shuffled and concatenated, the first n_seqs*pages_per_seq taken; sequence
    s owns pages[s*pps:(s+1)*pps] and its tokens fill them in order; 2% of
    the token positions are then tombstoned (-1)."""
    ps, P = shape.page_size, shape.num_pages
    rng = rng_for(shape.seed, S_TABLE, 0)
    runs, p = [], 1
    while p < P:
        k = int(rng.integers(1, 9))
        runs.append(np.arange(p, min(P, p + k), dtype=np.int64))
        p += k
    order = rng.permutation(len(runs))
    pages = np.concatenate([runs[i] for i in order])[: n_seqs * pages_per_seq]
    assert pages.size == n_seqs * pages_per_seq
    slots = (pages[:, None] * ps + np.arange(ps, dtype=np.int64)[None, :]).reshape(-1)
    n_tomb = int(round(0.02 * slots.size))
    slots = with_tombstones(rng_for(shape.seed, S_TOMB, 0), slots, n_tomb)
    return slots, pages.reshape(n_seqs, pages_per_seq).astype(np.int32)


def swa_batch(shape: Shape, n_seqs: int = 512, window: int = 128, pages_per_seq: int = 5):
    """SWA decode step: context c_s = 128 + U[0, 32); 5 pages per sequence,
    distinct across all sequences; the new token sits at position c_s - 1 and
    the window read is [c_s - 128, c_s). Returns (store slots, GatherBatch)."""
    ps, P = shape.page_size, shape.num_pages
    rng = rng_for(shape.seed, S_TABLE, 0)
    ctx = window + rng.integers(0, 32, size=n_seqs)
    pages = (1 + rng.permutation(P - 1)[: n_seqs * pages_per_seq]).astype(np.int32)
    bt = pages.reshape(n_seqs, pages_per_seq)
    pos = ctx - 1
    slots = bt[np.arange(n_seqs), pos // ps].astype(np.int64) * ps + pos % ps
    g = GatherBatch(bt, (ctx - window).astype(np.int32), ctx.astype(np.int32))
    return slots.astype(np.int64), g


def gather_batch(shape: Shape) -> GatherBatch:
    """The block-table read of this workload."""
    ps, P = shape.page_size, shape.num_pages
    rng = rng_for(shape.seed, S_TABLE, 1)
    if shape.cfg == 1:
        pages = rng.choice(np.arange(1, P), size=8, replace=False).astype(np.int32)
        return GatherBatch(pages[None, :], np.zeros(1, np.int32), np.full(1, 8 * ps, np.int32))
    if shape.cfg == 2:
        S, npg = 256, 256
        npg = min(npg, P - 1)
        bt = np.stack([1 + rng.permutation(P - 1)[:npg] for _ in range(S)]).astype(np.int32)
        return GatherBatch(bt, np.zeros(S, np.int32), np.full(S, npg * ps, np.int32))
    if shape.cfg == 6:
        S, npg = 128, min(64, P - 1)
        bt = np.stack([1 + rng.permutation(P - 1)[:npg] for _ in range(S)]).astype(np.int32)
        return GatherBatch(bt, np.zeros(S, np.int32), np.full(S, npg * ps, np.int32))
    if shape.cfg == 3:
        _, bt = prefill_slots(shape)
        S = bt.shape[0]
        return GatherBatch(bt, np.zeros(S, np.int32), np.full(S, bt.shape[1] * ps, np.int32))
    if shape.cfg == 4:
        return swa_batch(shape)[1]
    if shape.cfg == 5:
        S, npg = 1024, 4
        bt = rng.integers(1, P, size=(S, npg)).astype(np.int32)
        bt[int(rng.integers(S)), int(rng.integers(npg))] = P - 1
        return GatherBatch(bt, np.zeros(S, np.int32), np.full(S, npg * ps, np.int32))
    raise ValueError(shape.cfg)


def move_slots(shape: Shape, m: int | None = None, avoid: np.ndarray | None = None):
    """m disjoint (src, dst) slot pairs on pages 1..P-1 (never tombstones).
    Sources avoid nothing; destinations avoid ``avoid`` when given."""
    ps, P = shape.page_size, shape.num_pages
    rng = rng_for(shape.seed, S_MOVE, 0)
    if m is None:
        m = {1: 20, 2: 8192, 3: 8192, 4: 8192, 5: 8192, 6: 4096}.get(shape.cfg, 256)
    if avoid is not None and avoid.size:
        pool = np.setdiff1d(np.arange(ps, P * ps, dtype=np.int64), avoid)
        dst = rng.choice(pool, size=m, replace=False)
        rest = np.setdiff1d(np.arange(ps, P * ps, dtype=np.int64), dst)
        src = rng.choice(rest, size=m, replace=False)
        return src.astype(np.int64), dst.astype(np.int64)
    both = distinct_slots(rng, ps, P * ps, 2 * m)
    return both[:m].copy(), both[m:].copy()


def sentinel_rows_torch(fill_seed: int, byte_offsets, row_bytes: int, chunk_rows: int = 1 << 16):
    """Sentinel content of many rows, computed on the offsets' device:
    uint8 [n, row_bytes]. Offsets and row_bytes must be multiples of 8."""
    import torch

    assert row_bytes % 8 == 0
    offs = byte_offsets.to(torch.int64)
    n = offs.numel()
    out = torch.empty((n, row_bytes), dtype=torch.uint8, device=offs.device)
    words_out = out.view(torch.int64).view(n, row_bytes // 8)
    inc, m1, m2 = _i64(0x9E3779B97F4A7C15), _i64(0xBF58476D1CE4E5B9), _i64(0x94D049BB133111EB)
    mask = {k: (1 << (64 - k)) - 1 for k in (30, 27, 31)}
    lane = torch.arange(row_bytes // 8, dtype=torch.int64, device=offs.device)
    for r0 in range(0, n, chunk_rows):
        r1 = min(n, r0 + chunk_rows)
        z = (offs[r0:r1, None] // 8) + lane[None, :]
        z.bitwise_xor_(int(fill_seed))
        z.add_(inc)
        z.bitwise_xor_(torch.bitwise_right_shift(z, 30).bitwise_and_(mask[30])).mul_(m1)
        z.bitwise_xor_(torch.bitwise_right_shift(z, 27).bitwise_and_(mask[27])).mul_(m2)
        z.bitwise_xor_(torch.bitwise_right_shift(z, 31).bitwise_and_(mask[31]))
        words_out[r0:r1].copy_(z)
    return out
