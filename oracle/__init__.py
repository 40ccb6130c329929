"""CPU oracle for the unified page-major KV-cache pool (ctypes over kv_oracle.c).

TEST INFRASTRUCTURE ONLY. The test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` are the only callers. The CUDA library
(``gather_translate_kv_gb300``) never imports this package, and this package
imports nothing from it.

The arithmetic lives in ``kv_oracle.c`` (plain loops and memcpy over a host
byte mirror of the pool); this module only builds it with gcc and marshals
numpy arrays. Its source is the prhub report on sglang PR #34602,
"feat(unified-memory): dense KV views for uniform-row MHA/SWA models".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kv_oracle.c")
_LIB = os.path.join(_HERE, "libkv_oracle.so")

# Error bits returned by the oracle routines (kv_oracle.c).
E_ROW, E_V2P, E_TABLE, E_FORM = 1, 2, 4, 8
# Check codes of check_desc (kv_oracle.c).
CHECK_NAMES = {0: "ok", 1: "bad_arg", 2: "asymmetric", 3: "id_bound", 4: "tail_pad", 5: "anchor"}


def build(force: bool = False) -> str:
    """Compile kv_oracle.c into a shared library next to it (gcc, -O2)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c99", "-Wall", "-shared", "-fPIC", _SRC, "-o", tmp]
        )
        os.replace(tmp, _LIB)
    return _LIB


class _Desc(ctypes.Structure):
    _fields_ = [
        ("layer_num", ctypes.c_int32),
        ("head_num", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("v_head_dim", ctypes.c_int32),
        ("itemsize", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("num_pages", ctypes.c_int64),
        ("anchor", ctypes.c_int64),
        ("latent_only", ctypes.c_int32),
        ("reserved_", ctypes.c_int32),
    ]


@dataclass(frozen=True)
class Geometry:
    """Pool geometry in the report's notation (L, H, D, itemsize, ps, P)."""

    layer_num: int
    head_num: int
    head_dim: int
    itemsize: int
    page_size: int
    num_pages: int
    anchor: int = 0
    v_head_dim: int | None = None
    latent_only: bool = False  # MLA: one latent row per layer per token, no V

    @property
    def blocks(self) -> int:
        return self.layer_num if self.latent_only else 2 * self.layer_num

    def desc(self) -> _Desc:
        return _Desc(
            self.layer_num,
            self.head_num,
            self.head_dim,
            self.head_dim if self.v_head_dim is None else self.v_head_dim,
            self.itemsize,
            self.page_size,
            self.num_pages,
            self.anchor,
            1 if self.latent_only else 0,
            0,
        )


_lib = None


def lib(path: str | None = None):
    global _lib
    if _lib is None or path is not None:
        so = path or build()
        L = ctypes.CDLL(so)
        P = ctypes.POINTER
        c64, c32 = ctypes.c_int64, ctypes.c_int32
        vp = ctypes.c_void_p
        L.ora_sizes.argtypes = [P(_Desc), P(c64)]
        L.ora_sizes.restype = None
        L.ora_check_desc.argtypes = [P(_Desc), c64]
        L.ora_check_desc.restype = ctypes.c_int
        L.ora_translate.argtypes = [P(_Desc), vp, c64, vp, c64, vp]
        L.ora_translate.restype = ctypes.c_int
        L.ora_slot_row_byte.argtypes = [P(_Desc), c64, vp, c64, c32]
        L.ora_slot_row_byte.restype = c64
        L.ora_id_row_byte.argtypes = [P(_Desc), c64, c32]
        L.ora_id_row_byte.restype = c64
        L.ora_store.argtypes = [P(_Desc), vp, c32, vp, c64, vp, c64, vp, vp]
        L.ora_store.restype = ctypes.c_int
        L.ora_store_all.argtypes = [P(_Desc), vp, vp, c64, vp, c64, vp, vp]
        L.ora_store_all.restype = ctypes.c_int
        L.ora_gather.argtypes = [P(_Desc), vp, c32, vp, c32, c32, vp, vp, vp, vp, vp, c64]
        L.ora_gather.restype = ctypes.c_int
        L.ora_gather_kf.argtypes = [P(_Desc), vp, c32, vp, c32, c32, vp, vp, vp, vp, vp, c64]
        L.ora_gather_kf.restype = ctypes.c_int
        L.ora_gather_kf_rows.argtypes = [P(_Desc), c32, vp, c32, c32, vp, vp, vp, c64, vp, vp]
        L.ora_gather_kf_rows.restype = ctypes.c_int
        L.ora_move.argtypes = [P(_Desc), vp, vp, vp, c64]
        L.ora_move.restype = ctypes.c_int
        L.ora_store_rows.argtypes = [P(_Desc), c32, vp, c64, vp, c64, vp, vp]
        L.ora_store_rows.restype = ctypes.c_int
        L.ora_gather_rows.argtypes = [P(_Desc), c32, vp, c32, c32, vp, vp, vp, c64, vp, vp]
        L.ora_gather_rows.restype = ctypes.c_int
        L.ora_move_rows.argtypes = [P(_Desc), vp, vp, c64, vp, vp]
        L.ora_move_rows.restype = ctypes.c_int
        L.ora_block_table_kf.argtypes = [P(_Desc), vp, c32, c32, vp, vp, c64, vp]
        L.ora_block_table_kf.restype = ctypes.c_int
        L.ora_translate_mapped.argtypes = [P(_Desc), vp, c64, vp, c64, vp, c64, vp]
        L.ora_translate_mapped.restype = ctypes.c_int
        L.ora_translate_multiplier.argtypes = [P(_Desc), vp, c64, c32, vp]
        L.ora_translate_multiplier.restype = ctypes.c_int
        if path is not None:
            return L
        _lib = L
    return _lib


def _ptr(a: np.ndarray | None, dtype=None):
    if a is None:
        return None
    if dtype is not None:
        assert a.dtype == dtype, (a.dtype, dtype)
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


class Oracle:
    """Thin marshalling layer; every method calls one routine of kv_oracle.c."""

    def __init__(self, geom: Geometry, so_path: str | None = None):
        self.geom = geom
        self._d = geom.desc()
        self._L = lib(so_path) if so_path else lib()

    # sizes ---------------------------------------------------------------
    def sizes(self) -> dict:
        out = (ctypes.c_int64 * 7)()
        self._L.ora_sizes(ctypes.byref(self._d), out)
        keys = ["row_bytes", "entry_bytes", "page_bytes", "total", "tail_pad", "n_rows", "last_view_end"]
        return dict(zip(keys, list(out)))

    def check(self, raw_bytes: int = -1) -> str:
        return CHECK_NAMES[self._L.ora_check_desc(ctypes.byref(self._d), raw_bytes)]

    def raw_bytes(self) -> int:
        s = self.sizes()
        return self.geom.anchor + s["total"] + s["tail_pad"]

    # translate -----------------------------------------------------------
    def translate(self, slots: np.ndarray, v2p: np.ndarray | None = None):
        slots = np.ascontiguousarray(slots, dtype=np.int64)
        ids = np.empty(slots.shape, dtype=np.int32)
        v = None if v2p is None else np.ascontiguousarray(v2p, dtype=np.int32)
        err = self._L.ora_translate(
            ctypes.byref(self._d), _ptr(slots), slots.size, _ptr(v), 0 if v is None else v.size, _ptr(ids)
        )
        return ids, err

    def translate_multiplier(self, slots: np.ndarray, multiplier: int):
        """Test only: ids with an explicit kernel_page_multiplier (the library's is
        always blocks_per_page); used to pin the multiplier-1 collapse."""
        slots = np.ascontiguousarray(slots, dtype=np.int64)
        ids = np.empty(slots.shape, dtype=np.int32)
        err = self._L.ora_translate_multiplier(ctypes.byref(self._d), _ptr(slots), slots.size, int(multiplier),
                                               _ptr(ids))
        return ids, err

    def translate_mapped(self, slots: np.ndarray, tmap: np.ndarray, v2p: np.ndarray | None = None):
        """Full-pool slots -> this (SWA) pool's ids through a token map."""
        slots = np.ascontiguousarray(slots, dtype=np.int64)
        tm = np.ascontiguousarray(tmap, dtype=np.int64)
        ids = np.empty(slots.shape, dtype=np.int32)
        v = None if v2p is None else np.ascontiguousarray(v2p, dtype=np.int32)
        err = self._L.ora_translate_mapped(ctypes.byref(self._d), _ptr(slots), slots.size, _ptr(tm), tm.size,
                                           _ptr(v), 0 if v is None else v.size, _ptr(ids))
        return ids, err

    def slot_row_byte(self, slot: int, block: int, v2p: np.ndarray | None = None) -> int:
        v = None if v2p is None else np.ascontiguousarray(v2p, dtype=np.int32)
        return self._L.ora_slot_row_byte(
            ctypes.byref(self._d), int(slot), _ptr(v), 0 if v is None else v.size, int(block)
        )

    def id_row_byte(self, kid: int, block: int) -> int:
        return self._L.ora_id_row_byte(ctypes.byref(self._d), int(kid), int(block))

    # store ---------------------------------------------------------------
    def store(self, M: np.ndarray, layer: int, slots, K: np.ndarray, V: np.ndarray, v2p=None) -> int:
        assert M.dtype == np.uint8 and M.size >= self.raw_bytes()
        slots = np.ascontiguousarray(slots, dtype=np.int64)
        Kb = np.ascontiguousarray(K).view(np.uint8)
        Vb = None if V is None else np.ascontiguousarray(V).view(np.uint8)
        R = self.sizes()["row_bytes"]
        assert Kb.size == slots.size * R and (Vb is None or Vb.size == slots.size * R)
        assert Vb is not None or self.geom.latent_only
        v = None if v2p is None else np.ascontiguousarray(v2p, dtype=np.int32)
        return self._L.ora_store(
            ctypes.byref(self._d), _ptr(M), int(layer), _ptr(slots), slots.size,
            _ptr(v), 0 if v is None else v.size, _ptr(Kb), _ptr(Vb),
        )

    def store_all(self, M: np.ndarray, slots, K_all: np.ndarray, V_all: np.ndarray, v2p=None) -> int:
        assert M.dtype == np.uint8 and M.size >= self.raw_bytes()
        slots = np.ascontiguousarray(slots, dtype=np.int64)
        Kb = np.ascontiguousarray(K_all).view(np.uint8)
        Vb = None if V_all is None else np.ascontiguousarray(V_all).view(np.uint8)
        R = self.sizes()["row_bytes"]
        assert Kb.size == self.geom.layer_num * slots.size * R
        assert Vb is not None or self.geom.latent_only
        v = None if v2p is None else np.ascontiguousarray(v2p, dtype=np.int32)
        return self._L.ora_store_all(
            ctypes.byref(self._d), _ptr(M), _ptr(slots), slots.size,
            _ptr(v), 0 if v is None else v.size, _ptr(Kb), _ptr(Vb),
        )

    # gather --------------------------------------------------------------
    def gather(self, M, layer, block_table, seq_len, cu, seq_start=None, out_rows=None,
               outK=None, outV=None):
        """Returns (outK, outV, err) with outK/outV uint8 [out_rows, R]."""
        return self._gather(self._L.ora_gather, M, layer, block_table, seq_len, cu, seq_start, out_rows, outK,
                            outV)

    def gather_kf(self, M, layer, kf_table, seq_len, cu, seq_start=None, out_rows=None,
                  outK=None, outV=None):
        """Gather through a kernel-facing block table (block_table_kf's output):
        (outK, outV, err) as gather()."""
        return self._gather(self._L.ora_gather_kf, M, layer, kf_table, seq_len, cu, seq_start, out_rows, outK,
                            outV)

    def _gather(self, fn, M, layer, block_table, seq_len, cu, seq_start, out_rows, outK, outV):
        bt = np.ascontiguousarray(block_table, dtype=np.int32)
        n_seqs, max_pages = bt.shape
        ln = np.ascontiguousarray(seq_len, dtype=np.int32)
        cu = np.ascontiguousarray(cu, dtype=np.int64)
        st = None if seq_start is None else np.ascontiguousarray(seq_start, dtype=np.int32)
        R = self.sizes()["row_bytes"]
        if out_rows is None:
            out_rows = int(cu[-1]) if n_seqs > 0 else 0
        if outK is None:
            outK = np.zeros((out_rows, R), dtype=np.uint8)
        if outV is None and not self.geom.latent_only:
            outV = np.zeros((out_rows, R), dtype=np.uint8)
        err = fn(ctypes.byref(self._d), _ptr(M), int(layer), _ptr(bt), n_seqs, max_pages,
                 _ptr(st), _ptr(ln), _ptr(cu), _ptr(outK), _ptr(outV), out_rows)
        return outK, outV, err

    # move ----------------------------------------------------------------
    def move(self, M, src_ids, dst_ids) -> int:
        s = np.ascontiguousarray(src_ids, dtype=np.int32)
        d = np.ascontiguousarray(dst_ids, dtype=np.int32)
        assert s.size == d.size
        return self._L.ora_move(ctypes.byref(self._d), _ptr(M), _ptr(s), _ptr(d), s.size)

    # address mode ----------------------------------------------------------
    def store_rows(self, layer: int, slots, v2p=None):
        """Byte offsets a store of ``slots`` writes: (kdst[n], vdst[n], err)."""
        slots = np.ascontiguousarray(slots, dtype=np.int64)
        kd = np.empty(slots.size, np.int64)
        vd = np.empty(slots.size, np.int64)
        v = None if v2p is None else np.ascontiguousarray(v2p, dtype=np.int32)
        err = self._L.ora_store_rows(ctypes.byref(self._d), int(layer), _ptr(slots), slots.size,
                                     _ptr(v), 0 if v is None else v.size, _ptr(kd), _ptr(vd))
        return kd, vd, err

    def gather_rows(self, layer, block_table, seq_len, cu, seq_start=None, out_rows=None, kernel_facing=False):
        """Byte offsets each output row reads: (ksrc[out_rows], vsrc[out_rows], err), -1 = untouched.
        kernel_facing=True reads the table as gather_kf does."""
        bt = np.ascontiguousarray(block_table, dtype=np.int32)
        n_seqs, max_pages = bt.shape
        ln = np.ascontiguousarray(seq_len, dtype=np.int32)
        cu = np.ascontiguousarray(cu, dtype=np.int64)
        st = None if seq_start is None else np.ascontiguousarray(seq_start, dtype=np.int32)
        if out_rows is None:
            out_rows = int(cu[-1]) if n_seqs > 0 else 0
        ks = np.full(out_rows, -1, np.int64)
        vs = np.full(out_rows, -1, np.int64)
        fn = self._L.ora_gather_kf_rows if kernel_facing else self._L.ora_gather_rows
        err = fn(ctypes.byref(self._d), int(layer), _ptr(bt), n_seqs, max_pages,
                 _ptr(st), _ptr(ln), _ptr(cu), out_rows, _ptr(ks), _ptr(vs))
        return ks, vs, err

    def move_rows(self, src_ids, dst_ids):
        """Byte offsets a move reads and writes: (src[m*B], dst[m*B], err), B the
        row-blocks per page (2L, or L for an MLA pool)."""
        s = np.ascontiguousarray(src_ids, dtype=np.int32)
        d = np.ascontiguousarray(dst_ids, dtype=np.int32)
        nb = self.geom.blocks
        sb = np.empty(s.size * nb, np.int64)
        db = np.empty(s.size * nb, np.int64)
        err = self._L.ora_move_rows(ctypes.byref(self._d), _ptr(s), _ptr(d), s.size, _ptr(sb), _ptr(db))
        return sb, db, err

    # kernel-facing block table ---------------------------------------------
    def block_table_kf(self, virt_bt, seq_len, v2p, out=None):
        """Prefix-only kernel-facing table: (out int32 [S, maxp], err)."""
        vb = np.ascontiguousarray(virt_bt, dtype=np.int32)
        n_seqs, max_pages = vb.shape
        ln = np.ascontiguousarray(seq_len, dtype=np.int32)
        v = np.ascontiguousarray(v2p, dtype=np.int32)
        out = np.full(vb.shape, -7, np.int32) if out is None else np.ascontiguousarray(out, dtype=np.int32)
        err = self._L.ora_block_table_kf(ctypes.byref(self._d), _ptr(vb), n_seqs, max_pages, _ptr(ln), _ptr(v),
                                         v.size, _ptr(out))
        return out, err
