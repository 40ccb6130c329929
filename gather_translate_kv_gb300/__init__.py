"""Python binding of libgtkv.so, the C-ABI page-major KV-cache pool for GB300.

Argument marshalling only: every function below checks tensor dtypes, shapes,
devices and contiguity, then calls the C entry point of the same name in
``include/kv_pool.h``; every step of the data path runs in that library's
CUDA kernels. PyTorch provides device memory and streams. There is no other
implementation to fall back to: if ``libgtkv.so`` is missing, every call
raises ``RuntimeError``.

Layout and operations follow the prhub report on sglang PR #34602,
"feat(unified-memory): dense KV views for uniform-row MHA/SWA models".
"""
from __future__ import annotations

import ctypes
import os
import re
from dataclasses import dataclass

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgtkv.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "kv_pool.h")

KV_OK = 0
STATUS = {
    0: "KV_OK", -1: "KV_ERR_INVALID", -2: "KV_ERR_ASYMMETRIC", -3: "KV_ERR_ID_BOUND",
    -4: "KV_ERR_TAIL_PAD", -5: "KV_ERR_ALIGN", -6: "KV_ERR_CUDA", -7: "KV_ERR_DEVICE",
    -8: "KV_ERR_CAPACITY",
}
KV_DEV_ERR_ROW, KV_DEV_ERR_V2P, KV_DEV_ERR_TABLE, KV_DEV_ERR_FORM, KV_DEV_ERR_TIMEOUT = 1, 2, 4, 8, 16


class KVError(RuntimeError):
    def __init__(self, fn: str, code: int):
        self.code = code
        self.name = STATUS.get(code, f"code {code}")
        super().__init__(f"{fn} failed: {self.name}")


class kv_pool_desc(ctypes.Structure):
    _fields_ = [
        ("layer_num", ctypes.c_int32),
        ("head_num", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("v_head_dim", ctypes.c_int32),
        ("itemsize", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("num_pages", ctypes.c_int64),
        ("anchor_bytes", ctypes.c_int64),
        ("latent_only", ctypes.c_int32),
        ("reserved", ctypes.c_int32),
    ]


class kv_pool_info_t(ctypes.Structure):
    _fields_ = [
        ("raw_dev", ctypes.c_void_p),
        ("raw_bytes", ctypes.c_int64),
        ("row_bytes", ctypes.c_int64),
        ("page_bytes", ctypes.c_int64),
        ("total_bytes", ctypes.c_int64),
        ("tail_pad_bytes", ctypes.c_int64),
        ("n_rows", ctypes.c_int64),
        ("last_view_end", ctypes.c_int64),
        ("device", ctypes.c_int32),
        ("owns_raw", ctypes.c_int32),
        ("blocks_per_page", ctypes.c_int32),
        ("latent_only", ctypes.c_int32),
    ]


def make_desc(layer_num, head_num, head_dim, itemsize, page_size, num_pages, anchor_bytes=0,
              v_head_dim=None, latent_only=False) -> kv_pool_desc:
    """Pool geometry; latent_only=True makes an MLA pool (one latent row of
    head_num * head_dim elements per layer per token, no V)."""
    return kv_pool_desc(layer_num, head_num, head_dim, head_dim if v_head_dim is None else v_head_dim,
                        itemsize, page_size, num_pages, anchor_bytes, 1 if latent_only else 0, 0)


_lib = None


def header_functions() -> list[str]:
    """Names of the functions include/kv_pool.h declares."""
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(kv_\w+)\s*\(", src, flags=re.M)


def lib():
    """Load libgtkv.so (built in-tree by gather_translate_kv_gb300.build)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'` "
            "(there is no fallback implementation)"
        )
    _lib = load(LIB_PATH)
    return _lib


def load(path: str) -> ctypes.CDLL:
    """A library built from these sources (libgtkv.so, or a build with other
    flags), with the argument types of include/kv_pool.h set."""
    L = ctypes.CDLL(path)
    P, vp, i32, i64 = ctypes.POINTER, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    sig = {
        "kv_pool_required_bytes": [P(kv_pool_desc), P(i64), P(i64)],
        "kv_pool_create": [P(kv_pool_desc), vp, i64, P(vp)],
        "kv_pool_destroy": [vp],
        "kv_pool_info": [vp, P(kv_pool_info_t)],
        "kv_translate": [vp, vp, i64, vp, i64, vp, vp],
        "kv_translate_mapped": [vp, vp, i64, vp, i64, vp, i64, vp, vp],
        "kv_store_layer": [vp, i32, vp, i64, vp, vp, vp],
        "kv_store_all_layers": [vp, vp, i64, vp, vp, vp],
        "kv_store_layer_slots": [vp, i32, vp, i64, vp, i64, vp, vp, vp],
        "kv_store_all_layers_slots": [vp, vp, i64, vp, i64, vp, vp, vp],
        "kv_gather_layer": [vp, i32, vp, i32, i32, vp, vp, vp, vp, vp, i64, vp],
        "kv_move": [vp, vp, vp, i64, vp],
        "kv_gather_plan_bytes": [vp, i32, i32, P(i64)],
        "kv_gather_plan": [vp, vp, i32, i32, vp, vp, vp, i64, vp],
        "kv_gather_plan_noalloc": [vp, vp, i32, i32, vp, vp, vp, i64, vp],
        "kv_gather_layer_planned": [vp, i32, vp, i64, vp, i32, i32, vp, vp, vp, vp, vp, i64, vp],
        "kv_translate_block_table": [vp, vp, i32, i32, vp, vp, i64, vp, vp],
        "kv_gather_layer_kf": [vp, i32, vp, i32, i32, vp, vp, vp, vp, vp, i64, vp],
        "kv_gather_plan_kf": [vp, vp, i32, i32, vp, vp, vp, i64, vp],
        "kv_gather_layer_planned_kf": [vp, i32, vp, i64, vp, i32, i32, vp, vp, vp, vp, vp, i64, vp],
        "kv_pool_last_error": [vp, vp, P(i32)],
    }
    for name, args in sig.items():
        f = getattr(L, name)
        f.argtypes = args
        f.restype = ctypes.c_int
    L.kv_status_string.argtypes = [ctypes.c_int]
    L.kv_status_string.restype = ctypes.c_char_p
    return L


def _check(fn: str, rc: int) -> None:
    if rc != KV_OK:
        raise KVError(fn, rc)


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _dev(t: torch.Tensor | None, name: str, dtype=None, nbytes=None):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.device.index != torch.cuda.current_device():
        # every call runs on the current device, which must be the pool's
        raise ValueError(f"{name} is on {t.device}, the current device is cuda:{torch.cuda.current_device()}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if nbytes is not None and t.numel() * t.element_size() != nbytes:
        raise ValueError(f"{name} holds {t.numel() * t.element_size()} bytes, expected {nbytes}")
    return ctypes.c_void_p(t.data_ptr())


@dataclass
class KVPool:
    """A pool handle. Keeps the borrowed raw buffer alive."""

    handle: ctypes.c_void_p
    desc: kv_pool_desc
    raw: torch.Tensor | None
    info: dict

    @property
    def row_bytes(self) -> int:
        return self.info["row_bytes"]

    def __del__(self):
        try:
            if self.handle:
                lib().kv_pool_destroy(self.handle)
                self.handle = None
        except Exception:
            pass


def kv_pool_required_bytes(desc: kv_pool_desc) -> tuple[int, int]:
    total, pad = ctypes.c_int64(), ctypes.c_int64()
    _check("kv_pool_required_bytes", lib().kv_pool_required_bytes(ctypes.byref(desc), ctypes.byref(total),
                                                                  ctypes.byref(pad)))
    return total.value, pad.value


def kv_pool_create(desc: kv_pool_desc, raw: torch.Tensor | None = None, raw_bytes: int | None = None) -> KVPool:
    """Create a pool on the current CUDA device; ``raw`` (uint8, CUDA) is
    borrowed, else the library allocates the buffer."""
    h = ctypes.c_void_p()
    if raw is not None:
        ptr = _dev(raw, "raw", torch.uint8)
        nbytes = raw.numel() if raw_bytes is None else raw_bytes
    else:
        ptr, nbytes = None, 0
    _check("kv_pool_create", lib().kv_pool_create(ctypes.byref(desc), ptr, nbytes, ctypes.byref(h)))
    pool = KVPool(h, desc, raw, {})
    pool.info = kv_pool_info(pool)
    return pool


def kv_pool_destroy(pool: KVPool) -> None:
    if pool.handle:
        rc = lib().kv_pool_destroy(pool.handle)
        pool.handle = None
        _check("kv_pool_destroy", rc)


def kv_pool_info(pool: KVPool) -> dict:
    out = kv_pool_info_t()
    _check("kv_pool_info", lib().kv_pool_info(pool.handle, ctypes.byref(out)))
    return {f: getattr(out, f) for f, _ in kv_pool_info_t._fields_}


def kv_translate(pool: KVPool, slots: torch.Tensor, ids_out: torch.Tensor, v2p: torch.Tensor | None = None,
                 stream=None) -> torch.Tensor:
    n = slots.numel()
    if ids_out.numel() != n:
        raise ValueError("ids_out must have one entry per slot")
    _check("kv_translate", lib().kv_translate(
        pool.handle, _dev(slots, "slots", torch.int64), n, _dev(v2p, "v2p", torch.int32),
        0 if v2p is None else v2p.numel(), _dev(ids_out, "ids_out", torch.int32), _stream(stream)))
    return ids_out


def kv_translate_mapped(pool: KVPool, slots: torch.Tensor, ids_out: torch.Tensor, tmap: torch.Tensor,
                        v2p: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Full-pool slots -> this (SWA) pool's ids through a full -> SWA token map."""
    n = slots.numel()
    if ids_out.numel() != n:
        raise ValueError("ids_out must have one entry per slot")
    _check("kv_translate_mapped", lib().kv_translate_mapped(
        pool.handle, _dev(slots, "slots", torch.int64), n, _dev(tmap, "tmap", torch.int64), tmap.numel(),
        _dev(v2p, "v2p", torch.int32), 0 if v2p is None else v2p.numel(), _dev(ids_out, "ids_out", torch.int32),
        _stream(stream)))
    return ids_out


def kv_store_layer(pool: KVPool, layer: int, ids: torch.Tensor, k: torch.Tensor, v: torch.Tensor | None,
                   stream=None) -> None:
    n = ids.numel()
    nb = n * pool.row_bytes
    _check("kv_store_layer", lib().kv_store_layer(
        pool.handle, layer, _dev(ids, "ids", torch.int32), n, _dev(k, "k", nbytes=nb), _dev(v, "v", nbytes=nb),
        _stream(stream)))


def kv_store_all_layers(pool: KVPool, ids: torch.Tensor, k_all: torch.Tensor, v_all: torch.Tensor | None,
                        stream=None) -> None:
    n = ids.numel()
    nb = pool.desc.layer_num * n * pool.row_bytes
    _check("kv_store_all_layers", lib().kv_store_all_layers(
        pool.handle, _dev(ids, "ids", torch.int32), n, _dev(k_all, "k_all", nbytes=nb),
        _dev(v_all, "v_all", nbytes=nb), _stream(stream)))


def kv_store_layer_slots(pool: KVPool, layer: int, slots: torch.Tensor, k: torch.Tensor, v: torch.Tensor | None,
                         v2p: torch.Tensor | None = None, stream=None) -> None:
    n = slots.numel()
    nb = n * pool.row_bytes
    _check("kv_store_layer_slots", lib().kv_store_layer_slots(
        pool.handle, layer, _dev(slots, "slots", torch.int64), n, _dev(v2p, "v2p", torch.int32),
        0 if v2p is None else v2p.numel(), _dev(k, "k", nbytes=nb), _dev(v, "v", nbytes=nb), _stream(stream)))


def kv_store_all_layers_slots(pool: KVPool, slots: torch.Tensor, k_all: torch.Tensor, v_all: torch.Tensor | None,
                              v2p: torch.Tensor | None = None, stream=None) -> None:
    n = slots.numel()
    nb = pool.desc.layer_num * n * pool.row_bytes
    _check("kv_store_all_layers_slots", lib().kv_store_all_layers_slots(
        pool.handle, _dev(slots, "slots", torch.int64), n, _dev(v2p, "v2p", torch.int32),
        0 if v2p is None else v2p.numel(), _dev(k_all, "k_all", nbytes=nb), _dev(v_all, "v_all", nbytes=nb),
        _stream(stream)))


def _gather(fn: str, pool: KVPool, layer: int, block_table: torch.Tensor, seq_len: torch.Tensor,
            cu_out: torch.Tensor, out_k: torch.Tensor, out_v: torch.Tensor | None, seq_start, stream) -> None:
    if block_table.dim() != 2:
        raise ValueError("block_table must be [n_seqs, max_pages]")
    n_seqs, max_pages = block_table.shape
    if seq_len.numel() != n_seqs or cu_out.numel() != n_seqs + 1:
        raise ValueError("seq_len must be [n_seqs] and cu_out [n_seqs + 1]")
    if seq_start is not None and seq_start.numel() != n_seqs:
        raise ValueError("seq_start must be [n_seqs]")
    R = pool.row_bytes
    ob = out_k.numel() * out_k.element_size()
    if ob % R != 0 or (out_v is not None and out_v.numel() * out_v.element_size() != ob):
        raise ValueError("out_k and out_v must be the same size, a whole number of rows")
    _check(fn, getattr(lib(), fn)(
        pool.handle, layer, _dev(block_table, "block_table", torch.int32), n_seqs, max_pages,
        _dev(seq_start, "seq_start", torch.int32), _dev(seq_len, "seq_len", torch.int32),
        _dev(cu_out, "cu_out", torch.int64), _dev(out_k, "out_k"), _dev(out_v, "out_v"), ob // R,
        _stream(stream)))


def kv_gather_layer(pool: KVPool, layer: int, block_table: torch.Tensor, seq_len: torch.Tensor,
                    cu_out: torch.Tensor, out_k: torch.Tensor, out_v: torch.Tensor | None,
                    seq_start: torch.Tensor | None = None, stream=None) -> None:
    _gather("kv_gather_layer", pool, layer, block_table, seq_len, cu_out, out_k, out_v, seq_start, stream)


def kv_gather_layer_kf(pool: KVPool, layer: int, kf_table: torch.Tensor, seq_len: torch.Tensor,
                       cu_out: torch.Tensor, out_k: torch.Tensor, out_v: torch.Tensor | None,
                       seq_start: torch.Tensor | None = None, stream=None) -> None:
    """kv_gather_layer through a kernel-facing table (kv_translate_block_table's output)."""
    _gather("kv_gather_layer_kf", pool, layer, kf_table, seq_len, cu_out, out_k, out_v, seq_start, stream)


def kv_gather_plan_bytes(pool: KVPool, n_seqs: int, max_pages: int) -> int:
    out = ctypes.c_int64()
    _check("kv_gather_plan_bytes", lib().kv_gather_plan_bytes(pool.handle, n_seqs, max_pages, ctypes.byref(out)))
    return out.value


def _plan(fn: str, pool: KVPool, block_table, seq_len, seq_start, plan, stream) -> torch.Tensor:
    n_seqs, max_pages = block_table.shape
    nbytes = kv_gather_plan_bytes(pool, n_seqs, max_pages)
    if plan is None:
        plan = torch.empty(nbytes // 4, dtype=torch.int32, device=block_table.device)
    _check(fn, getattr(lib(), fn)(
        pool.handle, _dev(block_table, "block_table", torch.int32), n_seqs, max_pages,
        _dev(seq_start, "seq_start", torch.int32), _dev(seq_len, "seq_len", torch.int32),
        _dev(plan, "plan", torch.int32), plan.numel() * 4, _stream(stream)))
    return plan


def kv_gather_plan(pool: KVPool, block_table: torch.Tensor, seq_len: torch.Tensor,
                   seq_start: torch.Tensor | None = None, plan: torch.Tensor | None = None,
                   stream=None) -> torch.Tensor:
    """Page-major plan of a block table (an int32 device tensor, allocated
    here when not given); reuse it for every layer's gather of the step."""
    return _plan("kv_gather_plan", pool, block_table, seq_len, seq_start, plan, stream)


def kv_gather_plan_kf(pool: KVPool, kf_table: torch.Tensor, seq_len: torch.Tensor,
                      seq_start: torch.Tensor | None = None, plan: torch.Tensor | None = None,
                      stream=None) -> torch.Tensor:
    """kv_gather_plan over a kernel-facing table (entries phys * 2L)."""
    return _plan("kv_gather_plan_kf", pool, kf_table, seq_len, seq_start, plan, stream)


def kv_gather_plan_noalloc(pool: KVPool, block_table: torch.Tensor, seq_len: torch.Tensor, plan: torch.Tensor,
                           seq_start: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """kv_gather_plan for callers that cannot allocate device memory: the plan
    buffer (int32, at least kv_gather_plan_bytes() long) is theirs, and the
    sort's counters live in a fixed array of the library (pools of at most
    65536 pages, else KV_ERR_CAPACITY). Nothing is allocated here either.
    Calls that overlap on the GPU share that array and race; the first call
    on a device looks up its address and should precede any stream capture."""
    n_seqs, max_pages = block_table.shape
    _check("kv_gather_plan_noalloc", lib().kv_gather_plan_noalloc(
        pool.handle, _dev(block_table, "block_table", torch.int32), n_seqs, max_pages,
        _dev(seq_start, "seq_start", torch.int32), _dev(seq_len, "seq_len", torch.int32),
        _dev(plan, "plan", torch.int32), plan.numel() * 4, _stream(stream)))
    return plan


def _gather_planned(fn: str, pool: KVPool, layer: int, plan: torch.Tensor, block_table: torch.Tensor,
                    seq_len: torch.Tensor, cu_out: torch.Tensor, out_k: torch.Tensor, out_v: torch.Tensor | None,
                    seq_start, stream) -> None:
    n_seqs, max_pages = block_table.shape
    R = pool.row_bytes
    ob = out_k.numel() * out_k.element_size()
    if ob % R != 0 or (out_v is not None and out_v.numel() * out_v.element_size() != ob):
        raise ValueError("out_k and out_v must be the same size, a whole number of rows")
    _check(fn, getattr(lib(), fn)(
        pool.handle, layer, _dev(plan, "plan", torch.int32), plan.numel() * 4,
        _dev(block_table, "block_table", torch.int32),
        n_seqs, max_pages, _dev(seq_start, "seq_start", torch.int32), _dev(seq_len, "seq_len", torch.int32),
        _dev(cu_out, "cu_out", torch.int64), _dev(out_k, "out_k"), _dev(out_v, "out_v"), ob // R, _stream(stream)))


def kv_gather_layer_planned(pool: KVPool, layer: int, plan: torch.Tensor, block_table: torch.Tensor,
                            seq_len: torch.Tensor, cu_out: torch.Tensor, out_k: torch.Tensor,
                            out_v: torch.Tensor | None, seq_start: torch.Tensor | None = None, stream=None) -> None:
    _gather_planned("kv_gather_layer_planned", pool, layer, plan, block_table, seq_len, cu_out, out_k, out_v,
                    seq_start, stream)


def kv_gather_layer_planned_kf(pool: KVPool, layer: int, plan: torch.Tensor, kf_table: torch.Tensor,
                               seq_len: torch.Tensor, cu_out: torch.Tensor, out_k: torch.Tensor,
                               out_v: torch.Tensor | None, seq_start: torch.Tensor | None = None,
                               stream=None) -> None:
    """kv_gather_layer_planned over a kernel-facing table, with a kv_gather_plan_kf plan."""
    _gather_planned("kv_gather_layer_planned_kf", pool, layer, plan, kf_table, seq_len, cu_out, out_k, out_v,
                    seq_start, stream)


def kv_move(pool: KVPool, src_ids: torch.Tensor, dst_ids: torch.Tensor, stream=None) -> None:
    n = src_ids.numel()
    if dst_ids.numel() != n:
        raise ValueError("src_ids and dst_ids must have the same length")
    _check("kv_move", lib().kv_move(pool.handle, _dev(src_ids, "src_ids", torch.int32),
                                    _dev(dst_ids, "dst_ids", torch.int32), n, _stream(stream)))


def kv_translate_block_table(pool: KVPool, virt_bt: torch.Tensor, seq_len: torch.Tensor, v2p: torch.Tensor,
                             out_bt: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Prefix-only kernel-facing block table (entries phys * 2L); in place
    when out_bt is virt_bt or None."""
    if virt_bt.dim() != 2:
        raise ValueError("virt_bt must be [n_seqs, max_pages]")
    n_seqs, max_pages = virt_bt.shape
    out_bt = virt_bt if out_bt is None else out_bt
    if out_bt.shape != virt_bt.shape or seq_len.numel() != n_seqs:
        raise ValueError("out_bt must match virt_bt; seq_len must be [n_seqs]")
    _check("kv_translate_block_table", lib().kv_translate_block_table(
        pool.handle, _dev(virt_bt, "virt_bt", torch.int32), n_seqs, max_pages, _dev(seq_len, "seq_len", torch.int32),
        _dev(v2p, "v2p", torch.int32), v2p.numel(), _dev(out_bt, "out_bt", torch.int32), _stream(stream)))
    return out_bt


def kv_pool_last_error(pool: KVPool, stream=None) -> int:
    code = ctypes.c_int32()
    _check("kv_pool_last_error", lib().kv_pool_last_error(pool.handle, _stream(stream), ctypes.byref(code)))
    return code.value


def kv_status_string(status: int) -> str:
    return lib().kv_status_string(status).decode()
