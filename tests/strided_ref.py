"""Independent second reference: the pool as a 5-D [page, 2L, ps, H, D] array.

This is the retired strided page-major view the report says the dense views
replaced (sglang PR #34602 report, 关键文件: build_page_major_mha_views in
layout/page_major.py, and the 4D strided store_cache_4d kernel in
cache_move.py). It is rebuilt here from the envelope statement alone --
"[L0_K*ps | L0_V*ps | L1_K*ps | ...], layer l's K in block 2l and its V in
block 2l+1" (实现拆解 step 1) -- by reshaping the pool bytes into a C-order
5-D array. It computes no byte offsets and never forms a kernel-facing id,
so it shares no arithmetic with the oracle (which uses an explicit
envelope-offset formula) or with the CUDA library (which uses ids).

The report's own test file anchors its dense views against such a strided
builder ("test_addressing_matches_strided_reference", 评论区精华).
"""
from __future__ import annotations

import numpy as np

_DT = {1: np.uint8, 2: np.uint16, 4: np.uint32}


def envelope(buf: np.ndarray, L, H, D, itemsize, ps, P, anchor=0, latent=False) -> np.ndarray:
    """View of the pool region of ``buf`` (uint8) as [P, 2L, ps, H, D], or as
    [P, L, ps, H, D] for an MLA pool (one latent block per layer, 实现拆解
    step 2: blocks_per_page() = layer_num for MLA)."""
    R = H * D * itemsize
    B = L if latent else 2 * L
    region = buf[anchor : anchor + P * B * ps * R]
    return region.view(_DT[itemsize]).reshape(P, B, ps, H, D)


def _where(t, ps, v2p):
    """(page, offset) of token slot t, or the sink (0, 0) for a tombstone."""
    if t < 0:
        return 0, 0
    page, off = divmod(int(t), ps)
    if v2p is not None:
        if page >= len(v2p):
            return 0, 0
        page = int(v2p[page])
        if page < 0:
            return 0, 0
    return page, off


def store(env, layer, slots, K, V, v2p=None, latent=False):
    """K[i] -> env[page, 2*layer, off], V[i] -> env[page, 2*layer+1, off];
    for an MLA pool the latent row K[i] -> env[page, layer, off]."""
    P, B, ps, H, D = env.shape
    Kd = np.asarray(K).reshape(-1, H, D)
    Vd = None if latent else np.asarray(V).reshape(-1, H, D)
    for i, t in enumerate(np.asarray(slots)):
        p, o = _where(t, ps, v2p)
        if latent:
            env[p, layer, o] = Kd[i]
        else:
            env[p, 2 * layer, o] = Kd[i]
            env[p, 2 * layer + 1, o] = Vd[i]


def gather(env, layer, block_table, seq_start, seq_len, latent=False):
    """Rows of layer ``layer`` for every sequence's tokens [start, len), in
    (sequence, token) order; a negative page reads the sink (0, 0). For an
    MLA pool the V list is empty."""
    P, B, ps, H, D = env.shape
    kb = layer if latent else 2 * layer
    ks, vs = [], []
    for s in range(block_table.shape[0]):
        for j in range(int(seq_start[s]), int(seq_len[s])):
            page = int(block_table[s, j // ps])
            off = j % ps
            if page < 0:
                page, off = 0, 0
            ks.append(env[page, kb, off].copy())
            if not latent:
                vs.append(env[page, kb + 1, off].copy())
    z = np.zeros((0, H, D), env.dtype)
    return (np.stack(ks) if ks else z), (np.stack(vs) if vs else z)


def move(env, src_slots, dst_slots):
    """Every row-block of token src -> token dst, all sources read first."""
    P, B, ps, H, D = env.shape
    src = [_where(t, ps, None) for t in src_slots]
    dst = [_where(t, ps, None) for t in dst_slots]
    snap = [env[p, :, o].copy() for (p, o) in src]
    for (p, o), rows in zip(dst, snap):
        env[p, :, o] = rows
