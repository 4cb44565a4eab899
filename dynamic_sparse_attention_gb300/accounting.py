"""Algorithmic work of the hot path (host logic for the roofline numbers).

Decode bytes are the key rows the pruning stages must read plus the attended
K/V rows: a SelectRep tournament over a chunk evaluates the chunk's first
token and the midpoint of every range on its path, so the representative
alone fixes the whole path.  The rows of one (chunk, KV head) are the union of
the paths of the G query heads that share that KV head; each distinct row is
D elements once.  Prefill FLOPs count every listed 64x64 tile (block tiles and
gathered column tiles) as 2 GEMMs of 64 x 64 x D (4 * 64 * 64 * D flops),
whatever part of it the causal mask removes.
"""
from __future__ import annotations

import math

import numpy as np


def tournament_offsets(r_off: np.ndarray, lens: np.ndarray):
    """Evaluated offsets of every path: yields (head, chunk, offset) arrays.

    r_off [H, n]: representative offset inside its chunk; lens [n] chunk lengths.
    """
    H, n = r_off.shape
    a = np.zeros((H, n), np.int64)
    b = np.broadcast_to(lens - 1, (H, n)).copy()
    hh, jj = np.meshgrid(np.arange(H), np.arange(n), indexing="ij")
    out_h, out_j, out_o = [hh.ravel()], [jj.ravel()], [a.ravel().copy()]
    while True:
        act = a < b
        if not act.any():
            break
        mid = (a + b + 1) // 2
        out_h.append(hh[act])
        out_j.append(jj[act])
        out_o.append(mid[act])
        right = act & (r_off >= mid)
        left = act & ~(r_off >= mid)
        a = np.where(right, mid, a)
        b = np.where(left, mid - 1, b)
    return np.concatenate(out_h), np.concatenate(out_j), np.concatenate(out_o)


def stage_rows(reps: np.ndarray, chunk_start_pos, chunk_lists, lens: np.ndarray, G: int) -> int:
    """Distinct (chunk, KV head, row) triples one stage's tournaments read.

    reps [H_q, n] representative positions; chunk_lists: list of position
    arrays per chunk (ascending).
    """
    H_q, n = reps.shape
    r_off = np.empty((H_q, n), np.int64)
    for j in range(n):
        r_off[:, j] = np.searchsorted(chunk_lists[j], reps[:, j])
    h, j, o = tournament_offsets(r_off, lens)
    g = h // G
    Lmax = int(lens.max()) + 1
    key = (j * (H_q // G) + g) * Lmax + o
    return int(np.unique(key).size)


def decode_bytes(stage_rows_list, attended, H_kv, D, elem, T_q, H_q, extra_index_bytes=0):
    """Bytes of one decode step: tournament rows + K and V of the attended set + q/out."""
    rows = sum(stage_rows_list)
    return (rows * D * elem + attended * H_kv * D * elem * 2 + 2 * T_q * H_q * D * elem
            + extra_index_bytes)


def prefill_tile_flops(blk_cnt: np.ndarray, col_cnt: np.ndarray, D: int) -> float:
    """4 * 64 * 64 * D flops per listed tile (block tiles + ceil(columns / 64))."""
    tiles = blk_cnt.astype(np.int64).sum() + np.ceil(col_cnt.astype(np.int64) / 64.0).sum()
    return float(tiles) * 4.0 * 64 * 64 * D


def prefill_useful_flops(blk_cnt, blk_idx, col_cnt, col_idx, S: int, D: int) -> float:
    """4 * D flops per (query row, key) pair the lists make a row attend: a listed block
    before the row's own block counts 64 x 64 pairs, the diagonal block the causal
    triangle, a listed column j of query block m the rows of m at or after j; rows and
    keys past the sequence end count nothing.  Lists are [B, H, n_qblk(, max)] arrays."""
    nq = blk_cnt.shape[-1]
    m = np.arange(nq)[None, None, :]
    rows = np.minimum(64, S - 64 * m)                                 # rows of block m
    width = blk_idx.shape[-1]
    valid_b = np.arange(width)[None, None, None, :] < blk_cnt[..., None]
    n = np.where(valid_b, blk_idx, -1)
    key_w = np.clip(S - 64 * n, 0, 64)                                 # keys in block n
    below = (n >= 0) & (n < m[..., None])
    diag = (n == m[..., None])
    tri = rows * (rows + 1) // 2                                       # diagonal triangle
    pairs = (np.where(below, rows[..., None] * key_w, 0).sum() +
             np.where(diag, tri[..., None], 0).sum())
    cw = col_idx.shape[-1]
    if cw:
        valid_c = np.arange(cw)[None, None, None, :] < col_cnt[..., None]
        j = np.where(valid_c, col_idx, S)
        last = 64 * m[..., None] + rows[..., None]                     # one past the last row
        pairs += np.where(valid_c, np.clip(last - np.maximum(j, 64 * m[..., None]), 0, None), 0).sum()
    return float(pairs) * 4.0 * D


def vs_index_bytes(B, S, H_q, H_kv, D, n_vertical, elem=2) -> float:
    """Two passes over K (row statistics, then sums) + the estimate rows of Q."""
    return float(2 * B * S * H_kv * D * elem + 2 * B * 64 * H_q * D * elem)


def block_sparse_pool_bytes(B, S, H_q, H_kv, D, elem=2) -> float:
    """Block-Sparse pooling: every q and k row read once, fp32 pooled blocks written."""
    nb = -(-S // 64)
    return float(B) * (S * (H_q + H_kv) * D * elem + nb * (H_q + H_kv) * D * 4)


def causal_dense_tiles(S: int) -> int:
    n = math.ceil(S / 64)
    return n * (n + 1) // 2
