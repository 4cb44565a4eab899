"""MInference vertical-slash index and sparse causal prefill attention, in float64.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Source: "MInference 1.0: Accelerating Pre-filling for Long-Context LLMs via
Dynamic Sparse Attention" (paper-graph-ui summary of arXiv 2407.02490),
section 3.4: "The Optimization Problem" (Eq. 1, masked attention),
"Online Dynamic Index Estimation: Vertical-Slash Heads" (Alg. 2 steps 1-5)
and "Vertical-Slash Hybrid Kernel" (Alg. 4 two-way merge, Alg. 5 hybrid
block/column attention).

Readings of points the pages leave open:
  * slash offset o = query position - key position (o >= 0); the garbled
    diagonal-sum bounds are read as summing over the estimate rows i whose
    key i - o exists;
  * top-k ties -> smaller column / offset; both lists ascending;
  * Eq. 1's c = 1e5 is exact exclusion (exp(-1e5) is 0 in float64); a row
    with no attended key gives O = 0 and lse = -inf;
  * "rounding slash intersections to block boundaries": for query block m
    (nominal rows 64m .. 64m+63) a slash offset o selects every 64-aligned
    key block that the key range [64m-o, 64m+63-o] (clipped at 0) touches;
    block m then attends those whole blocks, causally masked;
  * a vertical column not inside a selected block stays a column entry;
  * nothing (no sink column, no local diagonal) is forced into the index.
"""
from __future__ import annotations

import math

import numpy as np

from .numerics import to_f64


# ---------------------------------------------------------------- estimate (Alg. 2)

def estimate_rows(S: int, last_q: int) -> np.ndarray:
    """Positions of the estimate rows: the last min(last_q, S) queries."""
    n = min(last_q, S)
    return np.arange(S - n, S, dtype=np.int64)


def approx_attention(q_rows: np.ndarray, rows: np.ndarray, K_g: np.ndarray, scale: float):
    """A~ = softmax(Q[-64:] K^T * scale + m_causal) (Alg. 2 step 1), row-wise, fp64."""
    z = scale * (q_rows @ K_g.T)
    S = K_g.shape[0]
    future = np.arange(S)[None, :] > rows[:, None]
    z[future] = -np.inf
    m = z.max(axis=1, keepdims=True)
    p = np.exp(z - m)
    return p / p.sum(axis=1, keepdims=True)


def vertical_sums(A: np.ndarray) -> np.ndarray:
    """sum_v(A~)_j = sum over the estimate rows of A~[i, j] (Alg. 2 step 2)."""
    return A.sum(axis=0)


def slash_sums(A: np.ndarray, rows: np.ndarray) -> np.ndarray:
    """sum_s(A~)_o = sum_i A~[i, p_i - o] over rows with p_i - o >= 0 (Alg. 2 step 3)."""
    S = A.shape[1]
    s = np.zeros(S)
    for i, p in enumerate(rows):
        # offsets o = 0 .. p map to keys j = p .. 0
        s[:p + 1] += A[i, p::-1]
    return s


def topk_ascending(x: np.ndarray, k: int) -> np.ndarray:
    """arg top-k (ties -> smaller index), returned in ascending index order."""
    n = len(x)
    k = min(k, n)
    order = np.lexsort((np.arange(n), -np.asarray(x, np.float64)))
    return np.sort(order[:k]).astype(np.int64)


def vs_estimate(q, k, S, H_q, H_kv, last_q, n_vertical, n_slash, scale):
    """Vertical and slash index for every head of one batch row.

    q: bf16 bits [S, H_q, D]; k: bf16 bits [S, H_kv, D].
    Returns (vertical [H_q, k_v], slash [H_q, k_s], vsum [H_q, S], ssum [H_q, S]).
    """
    G = H_q // H_kv
    rows = estimate_rows(S, last_q)
    vert, sl, vs_, ss_ = [], [], [], []
    for g in range(H_kv):
        K_g = to_f64(k[:S, g, :], "bf16")
        for h in range(g * G, (g + 1) * G):
            A = approx_attention(to_f64(q[rows, h, :], "bf16"), rows, K_g, scale)
            v = vertical_sums(A)
            s = slash_sums(A, rows)
            vert.append(topk_ascending(v, n_vertical))
            sl.append(topk_ascending(s, n_slash))
            vs_.append(v)
            ss_.append(s)
    return np.stack(vert), np.stack(sl), np.stack(vs_), np.stack(ss_)


# ---------------------------------------------------------------- conversion (Alg. 4)

def slash_blocks(slash: np.ndarray, m: int, block: int = 64) -> np.ndarray:
    """Key blocks of query block m touched by the slash lines, ascending.

    Offset o covers keys [block*m - o, block*m + block-1 - o] in this query
    block; every block-aligned key block that range touches (after clipping
    at key 0) is selected.
    """
    o = np.asarray(slash, np.int64)
    hi = block * m + block - 1 - o
    lo = np.maximum(block * m - o, 0)
    ok = hi >= 0
    return np.unique(np.concatenate([lo[ok] // block, hi[ok] // block]))


def vs_convert(vertical: np.ndarray, slash: np.ndarray, S: int, block: int = 64):
    """Two-way merge into per-query-block block lists and column lists.

    Returns (blk: list of ascending int arrays, col: list of ascending int
    arrays), one entry per query block m = 0 .. ceil(S/block)-1.  Vertical
    columns that fall inside a selected block are absorbed by it; the rest
    (up to the block's last nominal row) stay columns.
    """
    n_blk = math.ceil(S / block)
    vertical = np.asarray(vertical, np.int64)
    blk, col = [], []
    for m in range(n_blk):
        Bm = slash_blocks(slash, m, block)
        c = vertical[vertical <= block * m + block - 1]
        c = c[~np.isin(c // block, Bm)]
        blk.append(Bm)
        col.append(c)
    return blk, col


def tile_mask(blk: list, col: list, S: int, block: int = 64) -> np.ndarray:
    """Dense [S, S] boolean mask of the tiled format (small S only)."""
    M = np.zeros((S, S), bool)
    for m in range(len(blk)):
        r0, r1 = block * m, min(block * m + block, S)
        for n in blk[m]:
            M[r0:r1, block * n:min(block * n + block, S)] = True
        M[r0:r1, col[m]] = True
    return M & np.tril(np.ones((S, S), bool))


def exact_vs_mask(vertical, slash, S: int) -> np.ndarray:
    """Dense mask of the literal pattern: j in vertical or i - j in slash, j <= i."""
    i = np.arange(S)[:, None]
    j = np.arange(S)[None, :]
    M = np.isin(i - j, np.asarray(slash)) | np.isin(j, np.asarray(vertical))
    return M & (j <= i)


# ---------------------------------------------------------------- attention (Eq. 1, Alg. 5)

def block_keys(blk_m, col_m, S: int, block: int = 64) -> np.ndarray:
    """Key positions listed for one query block: whole blocks plus columns (as a set)."""
    parts = [np.arange(block * n, min(block * n + block, S)) for n in blk_m]
    parts.append(np.asarray(col_m, np.int64))
    return np.unique(np.concatenate(parts)) if parts else np.zeros(0, np.int64)


def prefill_block_attention(q, k, v, h, G, m, blk_m, col_m, S, scale, block: int = 64):
    """Masked softmax attention (Eq. 1, exact exclusion) for the rows of query block m.

    q: bf16 bits [S, H_q, D]; k, v: bf16 bits [S, H_kv, D].  Row i attends
    the listed keys j with j <= i.  Returns O [rows, D], lse [rows].
    """
    g = h // G
    rows = np.arange(block * m, min(block * m + block, S))
    keys = block_keys(blk_m, col_m, S, block)
    D = q.shape[-1]
    O = np.zeros((len(rows), D))
    lse = np.full(len(rows), -np.inf)
    if len(keys) == 0:
        return O, lse
    Q = to_f64(q[rows, h, :], "bf16")
    Kk = to_f64(k[keys, g, :], "bf16")
    Vk = to_f64(v[keys, g, :], "bf16")
    z = scale * (Q @ Kk.T)
    allowed = keys[None, :] <= rows[:, None]
    z[~allowed] = -np.inf
    has = allowed.any(axis=1)
    if not has.any():
        return O, lse
    zm = z[has]
    mx = zm.max(axis=1, keepdims=True)
    p = np.exp(zm - mx)
    l = p.sum(axis=1, keepdims=True)
    O[has] = (p @ Vk) / l
    lse[has] = mx[:, 0] + np.log(l[:, 0])
    return O, lse
