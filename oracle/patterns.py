"""MInference A-shape and Block-Sparse head patterns as per-query-block key-block lists,
in float64.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Source: "MInference 1.0: Accelerating Pre-filling for Long-Context LLMs via Dynamic
Sparse Attention" (paper-graph-ui summary of arXiv 2407.02490): "The Three Sparse
Patterns: Geometry and GPU Implications" (A-Shape Pattern), "Sparse GPU Kernel
Implementations (Appendix C.4)" (A-Shape Kernel: initial blocks plus a diagonal band
of blocks) and "Online Dynamic Index Estimation: Block-Sparse Heads (Algorithm 3)"
steps 1-4 (mean pooling, block-level causal softmax, top-k_b blocks per query block).
Both patterns feed the same block-sparse attention as the vertical-slash index, with
no column entries; `oracle.vs.prefill_block_attention` is the attention.

Readings of points the pages leave open:
  * A-shape at block granularity: query block m attends key block j <= m iff
    j < n_global / 64 (the initial tokens) or m - j < n_local / 64 (the local band,
    diagonal block included); rows are causal inside the diagonal block.  n_global
    and n_local are token counts, multiples of the block size (the pages' 1024 and
    4096 give 16 and 64 blocks);
  * mean pooling averages 64 consecutive tokens; a ragged last block averages the
    tokens it has;
  * the block-level causal mask removes key blocks after the query block (j > m);
    the diagonal block stays, as every query attends at least to itself;
  * top-k_b per row of the block-level softmax, ties -> smaller block index; a row
    with at most k_b unmasked blocks keeps all of them; lists ascending;
  * GQA: query head h pools its own queries and scores them against the pooled keys
    of KV head h // G.
"""
from __future__ import annotations

import math

import numpy as np

from .numerics import to_f64


# ---------------------------------------------------------------- A-shape

def ashape_blocks(m: int, n_global: int, n_local: int, block: int = 64) -> np.ndarray:
    """Key blocks of query block m: the initial blocks and the band ending at m."""
    if n_global % block or n_local % block:
        raise ValueError("n_global and n_local must be multiples of the block size")
    j = np.arange(m + 1, dtype=np.int64)
    keep = (j < n_global // block) | (m - j < n_local // block)
    return j[keep]


def ashape_lists(S: int, n_global: int, n_local: int, block: int = 64) -> list:
    return [ashape_blocks(m, n_global, n_local, block) for m in range(math.ceil(S / block))]


# ---------------------------------------------------------------- Block-Sparse (Alg. 3)

def mean_pool(X: np.ndarray, block: int = 64) -> np.ndarray:
    """Step 1: the mean of every `block` consecutive rows of X [S, D] (last block ragged)."""
    S = X.shape[0]
    n = math.ceil(S / block)
    out = np.empty((n,) + X.shape[1:])
    for j in range(n):
        out[j] = X[block * j:min(block * j + block, S)].mean(axis=0)
    return out


def block_attention(q_h: np.ndarray, k_g: np.ndarray, scale: float, block: int = 64) -> np.ndarray:
    """Step 2: A~ = softmax(Q~ K~^T * scale + causal block mask), [n, n], one query head.

    q_h [S, D] and k_g [S, D] in float64; masked entries are exactly 0.
    """
    Qp = mean_pool(q_h, block)
    Kp = mean_pool(k_g, block)
    z = scale * (Qp @ Kp.T)
    n = z.shape[0]
    z[np.triu(np.ones((n, n), bool), 1)] = -np.inf
    z = z - z.max(axis=1, keepdims=True)
    p = np.exp(z)
    return p / p.sum(axis=1, keepdims=True)


def topk_row(a: np.ndarray, m: int, k_b: int) -> np.ndarray:
    """Step 3 on row m: the k_b largest of a[0..m] (ties -> smaller index), ascending."""
    cand = np.arange(m + 1)
    if k_b >= m + 1:
        return cand.astype(np.int64)
    order = np.lexsort((cand, -a[:m + 1]))
    return np.sort(order[:k_b]).astype(np.int64)


def block_sparse_lists(q, k, h: int, G: int, k_b: int, scale: float, block: int = 64):
    """Steps 1-4 for one query head of one batch row: (key-block lists per query
    block, A~).  q: bf16 bits [S, H_q, D]; k: bf16 bits [S, H_kv, D]."""
    A = block_attention(to_f64(q[:, h, :], "bf16"), to_f64(k[:, h // G, :], "bf16"), scale, block)
    return [topk_row(A[m], m, k_b) for m in range(A.shape[0])], A
