"""InfiniteHiP hierarchical chunk pruning and sparse decode attention, in float64.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Source: "InfiniteHiP: Extending Language Model Context Up to 3 Million Tokens
on a Single GPU" (paper-graph-ui summary of arXiv 2502.08910), section 3.4 (and
"Prefill Latency Details" for the chunked sparse prefill):
"Formal Mechanism of a Single Pruning Stage" (Alg. 2 steps 1-8), "The
Representative Token Selection Algorithm (SelectRep)" (Alg. 3), "Important:
Sink and Streaming Tokens Are Never Pruned" (Alg. 1 line 1), "Formal
Background: Standard Multi-Head Attention", and "Block Sparse Attention
Implementation" (decode attention over the selected keys).  The InfLLM guide
("InfLLM Guide: Training-Free Long-Context Memory for LLMs", section
"Chunk-Level Attention Scoring Engine") states the same union-of-tiers softmax
with a 1/sqrt(d) scale.

Readings of points the pages leave open (each one is also a test pin or is
marked as unpinned):
  * midpoint: round half up, i.e. mid = (a + b + 1) // 2 for 0-based (a, b);
    the tournament stops once the range holds one index (same as
    ceil(log2 L) iterations for power-of-two L);
  * branch tie -> left branch; top-K tie -> smaller chunk index;
  * the partial last chunk (|I| not a multiple of l_c) is kept as the
    formula C_j = I[j*l_c : (j+1)*l_c] implies and competes like the others;
  * selection scores are raw q.k (a positive scale does not change order);
    attention uses 1/sqrt(D);
  * all T_q query rows of a decode block share one index set and sit at the
    newest position (no causal mask inside the block);
  * the attended set is [0, min(n_sink,T)) U I U [max(n_sink, T-n_stream), T).
Parity unpinned: the tie rules and the midpoint rounding above have no
printed worked example on the pages; they are pinned only by the written
reading and by the invariants in the tests.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

from .numerics import to_f64


# ---------------------------------------------------------------- candidate range

def candidate_range(T: int, n_sink: int, n_stream: int) -> np.ndarray:
    """I^(0) = [n_sink, T - n_stream): the middle tokens, the only ones pruned.

    Sink tokens [0, n_sink) and the newest n_stream tokens bypass pruning
    ("Important: Sink and Streaming Tokens Are Never Pruned", Alg. 1 line 1).
    """
    lo, hi = n_sink, T - n_stream
    return np.arange(lo, max(lo, hi), dtype=np.int64)


def attended_set(T: int, n_sink: int, n_stream: int, I: np.ndarray) -> np.ndarray:
    """Sink tokens, the pruned selection I and the streaming window, ascending."""
    sink = np.arange(min(n_sink, T), dtype=np.int64)
    window = np.arange(max(n_sink, T - n_stream), T, dtype=np.int64)
    return np.concatenate([sink, np.asarray(I, np.int64), window])


# ---------------------------------------------------------------- one pruning stage

def chunk_partition(I: np.ndarray, L: int) -> list:
    """Alg. 2 step 3: C_j = [I[j*l_c], ..., I[(j+1)*l_c - 1]] (last chunk may be short)."""
    return [I[j * L:(j + 1) * L] for j in range(math.ceil(len(I) / L))]


def block_score(q_h: np.ndarray, key: np.ndarray) -> float:
    """max over the query rows t of the block of q_t . k (Alg. 3, sigma_j)."""
    return float(np.max(q_h @ key))


def select_rep(q_h: np.ndarray, K_g, dtype: str, C: np.ndarray, trace: list | None = None):
    """SelectRep (Alg. 3), top-1 tournament over the positions C of one chunk.

    q_h: [T_q, D] float64 query block of one head; K_g(pos) -> key row.
    Each iteration splits the current range at the rounded midpoint, scores
    the first token of each half against the query block and keeps the half
    whose first token scores higher (left on ties).  Returns the chosen
    position, its score and the number of key evaluations (two per
    iteration, as the pages count them).
    """
    a, b = 0, len(C) - 1
    evals = 0
    while a < b:
        mid = (a + b + 1) // 2
        s1 = block_score(q_h, to_f64(K_g[C[a]], dtype))
        s2 = block_score(q_h, to_f64(K_g[C[mid]], dtype))
        evals += 2
        if trace is not None:
            trace.append((a, mid, b, s1, s2))
        if s2 > s1:
            a = mid
        else:
            b = mid - 1
    r = int(C[a])
    return r, block_score(q_h, to_f64(K_g[r], dtype)), evals


def select_rep_all(q: np.ndarray, K: np.ndarray, dtype: str, chunks: list, G: int):
    """SelectRep for every (query head h, chunk j) of one batch row.

    Same steps as ``select_rep``, run for all chunks and heads side by side
    (the chunks are independent).  q: [T_q, H_q, D] float64; K: raw
    [T, H_kv, D].  Head h reads KV head h // G.  Returns reps [H_q, n]
    (positions) and rho [H_q, n] (the representative's block score).
    """
    T_q, H_q, D = q.shape
    n = len(chunks)
    if n == 0:
        return np.zeros((H_q, 0), np.int64), np.zeros((H_q, 0))
    Lmax = max(len(c) for c in chunks)
    lens = np.array([len(c) for c in chunks], np.int64)
    pos = np.empty((n, Lmax), np.int64)
    for j, c in enumerate(chunks):
        pos[j, :len(c)] = c
        pos[j, len(c):] = c[-1]
    g_of_h = np.arange(H_q) // G
    cols = np.arange(n)[None, :]

    def score(idx):  # idx [H_q, n] offsets inside the chunks
        p = pos[cols, idx]
        keys = to_f64(K[p, g_of_h[:, None]], dtype)          # [H_q, n, D]
        return np.einsum("thd,hnd->thn", q, keys).max(axis=0)

    a = np.zeros((H_q, n), np.int64)
    b = np.broadcast_to(lens - 1, (H_q, n)).copy()
    while True:
        active = a < b
        if not active.any():
            break
        mid = np.where(active, (a + b + 1) // 2, a)
        s1 = score(a)
        s2 = score(mid)
        right = active & (s2 > s1)
        left = active & ~(s2 > s1)
        a = np.where(right, mid, a)
        b = np.where(left, mid - 1, b)
    return pos[cols, a], score(a)


def chunk_scores(rho: np.ndarray) -> np.ndarray:
    """Alg. 2 step 5: s_j = max over heads (and query rows, already in rho)."""
    return rho.max(axis=0) if rho.size else np.zeros(rho.shape[1])


def topk_chunks(s: np.ndarray, K: int) -> np.ndarray:
    """Alg. 2 step 6: indices of the K largest scores (ties -> smaller index), ascending.

    All chunks are kept when there are at most K of them.
    """
    n = len(s)
    if n <= K:
        return np.arange(n, dtype=np.int64)
    order = np.lexsort((np.arange(n), -np.asarray(s, np.float64)))
    return np.sort(order[:K]).astype(np.int64)


def assemble(chunks: list, kept: np.ndarray) -> np.ndarray:
    """Alg. 2 step 7: I' = union of the kept chunks' tokens (ascending chunk order)."""
    if len(kept) == 0:
        return np.zeros(0, np.int64)
    return np.concatenate([chunks[j] for j in kept]).astype(np.int64)


@dataclass
class StageResult:
    L: int
    K: int
    I_in: np.ndarray
    chunks: list
    reps: np.ndarray     # [H_q, n] representative positions
    rho: np.ndarray      # [H_q, n] representative scores
    s: np.ndarray        # [n] chunk scores
    kept: np.ndarray     # kept chunk ids, ascending
    I_out: np.ndarray    # assembled token list, ascending


def pruning_stage(q, K, dtype, I, L, keep, G) -> StageResult:
    """One pruning stage S^(i) = (b_q, l_c, k) applied to the retained list I."""
    Kc = keep // L                      # K^(i) = k^(i) / l_c^(i)
    chunks = chunk_partition(np.asarray(I, np.int64), L)
    reps, rho = select_rep_all(q, K, dtype, chunks, G)
    s = chunk_scores(rho)
    kept = topk_chunks(s, Kc)
    return StageResult(L, Kc, np.asarray(I, np.int64), chunks, reps, rho, s, kept,
                       assemble(chunks, kept))


def hip_select(q, K, dtype, T, chunk, keep, n_sink, n_stream, G):
    """Run all pruning stages for one batch row; return (stage results, final I)."""
    I = candidate_range(T, n_sink, n_stream)
    stages = []
    for L, k in zip(chunk, keep):
        st = pruning_stage(q, K, dtype, I, L, k, G)
        stages.append(st)
        I = st.I_out
    return stages, I


# ---------------------------------------------------------------- mask caching

def refresh_schedule(step: int, n_refresh) -> list:
    """Which stages recompute their output at decoding step `step` (counted from 0).

    Section 3.4 "Sparse Attention Mask Caching (Temporal Locality Exploitation)":
    stage i has a refresh interval n_refresh[i]; its stored output is recomputed when
    the step counter is a multiple of that interval and reused unchanged otherwise.
    """
    return [step % int(r) == 0 for r in n_refresh]


def hip_select_cached(q, K, dtype, T, chunk, keep, n_sink, n_stream, G, refresh, cache):
    """One decoding step of the pruning pipeline with per-stage mask caching, one row.

    Same section as refresh_schedule.  `cache[i]` holds stage i's stored output list
    (None before it first ran) and is updated in place for the stages with
    refresh[i] true; the others are skipped.  A recomputed stage 0 prunes the
    candidate range of the current context length T; a recomputed stage i > 0 prunes
    cache[i-1] as it stands at that point of the step (recomputed just before, or
    cached).  Returns ({stage: StageResult} for the recomputed stages, cache[-1]).
    """
    ran = {}
    for i, (L, k) in enumerate(zip(chunk, keep)):
        if not refresh[i]:
            continue
        if i == 0:
            I = candidate_range(T, n_sink, n_stream)
        else:
            if cache[i - 1] is None:
                raise ValueError(f"stage {i} refreshed before stage {i - 1} ever ran")
            I = cache[i - 1]
        st = pruning_stage(q, K, dtype, I, L, k, G)
        cache[i] = st.I_out
        ran[i] = st
    return ran, cache[-1]


# ---------------------------------------------------------------- sparse prefill

def prefill_block_len(S: int, m: int, b_q: int = 64) -> int:
    """Keys a query block sees: those up to its last row, T_m = min(S, b_q (m + 1)).

    Section 3.4 "Formal Mechanism of a Single Pruning Stage", step 1 (query blocks of
    b_q = 64 rows sharing one mask); prefill is causal, so block m prunes the keys
    before its end (the chunked prefill of "Prefill Latency Details" processes the
    blocks 32K queries at a time over the same keys).
    """
    return min(S, b_q * (m + 1))


def hip_prefill_select(q, K, dtype, S, chunk, keep, n_sink, n_stream, G, b_q: int = 64):
    """Every query block's final selection: hip_select with the block's rows as the
    query block and T = T_m.  q: float64 [S, H_q, D]; returns a list of index arrays."""
    out = []
    for m in range(math.ceil(S / b_q)):
        rows = slice(b_q * m, min(S, b_q * (m + 1)))
        _, I = hip_select(q[rows], K, dtype, prefill_block_len(S, m, b_q), chunk, keep,
                          n_sink, n_stream, G)
        out.append(I)
    return out


def prefill_attention(q, K, V, dtype, S, I_blocks, n_sink, n_stream, scale, G, b_q: int = 64,
                      blocks=None):
    """Causal attention of each query block's rows over sink + its selection + its
    window ("Block Sparse Attention Implementation", prefill), fp64.

    Row i of block m attends the keys j <= i of attended_set(T_m, n_sink, n_stream, I_m).
    Returns {m: (O [rows, H_q, D], lse [rows, H_q])} for the blocks asked (all by default).
    """
    res = {}
    H_q, D = q.shape[1], q.shape[2]
    for m in (range(len(I_blocks)) if blocks is None else blocks):
        r0, r1 = b_q * m, min(S, b_q * (m + 1))
        A = attended_set(prefill_block_len(S, m, b_q), n_sink, n_stream, I_blocks[m])
        O = np.zeros((r1 - r0, H_q, D))
        lse = np.full((r1 - r0, H_q), -np.inf)
        for h in range(H_q):
            keys = to_f64(K[A, h // G], dtype)
            vals = to_f64(V[A, h // G], dtype)
            z = scale * (q[r0:r1, h, :] @ keys.T)
            z[A[None, :] > np.arange(r0, r1)[:, None]] = -np.inf
            mx = z.max(axis=1, keepdims=True)
            p = np.exp(z - mx)
            l = p.sum(axis=1, keepdims=True)
            O[:, h, :] = (p @ vals) / l
            lse[:, h] = mx[:, 0] + np.log(l[:, 0])
        res[m] = (O, lse)
    return res


# ---------------------------------------------------------------- attention

def decode_attention(q, K, V, dtype, A, scale, G):
    """softmax(scale * q K_A^T) V_A for every query row and head (fp64).

    The masked-softmax of the MInference summary's Eq. 1 with the mask
    constant taken as exact exclusion: only the keys in A take part.
    Returns O [T_q, H_q, D] and lse [T_q, H_q] (natural log); an empty A
    gives O = 0 and lse = -inf.
    """
    T_q, H_q, D = q.shape
    O = np.zeros((T_q, H_q, D))
    lse = np.full((T_q, H_q), -np.inf)
    A = np.asarray(A, np.int64)
    if len(A) == 0:
        return O, lse
    for h in range(H_q):
        g = h // G
        keys = to_f64(K[A, g], dtype)
        vals = to_f64(V[A, g], dtype)
        z = scale * (q[:, h, :] @ keys.T)
        m = z.max(axis=1, keepdims=True)
        p = np.exp(z - m)
        l = p.sum(axis=1, keepdims=True)
        O[:, h, :] = (p @ vals) / l
        lse[:, h] = m[:, 0] + np.log(l[:, 0])
    return O, lse
