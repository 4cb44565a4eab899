"""Pins for the fp64 A-shape / Block-Sparse oracle (CPU only)."""
import itertools
import math

import numpy as np
import torch

from oracle import patterns, vs
from oracle.numerics import to_f64
from synth import prefill_case


def _tiny(S=300, H_q=2, H_kv=1, D=16, seed=61):
    return prefill_case("tiny", S=S, H_q=H_q, H_kv=H_kv, D=D, seed=seed)


def _sdpa_causal(c, h):
    Q = torch.from_numpy(to_f64(c.q[0, :, h], "bf16"))[None]
    K = torch.from_numpy(to_f64(c.k[0, :, h // c.G], "bf16"))[None]
    V = torch.from_numpy(to_f64(c.v[0, :, h // c.G], "bf16"))[None]
    return torch.nn.functional.scaled_dot_product_attention(Q, K, V, is_causal=True)[0].numpy()


# ------------------------------------------------------------ A-shape

def test_ashape_page_counts(golden):
    g = golden["ashape_1m"]
    m = 10000
    blk = patterns.ashape_blocks(m, g["n_global"], g["n_local"], g["block"])
    assert np.sum(blk < g["initial_blocks"]) == g["initial_blocks"]
    assert np.sum(blk > m - g["band_blocks"]) == g["band_blocks"]
    assert len(blk) == g["initial_blocks"] + g["band_blocks"]
    density = len(blk) * g["block"] / g["S"]
    assert abs(density - g["density_approx"]) <= g["rel_tol"] * g["density_approx"]


def test_ashape_keys_per_row_closed_form():
    """Row i of query block m >= n_g + n_l attends n_global initial keys, the
    n_local/64 - 1 full blocks before its own and the i - 64m + 1 keys of its own."""
    S, ng, nl = 2000, 128, 256
    lists = patterns.ashape_lists(S, ng, nl)
    M = vs.tile_mask(lists, [np.zeros(0, np.int64)] * len(lists), S)
    for i in range(64 * 6, S, 37):
        m = i // 64
        assert M[i].sum() == ng + (nl - 64) + (i - 64 * m + 1)
        assert M[i, :ng].all() and not M[i, ng:64 * (m - nl // 64 + 1)].any()
    for m, blk in enumerate(lists):
        assert np.all(np.diff(blk) > 0) and blk[-1] == m


def test_ashape_covering_everything_is_dense_causal():
    c = _tiny(S=200)
    lists = patterns.ashape_lists(c.S, 64, 256)
    ref = _sdpa_causal(c, 1)
    for m, blk in enumerate(lists):
        O, _ = vs.prefill_block_attention(c.q[0], c.k[0], c.v[0], 1, c.G, m, blk, [], c.S,
                                          c.scale)
        np.testing.assert_allclose(O, ref[64 * m:64 * m + len(O)], rtol=0, atol=1e-12)


# ------------------------------------------------------------ Block-Sparse (Alg. 3)

def test_block_sparse_page_counts(golden):
    g = golden["block_sparse_1m"]
    X = np.ones((g["S"], 1))
    n = patterns.mean_pool(X, g["block"]).shape[0]
    assert n == g["pooled_rows"]
    est = n * n * g["d"]   # multiply-adds of Q~ K~^T per head
    assert abs(est - g["estimate_flops_per_head"]) <= g["rel_tol"] * g["estimate_flops_per_head"]
    # tiles attended with k_b per row and the block-causal mask vs the page's S*k_b/64
    tiles = sum(min(g["k_b"], m + 1) for m in range(n))
    assert abs(tiles - g["S"] * g["k_b"] / g["block"]) <= g["rel_tol"] * tiles


def test_mean_pooling_commutes_with_the_product():
    """Q~ K~^T equals the 64x64 block means of Q K^T (the page's commutativity remark),
    ragged last block included."""
    rng = np.random.default_rng(3)
    S, D = 200, 8
    Q, K = rng.standard_normal((S, D)), rng.standard_normal((S, D))
    P = Q @ K.T
    n = math.ceil(S / 64)
    want = np.empty((n, n))
    for a in range(n):
        for b in range(n):
            want[a, b] = P[64 * a:64 * a + 64, 64 * b:64 * b + 64].mean()
    got = patterns.mean_pool(Q) @ patterns.mean_pool(K).T
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)
    # full blocks: the library's average pooling
    Qt = torch.from_numpy(Q[:192].T[None])
    np.testing.assert_allclose(patterns.mean_pool(Q[:192]),
                               torch.nn.functional.avg_pool1d(Qt, 64)[0].numpy().T, atol=1e-14)


def test_block_attention_matches_torch_softmax():
    c = _tiny(S=640)
    q = to_f64(c.q[0, :, 0], "bf16")
    k = to_f64(c.k[0, :, 0], "bf16")
    A = patterns.block_attention(q, k, c.scale)
    Qp = torch.nn.functional.avg_pool1d(torch.from_numpy(q.T[None]), 64)[0].T
    Kp = torch.nn.functional.avg_pool1d(torch.from_numpy(k.T[None]), 64)[0].T
    z = (Qp @ Kp.T) * c.scale
    z = z.masked_fill(torch.triu(torch.ones(10, 10, dtype=torch.bool), 1), float("-inf"))
    np.testing.assert_allclose(A, torch.softmax(z, -1).numpy(), rtol=0, atol=1e-15)
    assert np.allclose(A.sum(axis=1), 1.0) and np.all(np.triu(A, 1) == 0)


def test_topk_row_matches_exhaustive_subsets():
    rng = np.random.default_rng(4)
    for _ in range(40):
        n = int(rng.integers(1, 8))
        a = rng.integers(0, 3, size=n).astype(np.float64)   # many ties
        m = n - 1
        for k_b in range(1, n + 2):
            if k_b >= n:
                assert list(patterns.topk_row(a, m, k_b)) == list(range(n))
                continue
            best = min(itertools.combinations(range(n), k_b), key=lambda s: (-a[list(s)].sum(), s))
            assert list(patterns.topk_row(a, m, k_b)) == list(best)


def test_block_sparse_lists_shape_and_dense_case():
    c = _tiny(S=333, H_q=4, H_kv=2, D=16)
    lists, A = patterns.block_sparse_lists(c.q[0], c.k[0], 3, c.G, 2, c.scale)
    for m, blk in enumerate(lists):
        assert len(blk) == min(2, m + 1) and np.all(blk <= m) and np.all(np.diff(blk) > 0)
    # k_b >= every block: dense causal attention
    lists, _ = patterns.block_sparse_lists(c.q[0], c.k[0], 3, c.G, 100, c.scale)
    ref = _sdpa_causal(c, 3)
    for m, blk in enumerate(lists):
        O, _ = vs.prefill_block_attention(c.q[0], c.k[0], c.v[0], 3, c.G, m, blk, [], c.S,
                                          c.scale)
        np.testing.assert_allclose(O, ref[64 * m:64 * m + len(O)], rtol=0, atol=1e-12)


def test_block_sparse_finds_a_planted_block():
    """Keys of block 3 made equal to the mean query of block 9 (scaled up): row 9 keeps
    block 3 with k_b = 2 (the diagonal or another block is the second)."""
    c = _tiny(S=64 * 12, H_q=1, H_kv=1, D=16)
    q = to_f64(c.q[0, :, 0], "bf16")
    mean_q9 = q[64 * 9:64 * 10].mean(axis=0)
    k = c.k.copy()
    bits = ((8.0 * mean_q9).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    k[0, 64 * 3:64 * 4, 0] = bits
    lists, _ = patterns.block_sparse_lists(c.q[0], k[0], 0, 1, 2, c.scale)
    assert 3 in lists[9]
