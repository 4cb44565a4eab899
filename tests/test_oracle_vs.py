"""Pins for the fp64 vertical-slash / prefill oracle (CPU only)."""
import math

import numpy as np
import pytest
import torch

from oracle import vs
from oracle.numerics import to_f64
from synth import prefill_case


def _tiny(S=300, H_q=4, H_kv=2, D=32, seed=21, **kw):
    return prefill_case("tiny", S=S, H_q=H_q, H_kv=H_kv, D=D, seed=seed, **kw)


def test_approx_attention_matches_torch_softmax():
    c = _tiny()
    rows = vs.estimate_rows(c.S, c.last_q)
    K = to_f64(c.k[0, :, 0], "bf16")
    Q = to_f64(c.q[0, rows, 0], "bf16")
    A = vs.approx_attention(Q, rows, K, c.scale)
    z = torch.from_numpy(Q @ K.T * c.scale)
    z = z.masked_fill(torch.arange(c.S)[None, :] > torch.from_numpy(rows)[:, None], float("-inf"))
    np.testing.assert_allclose(A, torch.softmax(z, -1).numpy(), rtol=0, atol=1e-15)


def test_sums_conserve_mass_and_match_bruteforce():
    c = _tiny(S=150)
    rows = vs.estimate_rows(c.S, c.last_q)
    A = vs.approx_attention(to_f64(c.q[0, rows, 1], "bf16"), rows,
                            to_f64(c.k[0, :, 0], "bf16"), c.scale)
    v = vs.vertical_sums(A)
    s = vs.slash_sums(A, rows)
    assert abs(v.sum() - len(rows)) < 1e-12 and abs(s.sum() - len(rows)) < 1e-12
    # brute force from the key side: entry (i, j) lies on slash p_i - j
    s_bf = np.zeros(c.S)
    v_bf = np.zeros(c.S)
    for i, p in enumerate(rows):
        for j in range(c.S):
            v_bf[j] += A[i, j]
            if j <= p:
                s_bf[p - j] += A[i, j]
    np.testing.assert_allclose(s, s_bf, rtol=0, atol=1e-14)
    np.testing.assert_allclose(v, v_bf, rtol=0, atol=1e-14)


def test_short_sequence_uses_all_rows():
    rows = vs.estimate_rows(40, 64)
    assert np.array_equal(rows, np.arange(40))


def test_topk_ascending_pairwise():
    rng = np.random.default_rng(2)
    for n in range(1, 10):
        for k in range(1, n + 1):
            x = rng.integers(0, 4, size=n).astype(float)
            t = vs.topk_ascending(x, k)
            assert list(t) == sorted(t) and len(t) == k
            ts = set(t.tolist())
            for i in ts:
                for j in set(range(n)) - ts:
                    assert x[i] > x[j] or (x[i] == x[j] and i < j)


@pytest.mark.parametrize("block", [4, 8])
def test_slash_blocks_match_elementwise_definition(block):
    rng = np.random.default_rng(block)
    S = 13 * block + 3
    for _ in range(20):
        slash = np.sort(rng.choice(S, size=7, replace=False))
        for m in range(math.ceil(S / block)):
            want = set()
            for o in slash:
                for x in range(block * m - o, block * m + block - o):
                    if x >= 0:
                        want.add(x // block)
            got = vs.slash_blocks(slash, m, block)
            assert sorted(want) == list(got)


def test_tile_mask_contains_exact_mask():
    rng = np.random.default_rng(9)
    S, block = 200, 16
    for _ in range(10):
        vert = np.sort(rng.choice(S, 9, replace=False))
        sl = np.sort(rng.choice(S, 11, replace=False))
        blk, col = vs.vs_convert(vert, sl, S, block)
        M = vs.tile_mask(blk, col, S, block)
        E = vs.exact_vs_mask(vert, sl, S)
        assert np.all(M[E])
        for m in range(len(blk)):
            # columns never fall inside a selected block and are ascending
            assert not np.any(np.isin(col[m] // block, blk[m]))
            assert np.all(np.diff(col[m]) > 0) and np.all(np.diff(blk[m]) > 0)
            assert np.all(blk[m] <= m)


def test_all_offsets_give_dense_causal_attention():
    """k_s = S selects every offset -> tiled mask == causal mask -> SDPA(is_causal)."""
    c = _tiny(S=200, H_q=2, H_kv=1, D=16)
    S = c.S
    blk, col = vs.vs_convert(np.zeros(0, np.int64), np.arange(S), S)
    assert np.array_equal(vs.tile_mask(blk, col, S), np.tril(np.ones((S, S), bool)))
    Q = torch.from_numpy(to_f64(c.q[0], "bf16")).permute(1, 0, 2)
    K = torch.from_numpy(to_f64(c.k[0], "bf16")).permute(1, 0, 2).repeat_interleave(2, 0)
    V = torch.from_numpy(to_f64(c.v[0], "bf16")).permute(1, 0, 2).repeat_interleave(2, 0)
    ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V, is_causal=True)
    for h in range(2):
        for m in range(len(blk)):
            O, lse = vs.prefill_block_attention(c.q[0], c.k[0], c.v[0], h, 2, m, blk[m],
                                                col[m], S, c.scale)
            r0 = 64 * m
            np.testing.assert_allclose(O, ref[h, r0:r0 + len(O)].numpy(), rtol=0, atol=1e-12)


def test_prefill_exact_exclusion_matches_eq1_constant():
    c = _tiny(S=130, H_q=1, H_kv=1, D=16)
    rng = np.random.default_rng(1)
    vert = np.sort(rng.choice(130, 5, replace=False))
    sl = np.array([0, 3, 70])
    blk, col = vs.vs_convert(vert, sl, 130)
    M = vs.tile_mask(blk, col, 130)
    Q = to_f64(c.q[0, :, 0], "bf16")
    K = to_f64(c.k[0, :, 0], "bf16")
    V = to_f64(c.v[0, :, 0], "bf16")
    z = torch.from_numpy(Q @ K.T * c.scale - 1e5 * (1 - M))
    ref = torch.softmax(z, -1).numpy() @ V
    for m in range(len(blk)):
        O, _ = vs.prefill_block_attention(c.q[0], c.k[0], c.v[0], 0, 1, m, blk[m], col[m],
                                          130, c.scale)
        np.testing.assert_allclose(O, ref[64 * m:64 * m + len(O)], rtol=0, atol=1e-12)


def test_empty_rows_give_zero_output():
    c = _tiny(S=70, H_q=1, H_kv=1, D=16)
    # only column 65 listed for block 1 -> rows 64..64 have nothing (65 > 64)
    O, lse = vs.prefill_block_attention(c.q[0], c.k[0], c.v[0], 0, 1, 1, [], [65], 70, c.scale)
    assert np.all(O[0] == 0) and lse[0] == -np.inf
    assert np.isfinite(lse[1:]).all()


def test_planted_structure_is_recovered():
    """Generator self-check: planted columns and near offsets show up in the estimate."""
    c = prefill_case("plant", S=4096, H_q=4, H_kv=2, D=128, seed=5, n_vertical=100,
                     n_slash=400, n_far_offsets=2)
    vert, sl, _, _ = vs.vs_estimate(c.q[0], c.k[0], c.S, c.H_q, c.H_kv, c.last_q,
                                    c.n_vertical, c.n_slash, c.scale)
    for h in range(c.H_q):
        assert np.isin(c.planted_columns, vert[h]).mean() >= 0.9
        assert np.isin(c.planted_offsets, sl[h]).mean() >= 0.9


def test_page_cost_formulas(golden):
    g = golden["vs_estimate_flops_1m"]
    # one multiply-add per (estimate row, key, dim), as the page counts it
    assert abs(g["last_q"] * g["S"] * g["d"] - g["flops"]) <= g["rel_tol"] * g["flops"]
    b = golden["block_sparse_speedup_1m"]
    assert abs(b["S"] / (2 * b["B"] * b["k_b"]) - b["speedup_approx"]) <= b["rel_tol"] * 78


def test_useful_flop_count_matches_the_tile_mask():
    """The bench's count of attended (row, key) pairs equals the dense mask's count."""
    from dynamic_sparse_attention_gb300 import accounting
    for S in (300, 256, 97):
        rng = np.random.default_rng(S)
        nq = (S + 63) // 64
        blk, col = [], []
        for m in range(nq):
            b = np.sort(rng.choice(m + 1, size=int(rng.integers(0, m + 2)), replace=False))
            covered = np.zeros(S, bool)
            for n in b:
                covered[64 * n:min(S, 64 * n + 64)] = True
            cand = np.nonzero(~covered[:min(S, 64 * m + 64)])[0]
            c = np.sort(rng.choice(cand, size=min(5, len(cand)), replace=False)) if len(cand) else np.zeros(0, int)
            blk.append(b)
            col.append(c)
        M = vs.tile_mask(blk, col, S)
        bc = np.array([[[len(b) for b in blk]]])
        cc = np.array([[[len(c) for c in col]]])
        bi = np.full((1, 1, nq, nq), -1)
        ci = np.full((1, 1, nq, 5), -1)
        for m in range(nq):
            bi[0, 0, m, :len(blk[m])] = blk[m]
            ci[0, 0, m, :len(col[m])] = col[m]
        assert accounting.prefill_useful_flops(bc, bi, cc, ci, S, 1) == 4.0 * M.sum()
