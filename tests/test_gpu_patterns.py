"""GPU parity of the MInference A-shape and Block-Sparse index builders, and of the
prefill attention over their lists, against the fp64 oracle."""
import numpy as np
import pytest
import torch

import dynamic_sparse_attention_gb300 as dsa
from dynamic_sparse_attention_gb300 import _build
from oracle import patterns, vs
from oracle.numerics import to_f64
from parity import attention_errors, check_topk_list, to_dev
from synth import prefill_case

pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS = 1e-2, 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    _build.build()
    dsa.load()


@pytest.fixture(autouse=True)
def _no_device_errors():
    yield
    torch.cuda.synchronize()
    assert dsa.device_error() == 0


def _dev(c):
    return to_dev(c.q, "bf16"), to_dev(c.k, "bf16"), to_dev(c.v, "bf16")


def _lists(idx, b, h, m):
    n = int(idx["blk_cnt"][b, h, m])
    return idx["blk_idx"][b, h, m, :n].cpu().numpy()


def _check_attention(c, idx, out, lse, triples):
    o = out.float().cpu().numpy()
    lse_g = lse.cpu().numpy()
    for (b, h, m) in triples:
        O64, l64 = vs.prefill_block_attention(c.q[b], c.k[b], c.v[b], h, c.G, m,
                                              _lists(idx, b, h, m), [], c.S, c.scale)
        r0 = 64 * m
        mx, mn = attention_errors(o[b, r0:r0 + len(O64), h], O64)
        assert mx <= MAX_ABS and mn <= MEAN_ABS, f"(b={b}, h={h}, m={m}): max {mx:.3e} mean {mn:.3e}"
        fin = np.isfinite(l64)
        lg = lse_g[b, h, r0:r0 + len(O64)]
        assert np.array_equal(fin, np.isfinite(lg))
        assert np.abs(lg[fin] - l64[fin]).max(initial=0) <= 1e-3


# ------------------------------------------------------------ A-shape

@pytest.mark.parametrize("S,ng,nl", [(1000, 128, 256), (64, 0, 64), (700, 640, 64), (300, 1024, 4096),
                                     (5000, 0, 0)])
def test_ashape_lists_exact(S, ng, nl):
    c = prefill_case("ashape", B=2, S=S, H_q=4, H_kv=2, D=64, seed=70)
    q, k, _ = _dev(c)
    idx = dsa.ashape_index_build(q, k, n_global=ng, n_local=nl)
    torch.cuda.synchronize()
    want = patterns.ashape_lists(S, ng, nl)
    assert int(idx["col_cnt"].abs().sum()) == 0
    for b in range(2):
        for h in range(4):
            for m, w in enumerate(want):
                assert np.array_equal(_lists(idx, b, h, m), w), (b, h, m)


@pytest.mark.parametrize("D,G", [(128, 4), (64, 1)])
def test_ashape_attention_parity(D, G):
    c = prefill_case("ashape_attn", S=4100, H_q=2 * G, H_kv=2, D=D, seed=71)
    q, k, v = _dev(c)
    idx = dsa.ashape_index_build(q, k, n_global=256, n_local=512)
    out, lse = dsa.sparse_attn_prefill(q, k, v, idx["blk_cnt"], idx["blk_idx"], idx["col_cnt"], None)
    torch.cuda.synchronize()
    nq = (c.S + 63) // 64
    _check_attention(c, idx, out, lse, [(0, h, m) for h in range(c.H_q) for m in (0, 3, 4, 9, 40, nq - 1)])


# ------------------------------------------------------------ Block-Sparse

def _check_block_sparse(c, idx, k_b, heads, rows=None):
    """Pooled blocks and logits against fp64, the kept lists against the top-k rule on
    the GPU's own logits exactly and against the fp64 softmax outside the tie band."""
    qp = idx["q_pool"].cpu().numpy()
    kp = idx["k_pool"].cpu().numpy()
    sc = idx["scores"].cpu().numpy()
    nq = qp.shape[2]
    for b in range(c.B):
        for g in range(c.H_kv):
            k64 = patterns.mean_pool(to_f64(c.k[b, :, g], "bf16"))
            np.testing.assert_allclose(kp[b, g], k64, rtol=1e-5, atol=1e-6)
        for h in heads:
            q64 = patterns.mean_pool(to_f64(c.q[b, :, h], "bf16"))
            np.testing.assert_allclose(qp[b, h], q64, rtol=1e-5, atol=1e-6)
            _, A = patterns.block_sparse_lists(c.q[b], c.k[b], h, c.G, k_b, c.scale)
            k64 = patterns.mean_pool(to_f64(c.k[b, :, h // c.G], "bf16"))
            z64 = c.scale * (q64 @ k64.T)
            mag = c.scale * (np.abs(q64) @ np.abs(k64).T)
            for m in (range(nq) if rows is None else rows):
                s32 = sc[b, h, m, :m + 1]
                assert np.all(np.abs(s32 - z64[m, :m + 1]) <= 1e-5 * mag[m, :m + 1] + 1e-6)
                check_topk_list(s32, A[m, :m + 1], min(k_b, m + 1), _lists(idx, b, h, m), floor=1e-9)


@pytest.mark.parametrize("S,D,G,k_b", [(1000, 128, 4, 5), (700, 64, 1, 3), (64, 128, 2, 1),
                                       (2000, 128, 8, 40), (333, 64, 2, 100)])
def test_block_sparse_small_full_parity(S, D, G, k_b):
    c = prefill_case("bs", B=2, S=S, H_q=2 * G, H_kv=2, D=D, seed=72 + S)
    q, k, v = _dev(c)
    idx = dsa.block_sparse_index_build(q, k, k_b=k_b, debug=True)
    out, lse = dsa.sparse_attn_prefill(q, k, v, idx["blk_cnt"], idx["blk_idx"], idx["col_cnt"], None)
    torch.cuda.synchronize()
    assert int(idx["col_cnt"].abs().sum()) == 0
    _check_block_sparse(c, idx, k_b, range(c.H_q))
    nq = (S + 63) // 64
    _check_attention(c, idx, out, lse, [(b, h, m) for b in range(2) for h in range(c.H_q)
                                        for m in sorted({0, nq // 2, nq - 1})])


def test_block_sparse_ties_go_to_the_smaller_block():
    """Every key block identical: all logits of a row tie, so row m keeps blocks 0..k_b-1."""
    c = prefill_case("bs_ties", S=64 * 20, H_q=2, H_kv=1, D=64, seed=73)
    c.k[0] = np.tile(c.k[0, :64], (20, 1, 1))
    q, k, _ = _dev(c)
    idx = dsa.block_sparse_index_build(q, k, k_b=4)
    torch.cuda.synchronize()
    for m in range(20):
        assert np.array_equal(_lists(idx, 0, 1, m), np.arange(min(4, m + 1)))


def test_block_sparse_128k_config():
    """S = 131072, 32 query / 8 KV heads, k_b = 100 (the pages' setting): sampled rows of
    three heads checked like the small cases, attention on sampled query blocks."""
    c = prefill_case("prefill_bs_S131072", S=131072, H_q=32, H_kv=8, D=128, seed=4)
    q, k, v = _dev(c)
    idx = dsa.block_sparse_index_build(q, k, k_b=100, debug=True)
    out, lse = dsa.sparse_attn_prefill(q, k, v, idx["blk_cnt"], idx["blk_idx"], idx["col_cnt"], None)
    torch.cuda.synchronize()
    nq = 2048
    # 64 rows spread over the sequence (the first and last among them) for three heads
    heads = (0, 13, 31)
    rows = sorted(set([0, 1, 99, 100] + np.linspace(0, nq - 1, 64).astype(int).tolist()))
    qp = idx["q_pool"].cpu().numpy()
    sc = idx["scores"].cpu().numpy()
    for h in heads:
        g = h // c.G
        k64 = patterns.mean_pool(to_f64(c.k[0, :, g], "bf16"))
        q64 = patterns.mean_pool(to_f64(c.q[0, :, h], "bf16"))
        np.testing.assert_allclose(qp[0, h], q64, rtol=1e-5, atol=1e-6)
        z64 = c.scale * (q64 @ k64.T)
        for m in rows:
            z = z64[m, :m + 1]
            A = np.exp(z - z.max())
            A /= A.sum()
            s32 = sc[0, h, m, :m + 1]
            assert np.all(np.abs(s32 - z) <= 1e-5 * np.abs(z).max() + 1e-6)
            check_topk_list(s32, A, min(100, m + 1), _lists(idx, 0, h, m), floor=1e-9)
    # attention: the same rows for the three heads, the first and last block of every head
    pairs = [(0, h, m) for h in heads for m in rows]
    pairs += [(0, h, m) for h in range(c.H_q) if h not in heads for m in (0, nq - 1)]
    _check_attention(c, idx, out, lse, pairs)


def test_ashape_128k_config():
    """S = 131072 with the pages' 1024 initial + 4096 local tokens: lists exact on
    sampled rows, attention on sampled query blocks."""
    c = prefill_case("prefill_ashape_S131072", S=131072, H_q=32, H_kv=8, D=128, seed=4)
    q, k, v = _dev(c)
    idx = dsa.ashape_index_build(q, k, n_global=1024, n_local=4096)
    out, lse = dsa.sparse_attn_prefill(q, k, v, idx["blk_cnt"], idx["blk_idx"], idx["col_cnt"], None)
    torch.cuda.synchronize()
    for m in (0, 15, 16, 79, 80, 1000, 2047):
        for h in (0, 31):
            assert np.array_equal(_lists(idx, 0, h, m), patterns.ashape_blocks(m, 1024, 4096))
    _check_attention(c, idx, out, lse, [(0, h, m) for h in (0, 17) for m in (0, 80, 2047)])


def test_block_sparse_crowded_boundary_bucket():
    """One key block far above the rest (every query all ones, block 50's keys all 8):
    in rows m >= 50 the other scores crowd into the lowest value buckets, so the
    boundary bucket holds more than 32 blocks and the radix select decides."""
    c = prefill_case("bs_crowd", S=64 * 120, H_q=2, H_kv=1, D=64, seed=74)
    one = np.uint16(0x3F80)     # 1.0 in bf16
    eight = np.uint16(0x4100)   # 8.0
    c.q[:] = one
    c.k[0, 64 * 50:64 * 51] = eight
    q, k, v = _dev(c)
    idx = dsa.block_sparse_index_build(q, k, k_b=10, debug=True)
    torch.cuda.synchronize()
    _check_block_sparse(c, idx, 10, range(c.H_q), rows=[0, 9, 10, 49, 50, 51, 80, 119])
    for m in (50, 80, 119):
        assert 50 in _lists(idx, 0, 0, m)


# ------------------------------------------------------------ mixed per-head patterns

@pytest.mark.parametrize("S,D,G", [(1000, 128, 4), (700, 64, 1)])
def test_mixed_heads_equal_their_single_pattern_builders(S, D, G):
    H_kv = 2
    H_q = H_kv * G
    c = prefill_case("mixed", B=2, S=S, H_q=H_q, H_kv=H_kv, D=D, seed=75 + S,
                     n_vertical=40, n_slash=150)
    q, k, v = _dev(c)
    pats = [("vertical_slash", "a_shape", "block_sparse")[h % 3] for h in range(H_q)]
    mix = dsa.mixed_index_build(q, k, head_pattern=pats, n_vertical=40, n_slash=150,
                                n_global=128, n_local=256, k_b=5)
    vs_idx = dsa.vs_index_build(q, k, n_vertical=40, n_slash=150)
    ash = dsa.ashape_index_build(q, k, n_global=128, n_local=256)
    bsp = dsa.block_sparse_index_build(q, k, k_b=5)
    out, lse = dsa.sparse_attn_prefill(q, k, v, mix["blk_cnt"], mix["blk_idx"], mix["col_cnt"],
                                       mix["col_idx"])
    torch.cuda.synchronize()
    nq = (S + 63) // 64
    for b in range(2):
        for h in range(H_q):
            ref = {"vertical_slash": vs_idx, "a_shape": ash, "block_sparse": bsp}[pats[h]]
            for m in range(nq):
                nb_, nc = int(mix["blk_cnt"][b, h, m]), int(mix["col_cnt"][b, h, m])
                assert nb_ == int(ref["blk_cnt"][b, h, m])
                assert torch.equal(mix["blk_idx"][b, h, m, :nb_], ref["blk_idx"][b, h, m, :nb_])
                if pats[h] == "vertical_slash":
                    assert nc == int(ref["col_cnt"][b, h, m])
                    assert torch.equal(mix["col_idx"][b, h, m, :nc], ref["col_idx"][b, h, m, :nc])
                else:
                    assert nc == 0
    o = out.float().cpu().numpy()
    for (b, h, m) in [(0, h, m) for h in range(H_q) for m in (0, nq // 2, nq - 1)]:
        nb_, nc = int(mix["blk_cnt"][b, h, m]), int(mix["col_cnt"][b, h, m])
        O64, _ = vs.prefill_block_attention(c.q[b], c.k[b], c.v[b], h, c.G, m,
                                            mix["blk_idx"][b, h, m, :nb_].cpu().numpy(),
                                            mix["col_idx"][b, h, m, :nc].cpu().numpy(), c.S, c.scale)
        mx, mn = attention_errors(o[b, 64 * m:64 * m + len(O64), h], O64)
        assert mx <= MAX_ABS and mn <= MEAN_ABS
