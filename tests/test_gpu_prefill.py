"""GPU parity of the prefill half (vs_index_build + sparse_attn_prefill) against the fp64 oracle."""
import math

import numpy as np
import pytest
import torch

import dynamic_sparse_attention_gb300 as dsa
from dynamic_sparse_attention_gb300 import _build
from oracle import vs
from oracle.numerics import to_f64
from parity import attention_errors, check_topk_list, to_dev
from synth import prefill_128k, prefill_case

pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS = 1e-2, 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    _build.build()
    dsa.load()


def _dev(c):
    return to_dev(c.q, "bf16"), to_dev(c.k, "bf16"), to_dev(c.v, "bf16")


@pytest.fixture(autouse=True)
def _no_device_errors():
    yield
    torch.cuda.synchronize()
    assert dsa.device_error() == 0, "a prefill CTA gave up a bounded wait"


def _check_index(c, idx, heads=None, blocks=None):
    """Sums against fp64, top-k by the band rule, conversion exactly."""
    rows = vs.estimate_rows(c.S, c.last_q)
    vsum = idx["vsum"].cpu().numpy()
    ssum = idx["ssum"].cpu().numpy()
    vert = idx["vertical"].cpu().numpy()
    sl = idx["slash"].cpu().numpy()
    blk_cnt = idx["blk_cnt"].cpu().numpy()
    col_cnt = idx["col_cnt"].cpu().numpy()
    heads = range(c.H_q) if heads is None else heads
    for b in range(c.B):
        for h in heads:
            g = h // c.G
            A = vs.approx_attention(to_f64(c.q[b, rows, h], "bf16"), rows,
                                    to_f64(c.k[b, :, g], "bf16"), c.scale)
            v64, s64 = vs.vertical_sums(A), vs.slash_sums(A, rows)
            np.testing.assert_allclose(vsum[b, h], v64, rtol=2e-4, atol=1e-6)
            np.testing.assert_allclose(ssum[b, h], s64, rtol=2e-4, atol=1e-6)
            check_topk_list(vsum[b, h], v64, c.n_vertical, vert[b, h])
            check_topk_list(ssum[b, h], s64, c.n_slash, sl[b, h])
            blk, col = vs.vs_convert(vert[b, h], sl[b, h], c.S)
            ms = range(len(blk)) if blocks is None else blocks
            for m in ms:
                nb, nc = int(blk_cnt[b, h, m]), int(col_cnt[b, h, m])
                assert np.array_equal(idx["blk_idx"][b, h, m, :nb].cpu().numpy(), blk[m])
                assert np.array_equal(idx["col_idx"][b, h, m, :nc].cpu().numpy(), col[m])


def _check_attention(c, idx, out, lse, pairs):
    o = out.float().cpu().numpy()
    lse_g = lse.cpu().numpy()
    errs = []
    for (b, h, m) in pairs:
        nb = int(idx["blk_cnt"][b, h, m])
        nc = int(idx["col_cnt"][b, h, m])
        blk = idx["blk_idx"][b, h, m, :nb].cpu().numpy()
        col = idx["col_idx"][b, h, m, :nc].cpu().numpy()
        O64, l64 = vs.prefill_block_attention(c.q[b], c.k[b], c.v[b], h, c.G, m, blk, col, c.S,
                                              c.scale)
        r0 = 64 * m
        mx, mn = attention_errors(o[b, r0:r0 + len(O64), h], O64)
        assert mx <= MAX_ABS and mn <= MEAN_ABS, f"(b={b}, h={h}, m={m}): max {mx:.3e} mean {mn:.3e}"
        lg = lse_g[b, h, r0:r0 + len(O64)]
        fin = np.isfinite(l64)
        assert np.array_equal(fin, np.isfinite(lg))
        assert np.abs(lg[fin] - l64[fin]).max(initial=0) <= 1e-3
        errs.append(mx)
    return max(errs) if errs else 0.0


@pytest.mark.parametrize("S,D,G", [(700, 128, 2), (1000, 64, 4), (64, 128, 1), (130, 128, 8), (300, 64, 6)])
def test_vs_small_full_parity(S, D, G):
    H_kv = 2
    c = prefill_case("small", S=S, H_q=H_kv * G, H_kv=H_kv, D=D, seed=40 + S,
                     n_vertical=min(40, S), n_slash=min(150, S))
    q, k, v = _dev(c)
    idx = dsa.vs_index_build(q, k, last_q=c.last_q, n_vertical=c.n_vertical, n_slash=c.n_slash,
                             debug=True)
    out, lse = dsa.sparse_attn_prefill(q, k, v, idx["blk_cnt"], idx["blk_idx"], idx["col_cnt"],
                                       idx["col_idx"])
    torch.cuda.synchronize()
    _check_index(c, idx)
    nq = math.ceil(S / 64)
    _check_attention(c, idx, out, lse, [(0, h, m) for h in range(c.H_q) for m in range(nq)])


def test_short_estimate_window():
    """last_q < 64 and S < last_q: fewer estimate rows."""
    c = prefill_case("short", S=40, H_q=2, H_kv=1, D=64, seed=44, last_q=64, n_vertical=5,
                     n_slash=7)
    q, k, v = _dev(c)
    idx = dsa.vs_index_build(q, k, last_q=64, n_vertical=5, n_slash=7, debug=True)
    torch.cuda.synchronize()
    _check_index(c, idx)
    c2 = prefill_case("lq", S=500, H_q=2, H_kv=1, D=128, seed=45, last_q=17, n_vertical=20,
                      n_slash=30)
    q, k, v = _dev(c2)
    idx = dsa.vs_index_build(q, k, last_q=17, n_vertical=20, n_slash=30, debug=True)
    torch.cuda.synchronize()
    _check_index(c2, idx)


def _random_lists(rng, S, H_q, max_blk, max_col, dense=False):
    nq = math.ceil(S / 64)
    blk_cnt = np.zeros((1, H_q, nq), np.int32)
    col_cnt = np.zeros((1, H_q, nq), np.int32)
    blk_idx = np.full((1, H_q, nq, max_blk), -1, np.int32)
    col_idx = np.full((1, H_q, nq, max_col), -1, np.int32)
    for h in range(H_q):
        for m in range(nq):
            if dense:
                bl = np.arange(m + 1)
            else:
                nb = int(rng.integers(0, min(m + 1, max_blk) + 1))
                bl = np.sort(rng.choice(m + 1, size=nb, replace=False))
            blk_cnt[0, h, m] = len(bl)
            blk_idx[0, h, m, :len(bl)] = bl
            if not dense:
                free = np.setdiff1d(np.arange(min(S, 64 * m + 64)),
                                    np.concatenate([np.arange(64 * n, 64 * n + 64) for n in bl] or [[]]))
                ncol = int(rng.integers(0, min(len(free), max_col) + 1))
                cl = np.sort(rng.choice(free, size=ncol, replace=False)) if ncol else []
                col_cnt[0, h, m] = ncol
                col_idx[0, h, m, :ncol] = cl
    t = lambda a: torch.from_numpy(a).cuda()
    return t(blk_cnt), t(blk_idx), t(col_cnt), t(col_idx)


@pytest.mark.parametrize("D", [64, 128])
def test_generic_lists(D):
    """Arbitrary block lists and gathered columns (several column tiles, ragged tail, empty rows)."""
    rng = np.random.default_rng(50 + D)
    c = prefill_case("lists", S=777, H_q=4, H_kv=2, D=D, seed=51)
    q, k, v = _dev(c)
    lists = _random_lists(rng, c.S, c.H_q, max_blk=13, max_col=150)
    out, lse = dsa.sparse_attn_prefill(q, k, v, *lists)
    torch.cuda.synchronize()
    idx = dict(zip(["blk_cnt", "blk_idx", "col_cnt", "col_idx"], lists))
    _check_attention(c, idx, out, lse, [(0, h, m) for h in range(4) for m in range(13)])


def test_dense_lists_match_sdpa():
    c = prefill_case("dense", S=1000, H_q=4, H_kv=2, D=128, seed=52)
    q, k, v = _dev(c)
    lists = _random_lists(np.random.default_rng(0), c.S, c.H_q, 16, 1, dense=True)
    out, lse = dsa.sparse_attn_prefill(q, k, v, *lists)
    qt = q.float().permute(0, 2, 1, 3)
    kt = k.float().permute(0, 2, 1, 3).repeat_interleave(2, 1)
    vt = v.float().permute(0, 2, 1, 3).repeat_interleave(2, 1)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=True)
    err = (out.float().permute(0, 2, 1, 3) - ref).abs()
    assert err.max().item() <= MAX_ABS and err.mean().item() <= MEAN_ABS


def test_prefill_128k_config():
    """S=131072, 32q/8kv, d=128: full-size index build and attention, checked on samples."""
    c = prefill_128k()
    q, k, v = _dev(c)
    idx = dsa.vs_index_build(q, k, last_q=c.last_q, n_vertical=c.n_vertical, n_slash=c.n_slash,
                             debug=True)
    out, lse = dsa.sparse_attn_prefill(q, k, v, idx["blk_cnt"], idx["blk_idx"], idx["col_cnt"],
                                       idx["col_idx"])
    torch.cuda.synchronize()
    nq = c.S // 64
    # 64 query blocks spread over the sequence (the first and last among them) for three
    # heads, and the first and last blocks of every head
    blocks = sorted(set(np.linspace(0, nq - 1, 64).astype(int).tolist()))
    _check_index(c, idx, heads=[0, 13, 31], blocks=blocks)
    _check_index(c, idx, heads=[h for h in range(c.H_q) if h not in (0, 13, 31)], blocks=[0, nq - 1])
    pairs = [(0, h, m) for h in (0, 13, 31) for m in blocks]
    pairs += [(0, h, m) for h in range(c.H_q) if h not in (0, 13, 31) for m in (0, nq - 1)]
    _check_attention(c, idx, out, lse, pairs)
    # planted structure shows up in the estimate (generator self-check, not parity)
    vert = idx["vertical"].cpu().numpy()[0]
    sl = idx["slash"].cpu().numpy()[0]
    for h in (0, 13, 31):
        assert np.isin(c.planted_columns, vert[h]).mean() >= 0.9
        assert np.isin(c.planted_offsets, sl[h]).mean() >= 0.85


@pytest.mark.parametrize("D", [64, 128])
def test_vs_and_random_lists_every_block(D):
    """Every (head, query block) of an S = 1500 prefill against the fp64 oracle, once over
    the vertical-slash lists and once over arbitrary lists (several column tiles each)."""
    c = prefill_case("agree", S=1500, H_q=4, H_kv=2, D=D, seed=70 + D, n_vertical=50,
                     n_slash=300)
    q, k, v = _dev(c)
    idx = dsa.vs_index_build(q, k, last_q=c.last_q, n_vertical=c.n_vertical, n_slash=c.n_slash)
    rand = _random_lists(np.random.default_rng(D), c.S, c.H_q, max_blk=24, max_col=130)
    nq = math.ceil(c.S / 64)
    for lists in ((idx["blk_cnt"], idx["blk_idx"], idx["col_cnt"], idx["col_idx"]), rand):
        out, lse = dsa.sparse_attn_prefill(q, k, v, *lists)
        torch.cuda.synchronize()
        li = dict(zip(["blk_cnt", "blk_idx", "col_cnt", "col_idx"], lists))
        _check_attention(c, li, out, lse, [(0, h, m) for h in range(c.H_q) for m in range(nq)])


def _pair_lists(rng, S, H_q, max_col):
    """Column lists that the two query blocks of a CTA (2p, 2p + 1) share in every way:
    identical lists, one list inside the other, partial overlap, disjoint lists, one empty
    list; each block also lists its own diagonal block and one earlier block (columns
    avoid both blocks' listed blocks)."""
    nq = math.ceil(S / 64)
    blk_cnt = np.zeros((1, H_q, nq), np.int32)
    col_cnt = np.zeros((1, H_q, nq), np.int32)
    blk_idx = np.full((1, H_q, nq, 2), -1, np.int32)
    col_idx = np.full((1, H_q, nq, max_col), -1, np.int32)
    for h in range(H_q):
        for p in range((nq + 1) // 2):
            ms = [m for m in (2 * p, 2 * p + 1) if m < nq]
            bls = {}
            for m in ms:
                bl = sorted({m, int(rng.integers(0, m + 1))})
                bls[m] = bl
                blk_cnt[0, h, m] = len(bl)
                blk_idx[0, h, m, :len(bl)] = bl
            hi = min(S, 64 * ms[-1] + 64)
            taken = set()
            for m in ms:
                taken |= set(range(64 * bls[m][0], 64 * bls[m][0] + 64)) | set(range(64 * m, 64 * m + 64))
            pool = np.array(sorted(set(range(hi)) - taken), np.int64)
            kind = int(rng.integers(0, 5))
            n = min(len(pool), max_col)
            a = rng.choice(pool, size=int(rng.integers(0, n + 1)), replace=False) if n else pool[:0]
            if kind == 0:
                b = a
            elif kind == 1:
                b = a[:len(a) // 2]
            elif kind == 2:
                rest = np.setdiff1d(pool, a)
                extra = rng.choice(rest, size=min(len(rest), int(rng.integers(0, max_col - len(a) // 2 + 1))),
                                   replace=False) if len(rest) else rest
                b = np.concatenate([a[: len(a) // 2], extra])[:max_col]
            elif kind == 3:
                rest = np.setdiff1d(pool, a)
                b = rng.choice(rest, size=min(len(rest), max_col), replace=False) if len(rest) else rest
            else:
                b = pool[:0]
            for m, lst in zip(ms, (a, b)):
                lst = np.sort(np.asarray(lst, np.int64))
                col_cnt[0, h, m] = len(lst)
                col_idx[0, h, m, :len(lst)] = lst
    return blk_cnt, blk_idx, col_cnt, col_idx


@pytest.mark.parametrize("D", [64, 128])
def test_column_lists_shared_by_block_pairs(D):
    """Every (head, query block) against the fp64 oracle over column lists that the two
    query blocks of a CTA share in part, in full or not at all, and over the same lists
    in shuffled order (the kernel needs no order within a list)."""
    rng = np.random.default_rng(90 + D)
    c = prefill_case("pairs", S=1700, H_q=4, H_kv=2, D=D, seed=91 + D)
    q, k, v = _dev(c)
    blk_cnt, blk_idx, col_cnt, col_idx = _pair_lists(rng, c.S, c.H_q, max_col=420)
    shuffled = col_idx.copy()
    for h in range(c.H_q):
        for m in range(shuffled.shape[2]):
            n = int(col_cnt[0, h, m])
            shuffled[0, h, m, :n] = rng.permutation(shuffled[0, h, m, :n])
    t = lambda a: torch.from_numpy(a).cuda()
    nq = math.ceil(c.S / 64)
    for cols in (col_idx, shuffled):
        lists = (t(blk_cnt), t(blk_idx), t(col_cnt), t(cols))
        out, lse = dsa.sparse_attn_prefill(q, k, v, *lists)
        torch.cuda.synchronize()
        li = dict(zip(["blk_cnt", "blk_idx", "col_cnt", "col_idx"], lists))
        _check_attention(c, li, out, lse, [(0, h, m) for h in range(c.H_q) for m in range(nq)])


@pytest.mark.parametrize("D", [64, 128])
def test_lists_shared_by_head_pairs(D):
    """Every (head, query block) against the fp64 oracle when the two query heads of a
    head pair list the same blocks and columns for some query-block pairs (both blocks),
    for one block of a pair only, or not at all: the kernel takes the head-pair row
    groups exactly where both blocks' lists agree; G = 4, an odd query-block count."""
    rng = np.random.default_rng(110 + D)
    c = prefill_case("heads", S=1600, H_q=8, H_kv=2, D=D, seed=111 + D)
    q, k, v = _dev(c)
    lists = [x.cpu().numpy() for x in _random_lists(rng, c.S, c.H_q, max_blk=20, max_col=300)]
    blk_cnt, blk_idx, col_cnt, col_idx = lists
    nq = math.ceil(c.S / 64)
    for h0 in range(0, c.H_q, 2):
        for p in range((nq + 1) // 2):
            kind = (h0 // 2 + p) % 3   # 0: both blocks shared, 1: block 2p only, 2: none
            ms = [2 * p, 2 * p + 1] if kind == 0 else ([2 * p] if kind == 1 else [])
            for m in ms:
                if m < nq:
                    for a in lists:
                        a[0, h0 + 1, m] = a[0, h0, m]
    t = lambda a: torch.from_numpy(a).cuda()
    tl = tuple(t(a) for a in lists)
    out, lse = dsa.sparse_attn_prefill(q, k, v, *tl)
    torch.cuda.synchronize()
    li = dict(zip(["blk_cnt", "blk_idx", "col_cnt", "col_idx"], tl))
    _check_attention(c, li, out, lse, [(0, h, m) for h in range(c.H_q) for m in range(nq)])


def _run_lists(rng, S, H_q, max_col):
    """Column lists made of runs of consecutive keys (lengths 8, 5, 16, 1 in a random
    mix), ascending, outside the block's two listed blocks."""
    nq = math.ceil(S / 64)
    blk_cnt = np.zeros((1, H_q, nq), np.int32)
    col_cnt = np.zeros((1, H_q, nq), np.int32)
    blk_idx = np.full((1, H_q, nq, 2), -1, np.int32)
    col_idx = np.full((1, H_q, nq, max_col), -1, np.int32)
    for h in range(H_q):
        for m in range(nq):
            bl = sorted({m, int(rng.integers(0, m + 1))})
            blk_cnt[0, h, m] = len(bl)
            blk_idx[0, h, m, :len(bl)] = bl
            free = np.ones(min(S, 64 * m + 64), bool)
            for n in bl:
                free[64 * n:64 * n + 64] = False
            keys = []
            x = int(rng.integers(0, 20))
            while x < len(free) and len(keys) < max_col:
                run = int(rng.choice([8, 8, 8, 5, 16, 1]))
                seg = [y for y in range(x, min(x + run, len(free))) if free[y]]
                keys += seg[:max_col - len(keys)]
                x += run + int(rng.integers(0, 40))
            col_cnt[0, h, m] = len(keys)
            col_idx[0, h, m, :len(keys)] = keys
    return blk_cnt, blk_idx, col_cnt, col_idx


@pytest.mark.parametrize("D", [64, 128])
def test_column_runs(D):
    """Every (head, query block) against the fp64 oracle over column lists made of runs
    of consecutive keys, as the InfiniteHiP selection of consecutive-token chunks makes
    them, the same lists for the two heads of one head pair (head-pair row groups) and
    different ones for the other pair."""
    rng = np.random.default_rng(130 + D)
    c = prefill_case("runs", S=2100, H_q=4, H_kv=2, D=D, seed=131 + D)
    q, k, v = _dev(c)
    lists = _run_lists(rng, c.S, c.H_q, max_col=500)
    for a in lists:
        a[0, 1] = a[0, 0]   # heads 0 and 1 (one head pair of KV head 0) share their lists
    t = lambda a: torch.from_numpy(a).cuda()
    tl = tuple(t(a) for a in lists)
    out, lse = dsa.sparse_attn_prefill(q, k, v, *tl)
    torch.cuda.synchronize()
    li = dict(zip(["blk_cnt", "blk_idx", "col_cnt", "col_idx"], tl))
    nq = math.ceil(c.S / 64)
    _check_attention(c, li, out, lse, [(0, h, m) for h in range(c.H_q) for m in range(nq)])


def test_non_positive_scale_is_rejected():
    """The kernel orders scores by their raw value; a scale <= 0 is an argument error."""
    c = prefill_case("scale", S=128, H_q=2, H_kv=1, D=64, seed=9)
    q, k, v = _dev(c)
    lists = _random_lists(np.random.default_rng(1), c.S, c.H_q, 2, 4)
    for bad in (0.0, -0.125):
        with pytest.raises(dsa.DsaError) as ei:
            dsa.sparse_attn_prefill(q, k, v, *lists, scale=bad)
        assert ei.value.status == -1
