"""Pins for the fp64 selection/decode oracle (CPU only).

Each test ties the oracle to something other than itself: numbers the
InfiniteHiP summary prints, a library routine (torch SDPA in float64), a
brute-force characterisation on tiny inputs, or an invariant the pages state.
"""
import itertools
import math

import numpy as np
import pytest
import torch

from oracle import hip
from oracle.numerics import to_f64
from synth import decode_case, decode_tiny


def _f64_keys(rng, T, H_kv, D):
    return rng.standard_normal((T, H_kv, D)).astype(np.float32)


# ------------------------------------------------------------ page counts

def test_candidate_range_page_counts(golden):
    g = golden["sink_stream_1m"]
    I = hip.candidate_range(g["T"], g["n_sink"], g["n_stream"])
    assert len(I) == g["pruned_tokens"]
    A = hip.attended_set(g["T"], g["n_sink"], g["n_stream"], np.zeros(0, np.int64))
    assert len(A) == g["always_kept_tokens"]
    assert I[0] == g["n_sink"] and I[-1] == g["T"] - g["n_stream"] - 1


def test_stage_chunk_counts_at_1m(golden):
    g = golden["stage_chunk_counts_1m"]
    I = hip.candidate_range(g["T"], g["n_sink"], g["n_stream"])
    n_chunks = []
    for L, k in zip(g["chunk"], g["keep"]):
        chunks = hip.chunk_partition(I, L)
        n_chunks.append(len(chunks))
        Kc = k // L
        # keep the first K chunks: the count of surviving tokens is what matters here
        I = hip.assemble(chunks, np.arange(min(Kc, len(chunks))))
        assert len(I) <= k
    for got, want in zip(n_chunks, g["approx_chunks_per_stage"]):
        assert abs(got - want) <= g["rel_tol"] * want
    assert abs(sum(n_chunks) - g["approx_total"]) <= g["rel_tol"] * g["approx_total"]


def test_window_sizes(golden):
    g = golden["window_size_3k_5k"]
    for keep, total in zip(g["final_keep"], g["total_window"]):
        T = 1 << 20
        I = np.arange(g["n_sink"], g["n_sink"] + keep)
        assert len(hip.attended_set(T, g["n_sink"], g["n_stream"], I)) == total


@pytest.mark.parametrize("case", [0, 1])
def test_selectrep_evaluation_count(golden, case):
    c = golden["selectrep_evaluations"]["cases"][case]
    L = c["l_c"]
    rng = np.random.default_rng(10 + case)
    K = _f64_keys(rng, L, 1, 16)
    q = rng.standard_normal((3, 16))
    r, rho, evals = hip.select_rep(q, K[:, 0, :], "f32", np.arange(L))
    assert evals == c["evaluations"] == 2 * math.ceil(math.log2(L))


# ------------------------------------------------------------ tournament characterisation

def _leaf_path_ok(scores, r):
    """Independent characterisation of the tournament winner by enumeration.

    For leaf r, walk the halving tree: at every split of the range holding r,
    r's half must win (right half wins only on a strictly larger first score).
    """
    a, b = 0, len(scores) - 1
    while a < b:
        mid = (a + b + 1) // 2
        right_wins = scores[mid] > scores[a]
        if r >= mid and not right_wins:
            return False
        if r < mid and right_wins:
            return False
        a, b = (mid, b) if r >= mid else (a, mid - 1)
    return True


@pytest.mark.parametrize("L", [1, 2, 3, 4, 5, 7, 8, 11, 16])
def test_selectrep_matches_enumeration(L):
    rng = np.random.default_rng(L)
    D = 8
    for trial in range(40):
        # integer-valued keys so that ties really occur
        K = rng.integers(-2, 3, size=(L, D)).astype(np.float32)
        q = rng.integers(-2, 3, size=(2, D)).astype(np.float64)
        scores = np.max(q @ K.astype(np.float64).T, axis=0)
        winners = [r for r in range(L) if _leaf_path_ok(scores, r)]
        assert len(winners) == 1
        pos = np.arange(100, 100 + L)
        r, rho, _ = hip.select_rep(q, np.concatenate([np.zeros((100, D), np.float32), K]),
                                   "f32", pos)
        assert r == 100 + winners[0]
        assert rho == scores[winners[0]]


def test_selectrep_special_orders():
    D, L = 4, 16
    q = np.ones((1, D))
    inc = np.repeat(np.arange(L, dtype=np.float32)[:, None], D, axis=1)
    assert hip.select_rep(q, inc, "f32", np.arange(L))[0] == L - 1   # increasing -> last
    assert hip.select_rep(q, inc[::-1].copy(), "f32", np.arange(L))[0] == 0  # decreasing -> first
    flat = np.ones((L, D), np.float32)
    assert hip.select_rep(q, flat, "f32", np.arange(L))[0] == 0     # all tied -> left wins


@pytest.mark.parametrize("L", [1, 2])
def test_selectrep_exact_for_tiny_chunks(L):
    rng = np.random.default_rng(5)
    for _ in range(50):
        K = rng.standard_normal((L, 6)).astype(np.float32)
        q = rng.standard_normal((4, 6))
        s = np.max(q @ K.astype(np.float64).T, axis=0)
        assert hip.select_rep(q, K, "f32", np.arange(L))[0] == int(np.argmax(s))


def test_vectorised_tournament_equals_scalar():
    c = decode_case("t", B=1, T=700, T_q=2, H_q=4, H_kv=2, D=16, dtype="bf16",
                    chunk=(16,), keep=(64,), n_sink=4, n_stream=8, seed=7, plant="none")
    q = to_f64(c.q[0], "bf16")
    I = hip.candidate_range(700, 4, 8)
    for L in (1, 3, 16, 37):
        chunks = hip.chunk_partition(I, L)
        reps, rho = hip.select_rep_all(q, c.k[0], "bf16", chunks, c.G)
        for h in range(4):
            for j in range(0, len(chunks), 5):
                r, s, _ = hip.select_rep(q[:, h, :], c.k[0][:, h // c.G, :], "bf16", chunks[j])
                assert reps[h, j] == r and rho[h, j] == s


# ------------------------------------------------------------ top-K characterisation

def test_topk_pairwise_characterisation():
    rng = np.random.default_rng(3)
    for n in range(1, 9):
        for K in range(1, n + 2):
            for _ in range(10):
                s = rng.integers(0, 4, size=n).astype(np.float64)
                kept = hip.topk_chunks(s, K)
                assert list(kept) == sorted(kept)
                assert len(kept) == min(n, K)
                ks = set(kept.tolist())
                for i in ks:
                    for j in set(range(n)) - ks:
                        assert s[i] > s[j] or (s[i] == s[j] and i < j)


def test_topk_matches_exhaustive_subsets():
    rng = np.random.default_rng(4)
    n, K = 7, 3
    for _ in range(30):
        s = rng.integers(0, 3, size=n).astype(np.float64)
        # best subset: largest sum of scores, then lexicographically smallest indices
        best = min(itertools.combinations(range(n), K),
                   key=lambda c: (-sum(s[list(c)]), sorted(c)))
        assert list(hip.topk_chunks(s, K)) == sorted(best)


# ------------------------------------------------------------ invariants + dense case

def _run(c, b=0):
    q = to_f64(c.q[b], c.dtype)
    stages, I = hip.hip_select(q, c.k[b], c.dtype, int(c.kv_len[b]), c.chunk, c.keep,
                               c.n_sink, c.n_stream, c.G)
    return q, stages, I


def test_stage_invariants_tiny_config():
    c = decode_tiny()
    q, stages, I = _run(c)
    prev = hip.candidate_range(2048, c.n_sink, c.n_stream)
    for st, k in zip(stages, c.keep):
        assert len(st.I_out) <= k
        assert np.all(np.diff(st.I_out) > 0)
        assert np.all(np.isin(st.I_out, prev))
        prev = st.I_out
    A = hip.attended_set(2048, c.n_sink, c.n_stream, I)
    assert len(A) == 16 + 128 + 64
    assert np.all(np.isin(np.arange(16), A)) and np.all(np.isin(np.arange(2048 - 64, 2048), A))


def test_dense_special_case_matches_sdpa():
    """keep >= all chunks at every stage -> attention over every key == dense SDPA."""
    c = decode_case("dense", B=1, T=300, T_q=3, H_q=4, H_kv=2, D=32, dtype="bf16",
                    chunk=(16, 4), keep=(4096, 4096), n_sink=5, n_stream=7, seed=11,
                    plant="none")
    q, stages, I = _run(c)
    assert np.array_equal(I, hip.candidate_range(300, 5, 7))
    A = hip.attended_set(300, 5, 7, I)
    assert np.array_equal(A, np.arange(300))
    O, lse = hip.decode_attention(q, c.k[0], c.v[0], "bf16", A, c.scale, c.G)
    Qt = torch.from_numpy(q).permute(1, 0, 2)                       # [H, T_q, D]
    Kt = torch.from_numpy(to_f64(c.k[0], "bf16")).permute(1, 0, 2)  # [H_kv, T, D]
    Vt = torch.from_numpy(to_f64(c.v[0], "bf16")).permute(1, 0, 2)
    Kt = Kt.repeat_interleave(c.G, 0)
    Vt = Vt.repeat_interleave(c.G, 0)
    ref = torch.nn.functional.scaled_dot_product_attention(Qt, Kt, Vt)
    np.testing.assert_allclose(O, ref.permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)
    ref_lse = torch.logsumexp(c.scale * Qt @ Kt.transpose(1, 2), dim=-1)
    np.testing.assert_allclose(lse, ref_lse.T.numpy(), rtol=0, atol=1e-12)


def test_exact_exclusion_matches_eq1_constant():
    """Exact exclusion == softmax(QK^T/sqrt(d) - c(1-M)) with c = 1e5 (MInference Eq. 1)."""
    rng = np.random.default_rng(12)
    T, D = 200, 32
    K = rng.standard_normal((T, 1, D)).astype(np.float32)
    V = rng.standard_normal((T, 1, D)).astype(np.float32)
    q = rng.standard_normal((2, 1, D))
    A = np.sort(rng.choice(T, 40, replace=False))
    O, _ = hip.decode_attention(q, K, V, "f32", A, 1 / np.sqrt(D), 1)
    M = np.zeros(T)
    M[A] = 1
    z = torch.from_numpy(q[:, 0] @ K[:, 0].astype(np.float64).T / np.sqrt(D) - 1e5 * (1 - M))
    ref = torch.softmax(z, -1).numpy() @ V[:, 0].astype(np.float64)
    np.testing.assert_allclose(O[:, 0], ref, rtol=0, atol=1e-12)


def test_metamorphic_scale_and_shift():
    c = decode_case("meta", B=1, T=900, T_q=1, H_q=4, H_kv=1, D=32, dtype="f32",
                    chunk=(32, 8), keep=(256, 64), n_sink=8, n_stream=16, seed=13)
    q, stages, I = _run(c)
    stages2, I2 = hip.hip_select(2.5 * q, c.k[0], "f32", 900, c.chunk, c.keep, 8, 16, c.G)
    assert np.array_equal(I, I2)
    for a, b in zip(stages, stages2):
        assert np.array_equal(a.reps, b.reps) and np.array_equal(a.kept, b.kept)
    A = hip.attended_set(900, 8, 16, I)
    O, _ = hip.decode_attention(q, c.k[0], c.v[0], "f32", A, c.scale, c.G)
    V2 = (c.v[0].astype(np.float64) + 0.75)
    O2, _ = hip.decode_attention(q, c.k[0], V2, "f64", A, c.scale, c.G)
    np.testing.assert_allclose(O2, O + 0.75, rtol=0, atol=1e-12)


def test_partial_chunk_and_short_context():
    # context shorter than sink + window: nothing to prune, everything attended once
    I = hip.candidate_range(50, 32, 64)
    assert len(I) == 0
    A = hip.attended_set(50, 32, 64, I)
    assert np.array_equal(A, np.arange(50))
    # ragged last chunk keeps its true length
    chunks = hip.chunk_partition(np.arange(10, 31), 8)
    assert [len(x) for x in chunks] == [8, 8, 5]


# ------------------------------------------------------------ mask caching (section 3.4)

def test_refresh_timeline_matches_figure7_description(golden):
    g = golden["mask_refresh_timeline"]
    for i, want in enumerate(g["refresh_steps"]):
        got = [c for c in range(g["steps"]) if hip.refresh_schedule(c, g["n_refresh"])[i]]
        assert got == want, f"stage {i + 1}"
    # every preset of the table nests: a refresh of stage i is also one of each later stage
    for r in g["presets"].values():
        for c in range(2 * r[0] + 1):
            m = hip.refresh_schedule(c, r)
            assert m == sorted(m), (r, c, m)


def _growing_steps(n_steps, T0, T_max, H_q=4, H_kv=2, D=32, seed=40):
    c = decode_case("cache", B=1, T=T_max, T_q=1, H_q=H_q, H_kv=H_kv, D=D, dtype="f32",
                    chunk=(32, 8, 2), keep=(256, 64, 16), n_sink=8, n_stream=16, seed=seed)
    rng = np.random.default_rng(seed + 1)
    qs = [rng.standard_normal((1, H_q, D)) for _ in range(n_steps)]
    return c, qs, [T0 + s for s in range(n_steps)]


def test_cached_with_every_stage_refreshed_is_the_full_pipeline():
    c, qs, Ts = _growing_steps(6, 900, 1000)
    cache = [None] * 3
    for q, T in zip(qs, Ts):
        ran, I = hip.hip_select_cached(q, c.k[0], "f32", T, c.chunk, c.keep, c.n_sink,
                                       c.n_stream, c.G, [True] * 3, cache)
        stages, I_full = hip.hip_select(q, c.k[0], "f32", T, c.chunk, c.keep, c.n_sink,
                                        c.n_stream, c.G)
        assert np.array_equal(I, I_full)
        for i, st in enumerate(stages):
            assert np.array_equal(cache[i], st.I_out)
            assert np.array_equal(ran[i].kept, st.kept)


def test_cached_no_refresh_keeps_every_list():
    c, qs, Ts = _growing_steps(2, 900, 1000)
    cache = [None] * 3
    hip.hip_select_cached(qs[0], c.k[0], "f32", Ts[0], c.chunk, c.keep, c.n_sink, c.n_stream,
                          c.G, [True] * 3, cache)
    before = [x.copy() for x in cache]
    ran, I = hip.hip_select_cached(qs[1], c.k[0], "f32", Ts[1], c.chunk, c.keep, c.n_sink,
                                   c.n_stream, c.G, [False] * 3, cache)
    assert ran == {} and all(np.array_equal(a, b) for a, b in zip(before, cache))
    assert I is cache[-1]


def test_refreshed_stage_reads_the_cached_previous_stage():
    """Three key groups, worked out by hand: with query e1 the first two stages keep the
    chunks of groups A (score 3) and B (score 2) and the last keeps A; a later query e2
    prefers C (score 3, outside the cached lists) over B (2) over A (0).  Refreshing
    only the last stage must give B: C would mean it restarted from the full range, A
    that it reused its own list or the old query."""
    T, D = 1024, 16
    K = np.zeros((T, 1, D), np.float32)
    K[:, 0, 2:] = 0.01 * np.random.default_rng(5).standard_normal((T, D - 2))
    A, B, C = np.arange(96, 104), np.arange(512, 520), np.arange(800, 808)
    K[A, 0, 0] = 3.0
    K[B, 0, 0] = 2.0
    K[B, 0, 1] = 2.0
    K[C, 0, 1] = 3.0
    e1 = np.zeros((1, 1, D))
    e1[0, 0, 0] = 1.0
    e2 = np.zeros((1, 1, D))
    e2[0, 0, 1] = 1.0
    chunk, keep = (32, 8, 2), (64, 16, 8)
    cache = [None] * 3
    _, I0 = hip.hip_select_cached(e1, K, "f32", T, chunk, keep, 0, 0, 1, [True] * 3, cache)
    assert np.array_equal(cache[1], np.concatenate([A, B]))
    assert np.array_equal(I0, A)
    _, I1 = hip.hip_select_cached(e2, K, "f32", T, chunk, keep, 0, 0, 1,
                                  [False, False, True], cache)
    assert np.array_equal(I1, B)
    # refreshing every stage with e2 instead reaches C
    _, I2 = hip.hip_select_cached(e2, K, "f32", T, chunk, keep, 0, 0, 1, [True] * 3, cache)
    assert np.array_equal(I2, C)


def test_stale_stage0_list_and_the_attended_set():
    """Stage 0 cached at T0 while the context grows to T: the selection stays inside the
    candidate range of T0, the attended set has no repeats, and the tokens that left the
    streaming window in between are not attended until stage 0 runs again."""
    c, qs, Ts = _growing_steps(9, 900, 1000)
    cache = [None] * 3
    n_refresh = (8, 4, 2)
    for step, (q, T) in enumerate(zip(qs, Ts)):
        ran, I = hip.hip_select_cached(q, c.k[0], "f32", T, c.chunk, c.keep, c.n_sink,
                                       c.n_stream, c.G, hip.refresh_schedule(step, n_refresh),
                                       cache)
        T0 = Ts[step - step % 8]
        assert np.all(np.isin(I, hip.candidate_range(T0, c.n_sink, c.n_stream)))
        A = hip.attended_set(T, c.n_sink, c.n_stream, I)
        assert len(np.unique(A)) == len(A) == c.n_sink + len(I) + c.n_stream
        left = np.arange(T0 - c.n_stream, T - c.n_stream)
        assert not np.isin(left, A).any()
        assert (0 in ran) == (step % 8 == 0)


# ------------------------------------------------------------ FP8 E4M3 keys and values

def test_e4m3_decoding_matches_torch_float8():
    """Every one of the 256 codes against torch's float8_e4m3fn view (NaN codes too)."""
    from oracle.numerics import e4m3_to_f64
    codes = np.arange(256, dtype=np.uint8)
    got = e4m3_to_f64(codes)
    want = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(got), np.isnan(want)) and np.isnan(got).sum() == 2
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])
    # the format's landmarks: largest finite 448, smallest subnormal 2^-9, smallest normal 2^-6
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9 and got[0x08] == 2.0 ** -6
    assert got[0xFE] == -448.0 and got[0x80] == 0.0


# ------------------------------------------------------------ sparse prefill (query blocks of 64)

def test_prefill_keep_all_is_dense_causal():
    """Budgets holding every chunk: each query block attends every key before its rows,
    so the prefill equals SDPA(is_causal)."""
    c = decode_case("pf", B=1, T=300, T_q=300, H_q=4, H_kv=2, D=16, dtype="bf16",
                    chunk=(16, 4), keep=(4096, 4096), n_sink=5, n_stream=7, seed=41, plant="none")
    q64 = to_f64(c.q[0], "bf16")                                   # [S, H_q, D]
    I = hip.hip_prefill_select(q64, c.k[0], "bf16", 300, c.chunk, c.keep, 5, 7, c.G)
    for m, Im in enumerate(I):
        T_m = hip.prefill_block_len(300, m)
        assert np.array_equal(Im, hip.candidate_range(T_m, 5, 7))
    res = hip.prefill_attention(q64, c.k[0], c.v[0], "bf16", 300, I, 5, 7, c.scale, c.G)
    Q = torch.from_numpy(q64).permute(1, 0, 2)
    K = torch.from_numpy(to_f64(c.k[0], "bf16")).permute(1, 0, 2).repeat_interleave(c.G, 0)
    V = torch.from_numpy(to_f64(c.v[0], "bf16")).permute(1, 0, 2).repeat_interleave(c.G, 0)
    ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V, is_causal=True).permute(1, 0, 2)
    for m, (O, _) in res.items():
        np.testing.assert_allclose(O, ref[64 * m:64 * m + len(O)].numpy(), rtol=0, atol=1e-12)


def test_prefill_block_selection_is_causal_and_keeps_sink_and_window():
    c = decode_case("pf2", B=1, T=700, T_q=700, H_q=2, H_kv=1, D=16, dtype="bf16",
                    chunk=(32, 8), keep=(128, 32), n_sink=8, n_stream=64, seed=42, plant="none")
    q64 = to_f64(c.q[0], "bf16")
    I = hip.hip_prefill_select(q64, c.k[0], "bf16", 700, c.chunk, c.keep, 8, 64, c.G)
    for m, Im in enumerate(I):
        T_m = hip.prefill_block_len(700, m)
        assert np.all(Im < max(8, T_m - 64)) and np.all(Im >= 8) and len(Im) <= 32
        A = hip.attended_set(T_m, 8, 64, Im)
        assert np.all(np.isin(np.arange(min(8, T_m)), A))
        assert np.all(np.isin(np.arange(max(8, T_m - 64), T_m), A))
    # a row attends nothing after itself: the first row of block 3 and its window
    res = hip.prefill_attention(q64, c.k[0], c.v[0], "bf16", 700, I, 8, 64, c.scale, c.G, blocks=[3])
    O, lse = res[3]
    assert np.isfinite(lse).all()


def test_prefill_finds_a_planted_key_per_block():
    """Keys 100..103 equal the mean query of block 9 (scaled up): block 9's selection
    keeps them (chunk 8, budget 4 of the candidate chunks)."""
    rng = np.random.default_rng(43)
    S, D = 64 * 12, 16
    q = rng.standard_normal((S, 1, D))
    K = (0.3 * rng.standard_normal((S, 1, D))).astype(np.float32)
    K[100:104, 0] = 4.0 * q[64 * 9:64 * 10, 0].mean(axis=0)
    I = hip.hip_prefill_select(q, K, "f32", S, (8,), (32,), 4, 16, 1)
    assert np.all(np.isin(np.arange(100, 104), I[9]))
