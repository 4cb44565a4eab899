"""Comparison helpers: CUDA path vs the fp64 oracle (test code).

Selection parity follows a replay rule.  Tournament branch decisions, chunk
top-K and VS top-k are integer decisions taken from fp32 scores on the GPU
and fp64 scores in the oracle, so they may legitimately differ where two
scores are within the tie band (1e-3 relative).  The checks therefore:
  * walk the GPU's tournament path in fp64 and accept every branch that
    agrees with fp64 or lies inside the band;
  * check the GPU's fp32 representative scores against fp64;
  * check the GPU's kept set exactly against the top-K rule applied to its
    own fp32 scores, and against fp64 scores outside the band;
  * continue the next stage from the GPU's (validated) list.
"""
from __future__ import annotations

import numpy as np
import torch

from oracle import hip
from oracle.numerics import to_f64

REL_BAND = 1e-3


def to_dev(a: np.ndarray, dtype: str) -> torch.Tensor:
    """Stored bit patterns -> CUDA tensor of the matching torch dtype (FP8 E4M3 codes
    travel as uint8: the library reads the bytes)."""
    if dtype == "e4m3":
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)).cuda()
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def from_dev_bits(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return t.cpu().view(torch.int16).numpy().view(np.uint16)
    return t.cpu().numpy()


def near_tie(a, b, floor):
    return np.abs(a - b) <= REL_BAND * np.maximum(np.abs(a), np.abs(b)) + floor


def _scores(q64, K, dtype, pos, G):
    """fp64 block scores max_t q_t . k for positions pos [H_q, n] (head h reads KV h // G)."""
    H_q = q64.shape[1]
    g = (np.arange(H_q) // G)[:, None]
    keys = to_f64(K[pos, g], dtype)
    return np.einsum("thd,hnd->thn", q64, keys).max(axis=0)


def _abs_scale(q64, K, dtype, pos, G):
    """max_t sum_d |q_td k_d|: the magnitude an fp32 dot-product error scales with."""
    H_q = q64.shape[1]
    g = (np.arange(H_q) // G)[:, None]
    keys = np.abs(to_f64(K[pos, g], dtype))
    return np.einsum("thd,hnd->thn", np.abs(q64), keys).max(axis=0)


def check_tournament(q64, K, dtype, chunks, reps_gpu, rho_gpu, G, D):
    """Walk the GPU's SelectRep path for every (head, chunk) in fp64."""
    H_q = q64.shape[1]
    n = len(chunks)
    Lmax = max(len(c) for c in chunks)
    lens = np.array([len(c) for c in chunks])
    pos = np.empty((n, Lmax), np.int64)
    for j, c in enumerate(chunks):
        pos[j, :len(c)] = c
        pos[j, len(c):] = c[-1]
    cols = np.arange(n)[None, :]
    # GPU rep -> offset inside its chunk
    r_off = np.empty((H_q, n), np.int64)
    for j in range(n):
        o = np.searchsorted(chunks[j], reps_gpu[:, j])
        assert np.all(o < lens[j]) and np.all(chunks[j][np.minimum(o, lens[j] - 1)] == reps_gpu[:, j]), \
            f"chunk {j}: GPU representative not inside the chunk"
        r_off[:, j] = o
    floor = 1e-6 * np.sqrt(D)
    a = np.zeros((H_q, n), np.int64)
    b = np.broadcast_to(lens - 1, (H_q, n)).copy()
    flips = 0
    while True:
        act = a < b
        if not act.any():
            break
        mid = np.where(act, (a + b + 1) // 2, a)
        s1 = _scores(q64, K, dtype, pos[cols, a], G)
        s2 = _scores(q64, K, dtype, pos[cols, mid], G)
        gpu_right = r_off >= mid
        f64_right = s2 > s1
        dis = act & (gpu_right != f64_right)
        if dis.any():
            ok = near_tie(s1[dis], s2[dis], floor)
            assert ok.all(), f"{(~ok).sum()} tournament decisions differ outside the tie band"
            flips += int(dis.sum())
        a = np.where(act & gpu_right, mid, a)
        b = np.where(act & ~gpu_right, mid - 1, b)
    assert np.array_equal(a, r_off), "GPU representative is not the end of its own path"
    rho64 = _scores(q64, K, dtype, pos[cols, a], G)
    mag = _abs_scale(q64, K, dtype, pos[cols, a], G)
    err = np.abs(rho_gpu.astype(np.float64) - rho64)
    assert np.all(err <= 2e-6 * mag + 1e-6), f"representative scores off by up to {err.max():.3e}"
    return rho64, flips


def check_topk(s_gpu32, s64, K, kept_gpu, D):
    """Exact against the rule on GPU scores; band rule against fp64 scores."""
    n = len(s_gpu32)
    want_exact = hip.topk_chunks(s_gpu32.astype(np.float64), K)
    assert np.array_equal(kept_gpu, want_exact), "GPU top-K differs from the rule on its own scores"
    if n <= K:
        return 0
    order = np.lexsort((np.arange(n), -s64))
    hi, lo = s64[order[K - 1]], s64[order[K]]
    tol = REL_BAND * max(abs(hi), abs(lo)) + 1e-6 * np.sqrt(D)
    kept = np.zeros(n, bool)
    kept[kept_gpu] = True
    if hi - lo > tol:
        assert np.array_equal(np.sort(order[:K]), kept_gpu), "top-K set differs outside the tie band"
        return 0
    assert kept[s64 > hi + tol].all(), "a chunk above the tie band was dropped"
    assert not kept[s64 < lo - tol].any(), "a chunk below the tie band was kept"
    return int(np.sum(kept != np.isin(np.arange(n), order[:K])))


def check_hip_stage(case, b, dbg, i, I, stats):
    """Replay pruning stage i of batch row b from the input list I against the GPU's
    debug outputs of that stage; returns the GPU's (validated) output list."""
    q64 = to_f64(case.q[b], case.dtype)
    L, keep = case.chunk[i], case.keep[i]
    chunks = hip.chunk_partition(np.asarray(I, np.int64), L)
    n = len(chunks)
    cnt = int(dbg["stage_cnt"][i][b])
    lst = dbg["stage_idx"][i][b].cpu().numpy()
    if n == 0:
        assert cnt == 0 and np.all(lst == -1)
        return np.zeros(0, np.int64)
    reps = dbg["rep"][i][b, :, :n].cpu().numpy().astype(np.int64)
    rho = dbg["rep_score"][i][b, :, :n].cpu().numpy()
    s_gpu = dbg["chunk_score"][i][b, :n].cpu().numpy()
    rho64, flips = check_tournament(q64, case.k[b], case.kvd, chunks, reps, rho, case.G, case.D)
    stats["flips"] += flips
    assert np.array_equal(s_gpu, rho.max(axis=0)), "chunk score is not the max over heads"
    s64 = rho64.max(axis=0)
    # kept chunks from the GPU list
    got = lst[:cnt].astype(np.int64)
    assert np.all(lst[cnt:] == -1), "list not padded with -1"
    pos_in = {int(p): x for x, p in enumerate(I)}
    kept_gpu = np.unique([pos_in[int(p)] // L for p in got]) if cnt else np.zeros(0, np.int64)
    stats["band_diffs"] += check_topk(s_gpu, s64, keep // L, kept_gpu, case.D)
    want_list = hip.assemble(chunks, kept_gpu)
    assert np.array_equal(got, want_list), "assembled list differs"
    return got


def check_hip_row(case, b, dbg, sel_idx, sel_cnt):
    """Full replay check of one batch row's pruning stages; returns the GPU's final list."""
    I = hip.candidate_range(int(case.kv_len[b]), case.n_sink, case.n_stream)
    stats = {"flips": 0, "band_diffs": 0}
    for i in range(len(case.chunk)):
        I = check_hip_stage(case, b, dbg, i, I, stats)
    final = sel_idx[b, :int(sel_cnt[b])].cpu().numpy().astype(np.int64)
    assert np.array_equal(final, I)
    return I, stats


def attention_errors(o_gpu: np.ndarray, o64: np.ndarray):
    d = np.abs(o_gpu.astype(np.float64) - o64)
    return float(d.max()), float(d.mean())


def check_topk_list(vals32: np.ndarray, vals64: np.ndarray, k: int, got: np.ndarray, floor=1e-7):
    """VS top-k: exact against the rule on the GPU's fp32 values, band rule against fp64."""
    from oracle import vs as ovs
    want = ovs.topk_ascending(vals32.astype(np.float64), k)
    assert np.array_equal(got, want), "GPU top-k differs from the rule on its own values"
    n = len(vals64)
    if k >= n or k == 0:
        return 0
    order = np.lexsort((np.arange(n), -vals64))
    hi, lo = vals64[order[k - 1]], vals64[order[k]]
    tol = REL_BAND * max(abs(hi), abs(lo)) + floor
    kept = np.zeros(n, bool)
    kept[got] = True
    if hi - lo > tol:
        assert np.array_equal(np.sort(order[:k]), got), "top-k differs outside the tie band"
        return 0
    assert kept[vals64 > hi + tol].all(), "an entry above the tie band was dropped"
    assert not kept[vals64 < lo - tol].any(), "an entry below the tie band was kept"
    return int(np.sum(kept != np.isin(np.arange(n), order[:k])))
