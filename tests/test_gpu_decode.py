"""GPU parity of the decode half (hip_select + sparse_attn_decode) against the fp64 oracle."""
import dataclasses

import numpy as np
import pytest
import torch

import dynamic_sparse_attention_gb300 as dsa
from dynamic_sparse_attention_gb300 import _build
from oracle import hip
from oracle.numerics import to_f64
from parity import attention_errors, check_hip_row, check_hip_stage, from_dev_bits, to_dev
from synth import (decode_128k, decode_1m, decode_batch16, decode_case, decode_steps, decode_tiny,
                   with_fp8_kv)

pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS = 1e-2, 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    _build.build()
    dsa.load()


def _run(case):
    q = to_dev(case.q, case.dtype)
    k = to_dev(case.k, case.kvd)
    v = to_dev(case.v, case.kvd)
    kv_len = torch.from_numpy(case.kv_len).cuda()
    cfg = dsa.HipConfig(case.chunk, case.keep, case.n_sink, case.n_stream)
    sel_idx, sel_cnt, dbg = dsa.hip_select(q, k, kv_len, cfg, debug=True)
    out, lse = dsa.sparse_attn_decode(q, k, v, kv_len, sel_idx, sel_cnt, n_sink=case.n_sink,
                                      n_stream=case.n_stream)
    torch.cuda.synchronize()
    return sel_idx, sel_cnt, dbg, out, lse


def _check_case(case, rows=None):
    sel_idx, sel_cnt, dbg, out, lse = _run(case)
    o_gpu = from_dev_bits(out)
    if case.dtype == "bf16":
        o_gpu = to_f64(o_gpu, "bf16")
    lse_gpu = lse.cpu().numpy()
    report = []
    for b in (range(case.B) if rows is None else rows):
        I, stats = check_hip_row(case, b, dbg, sel_idx, sel_cnt)
        T = int(case.kv_len[b])
        A = hip.attended_set(T, case.n_sink, case.n_stream, I)
        q64 = to_f64(case.q[b], case.dtype)
        O64, lse64 = hip.decode_attention(q64, case.k[b], case.v[b], case.kvd, A, case.scale,
                                          case.G)
        mx, mn = attention_errors(o_gpu[b], O64)
        assert mx <= MAX_ABS and mn <= MEAN_ABS, f"row {b}: max {mx:.3e} mean {mn:.3e}"
        fin = np.isfinite(lse64)
        assert np.array_equal(fin, np.isfinite(lse_gpu[b]))
        assert np.abs(lse_gpu[b][fin] - lse64[fin]).max(initial=0) <= 1e-3
        report.append((b, stats, mx, mn))
    return report


def test_tiny_fp32_config():
    """1 head, d=64, fp32, 32 query rows, 64->16->4 chunks (the small oracle case)."""
    _check_case(decode_tiny())


@pytest.mark.parametrize("D,dtype", [(64, "bf16"), (128, "bf16"), (128, "f32"), (64, "f32")])
def test_gqa_small_ragged(D, dtype):
    """GQA, ragged batch lengths, partial last chunks, several tiles and splits."""
    c = decode_case("ragged", B=3, T=5000, T_q=1, H_q=8, H_kv=2, D=D, dtype=dtype,
                    chunk=(64, 16, 4), keep=(1024, 256, 64), n_sink=13, n_stream=100, seed=31,
                    plant="uniform", n_plant=16, kv_len=[5000, 3333, 1210])
    _check_case(c)


def test_multi_row_query_block():
    c = decode_case("block", B=2, T=3000, T_q=4, H_q=4, H_kv=1, D=128, dtype="bf16",
                    chunk=(32, 8), keep=(512, 128), n_sink=8, n_stream=32, seed=32,
                    plant="none", kv_len=[3000, 2001])
    _check_case(c)


def test_edge_cases_short_contexts():
    """Contexts shorter than sink + window, empty candidate ranges, keep-all stages."""
    c = decode_case("short", B=4, T=700, T_q=1, H_q=4, H_kv=4, D=64, dtype="bf16",
                    chunk=(16, 4), keep=(4096, 64), n_sink=32, n_stream=64, seed=33,
                    plant="none", kv_len=[700, 96, 50, 97])
    _check_case(c)


def test_non_power_of_two_chunks():
    c = decode_case("odd", B=1, T=4000, T_q=2, H_q=6, H_kv=3, D=64, dtype="f32",
                    chunk=(100, 13, 3), keep=(1300, 390, 90), n_sink=5, n_stream=21, seed=34,
                    plant="none")
    _check_case(c)


def test_more_chunks_than_register_topk():
    """Stage 0 with 17,971 chunks: past the register-resident top-K (16,384 chunks), so
    the selection takes the general kernel; stage 1 takes the register one."""
    c = decode_case("many", B=1, T=36000, T_q=1, H_q=2, H_kv=1, D=64, dtype="bf16",
                    chunk=(2, 1), keep=(4096, 1024), n_sink=7, n_stream=50, seed=36,
                    plant="uniform", n_plant=8)
    _check_case(c)


def test_topk_ties_in_boundary_bucket():
    """Keys repeat with period 61, so chunk scores take few distinct values and the
    bucket holding the K-th score holds several equal scores: ties go to the smaller
    chunk index."""
    c = decode_case("ties", B=1, T=12000, T_q=1, H_q=4, H_kv=1, D=64, dtype="bf16",
                    chunk=(16, 4), keep=(2048, 512), n_sink=4, n_stream=32, seed=37,
                    plant="none")
    c.k[0, 61:] = c.k[0, np.arange(61, 12000) % 61]
    _check_case(c)


def test_topk_all_scores_equal():
    """A zero query makes every chunk score 0: more equal scores than the exact-rank
    path takes, so the selection falls back to the radix select."""
    c = decode_case("zeroq", B=1, T=20000, T_q=1, H_q=4, H_kv=2, D=64, dtype="bf16",
                    chunk=(8, 2), keep=(4096, 1024), n_sink=4, n_stream=32, seed=38,
                    plant="none")
    c.q[:] = 0
    _check_case(c)


def test_dense_keep_all_matches_sdpa():
    c = decode_case("dense", B=2, T=1500, T_q=1, H_q=8, H_kv=2, D=128, dtype="bf16",
                    chunk=(64, 16), keep=(1 << 14, 1 << 14), n_sink=4, n_stream=16, seed=35,
                    plant="none")
    sel_idx, sel_cnt, dbg, out, lse = _run(c)
    assert np.array_equal(sel_cnt.cpu().numpy(), [1500 - 20] * 2)
    qt = to_dev(c.q, "bf16").float().permute(0, 2, 1, 3)
    kt = to_dev(c.k, "bf16").float().permute(0, 2, 1, 3).repeat_interleave(4, 1)
    vt = to_dev(c.v, "bf16").float().permute(0, 2, 1, 3).repeat_interleave(4, 1)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt).permute(0, 2, 1, 3)
    assert (out.float() - ref).abs().max().item() <= MAX_ABS


def test_value_shift_metamorphic():
    c = decode_case("shift", B=1, T=3000, T_q=1, H_q=8, H_kv=2, D=128, dtype="f32",
                    chunk=(64, 8), keep=(512, 128), n_sink=8, n_stream=64, seed=36)
    q, k, v = to_dev(c.q, "f32"), to_dev(c.k, "f32"), to_dev(c.v, "f32")
    kv_len = torch.from_numpy(c.kv_len).cuda()
    cfg = dsa.HipConfig(c.chunk, c.keep, c.n_sink, c.n_stream)
    sel_idx, sel_cnt = dsa.hip_select(q, k, kv_len, cfg)
    o1, _ = dsa.sparse_attn_decode(q, k, v, kv_len, sel_idx, sel_cnt, n_sink=8, n_stream=64)
    o2, _ = dsa.sparse_attn_decode(q, k, v + 0.5, kv_len, sel_idx, sel_cnt, n_sink=8, n_stream=64)
    sel2, cnt2 = dsa.hip_select(q * 2.0, k, kv_len, cfg)  # exact scaling: same decisions
    assert torch.equal(sel_idx, sel2) and torch.equal(sel_cnt, cnt2)
    assert (o2 - o1 - 0.5).abs().max().item() < 1e-5


def test_gqa_128k_config():
    """Llama-3-8B-shaped GQA decode at context 131072 (full size, replay parity)."""
    _check_case(decode_128k())


def test_gqa_1m_config():
    """The bench's decode workload at full size: context 1,048,576, 32/8 heads, d=128,
    4 pruning stages (4092 stage-0 chunks), in the launch configuration the bench times.
    Every stage is replayed against the oracle and the attention checked in full."""
    report = _check_case(decode_1m())
    assert report[0][1]["band_diffs"] <= 4


def test_batch16_config():
    """Batch 16 at 32K with one planted cluster per row (checks rows 0, 7 and 15 in full)."""
    _check_case(decode_batch16(), rows=[0, 7, 15])


# ------------------------------------------------------------ mask caching (section 3.4)

def _cache_case():
    return decode_case("decode_cache_B2_T16384", B=2, T=16384, T_q=1, H_q=32, H_kv=8, D=128,
                       dtype="bf16", chunk=(256, 64, 16, 4), keep=(2048, 1024, 512, 256),
                       n_sink=64, n_stream=256, seed=50, plant="uniform", n_plant=32,
                       kv_len=[16000, 11001])


def _upload(c):
    return (to_dev(c.q, c.dtype), to_dev(c.k, c.dtype), to_dev(c.v, c.dtype),
            torch.from_numpy(c.kv_len).cuda(), dsa.HipConfig(c.chunk, c.keep, c.n_sink, c.n_stream))


def test_cached_with_every_stage_is_hip_select():
    c = _cache_case()
    q, k, v, kv_len, cfg = _upload(c)
    ref_idx, ref_cnt, ref_dbg = dsa.hip_select(q, k, kv_len, cfg, debug=True)
    ws = torch.zeros(dsa.hip_select_workspace_bytes(q, k, cfg), dtype=torch.uint8, device="cuda")
    out = (torch.full_like(ref_idx, -9), torch.full_like(ref_cnt, -9))
    idx, cnt, dbg = dsa.hip_select_cached(q, k, kv_len, cfg, 0b1111, out=out, workspace=ws,
                                          debug=True)
    torch.cuda.synchronize()
    assert torch.equal(idx, ref_idx) and torch.equal(cnt, ref_cnt)
    for key in ref_dbg:
        for a, b in zip(dbg[key], ref_dbg[key]):
            torch.testing.assert_close(a, b, rtol=0, atol=0, equal_nan=True)


def test_cached_without_refresh_changes_nothing():
    c = _cache_case()
    q, k, v, kv_len, cfg = _upload(c)
    cache = dsa.HipSelectCache(q, k, cfg, (4, 2, 1, 1))
    idx, cnt = cache(q, k, kv_len)
    before = (idx.clone(), cnt.clone(), cache.workspace.clone())
    q2 = torch.randn_like(q)
    dsa.hip_select_cached(q2, k, kv_len + 7, cfg, 0, out=(cache.sel_idx, cache.sel_cnt),
                          workspace=cache.workspace)
    torch.cuda.synchronize()
    assert torch.equal(cache.sel_idx, before[0]) and torch.equal(cache.sel_cnt, before[1])
    assert torch.equal(cache.workspace, before[2])


@pytest.mark.parametrize("n_refresh", [(4, 2, 1, 1), (4, 3, 2, 1)])
def test_cached_decoding_loop_against_oracle(n_refresh):
    """Ten decoding steps, one new token and a drifting query per step.  Each refreshed
    stage is replayed against the oracle from the list the GPU holds for the stage
    before it (fresh or cached); skipped stages must leave their lists alone; the
    attention of every step is checked over sink + cached selection + current window.
    (4, 3, 2, 1) does not nest, so a stage can be refreshed while the one before it
    stays cached."""
    c = _cache_case()
    _, k, v, _, cfg = _upload(c)
    steps = decode_steps(c, 10, seed=51)
    cache = None
    held = [[None] * c.B for _ in c.chunk]
    for s, (q_np, kv_np) in enumerate(steps):
        cs = dataclasses.replace(c, q=q_np, kv_len=kv_np)
        q = to_dev(q_np, c.dtype)
        kv_len = torch.from_numpy(kv_np).cuda()
        if cache is None:
            cache = dsa.HipSelectCache(q, k, cfg, n_refresh)
        mask = cache.mask()
        assert mask == hip_refresh_bits(s, n_refresh)
        idx, cnt, dbg = cache(q, k, kv_len, debug=True)
        out, _ = dsa.sparse_attn_decode(q, k, v, kv_len, idx, cnt, n_sink=c.n_sink,
                                        n_stream=c.n_stream)
        torch.cuda.synchronize()
        o_gpu = to_f64(from_dev_bits(out), "bf16")
        stats = {"flips": 0, "band_diffs": 0}
        for b in range(c.B):
            T = int(kv_np[b])
            for i in range(len(c.chunk)):
                if mask >> i & 1:
                    I = hip.candidate_range(T, c.n_sink, c.n_stream) if i == 0 else held[i - 1][b]
                    held[i][b] = check_hip_stage(cs, b, dbg, i, I, stats)
                else:
                    assert int(dbg["stage_cnt"][i][b]) == -7, "a cached stage ran"
            final = idx[b, :int(cnt[b])].cpu().numpy().astype(np.int64)
            assert np.array_equal(final, held[-1][b])
            A = hip.attended_set(T, c.n_sink, c.n_stream, final)
            assert len(np.unique(A)) == len(A)
            O64, _ = hip.decode_attention(to_f64(q_np[b], c.dtype), c.k[b], c.v[b], c.dtype, A,
                                          c.scale, c.G)
            mx, mn = attention_errors(o_gpu[b], O64)
            assert mx <= MAX_ABS and mn <= MEAN_ABS, f"step {s} row {b}: max {mx:.3e} mean {mn:.3e}"


def hip_refresh_bits(step, n_refresh):
    return sum(1 << i for i, r in enumerate(hip.refresh_schedule(step, n_refresh)) if r)


def test_cached_lists_are_clamped_to_the_key_rows():
    """A workspace that never held a selection (arbitrary ints as cached lists and
    counts): the later stages and the attention read only rows inside the context."""
    c = _cache_case()
    q, k, v, kv_len, cfg = _upload(c)
    nbytes = dsa.hip_select_workspace_bytes(q, k, cfg)
    g = torch.Generator(device="cpu").manual_seed(52)
    junk = torch.randint(-(1 << 31), (1 << 31) - 1, (nbytes // 4,), generator=g, dtype=torch.int64)
    ws = junk.to(torch.int32).view(torch.uint8).cuda()
    out = (torch.empty(c.B, c.keep[-1], dtype=torch.int32, device="cuda"),
           torch.empty(c.B, dtype=torch.int32, device="cuda"))
    idx, cnt = dsa.hip_select_cached(q, k, kv_len, cfg, 0b1110, out=out, workspace=ws)
    o, lse = dsa.sparse_attn_decode(q, k, v, kv_len, idx, cnt, n_sink=c.n_sink,
                                    n_stream=c.n_stream)
    torch.cuda.synchronize()
    assert dsa.device_error() == 0
    assert ((cnt >= 0) & (cnt <= c.keep[-1])).all()
    assert torch.isfinite(o.float()).all()


# ------------------------------------------------------------ FP8 E4M3 keys and values

def test_fp8_kv_small_ragged():
    """bf16 queries over FP8 E4M3 keys and values: selection replayed against the oracle
    on the decoded keys, attention against the fp64 oracle (ragged batch, partial chunks)."""
    c = with_fp8_kv(decode_case("ragged", B=3, T=5000, T_q=1, H_q=8, H_kv=2, D=128,
                                dtype="bf16", chunk=(64, 16, 4), keep=(1024, 256, 64), n_sink=13,
                                n_stream=100, seed=31, plant="uniform", n_plant=16,
                                kv_len=[5000, 3333, 1210]))
    assert c.k.dtype == np.uint8 and c.kvd == "e4m3"
    _check_case(c)


def test_fp8_kv_sixteen_rows_per_kv_head():
    c = with_fp8_kv(decode_case("block", B=2, T=3000, T_q=4, H_q=8, H_kv=2, D=128, dtype="bf16",
                                chunk=(32, 8), keep=(512, 128), n_sink=8, n_stream=32, seed=39,
                                plant="none", kv_len=[3000, 2001]))
    _check_case(c)


def test_fp8_kv_128k_config():
    """The 128K GQA workload with its keys and values rounded to FP8 E4M3."""
    _check_case(with_fp8_kv(decode_128k()))


def test_fp8_kv_matches_float8_tensors():
    """A float8_e4m3fn tensor and a uint8 tensor of the same codes give the same results."""
    c = with_fp8_kv(decode_case("f8", B=1, T=2000, T_q=1, H_q=4, H_kv=1, D=128, dtype="bf16",
                                chunk=(32, 8), keep=(256, 64), n_sink=4, n_stream=16, seed=40))
    q = to_dev(c.q, "bf16")
    k8, v8 = to_dev(c.k, "e4m3"), to_dev(c.v, "e4m3")
    kv_len = torch.from_numpy(c.kv_len).cuda()
    cfg = dsa.HipConfig(c.chunk, c.keep, c.n_sink, c.n_stream)
    s1, n1 = dsa.hip_select(q, k8, kv_len, cfg)
    o1, _ = dsa.sparse_attn_decode(q, k8, v8, kv_len, s1, n1, n_sink=4, n_stream=16)
    kf, vf = k8.view(torch.float8_e4m3fn), v8.view(torch.float8_e4m3fn)
    s2, n2 = dsa.hip_select(q, kf, kv_len, cfg)
    o2, _ = dsa.sparse_attn_decode(q, kf, vf, kv_len, s2, n2, n_sink=4, n_stream=16)
    torch.cuda.synchronize()
    assert torch.equal(s1, s2) and torch.equal(n1, n2) and torch.equal(o1, o2)
