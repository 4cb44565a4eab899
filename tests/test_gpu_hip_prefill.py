"""GPU parity of the InfiniteHiP sparse prefill (per-64-row query block pruning, lists,
and the prefill kernel over them) against the fp64 oracle."""
import dataclasses

import numpy as np
import pytest
import torch

import dynamic_sparse_attention_gb300 as dsa
from dynamic_sparse_attention_gb300 import _build
from oracle import hip
from oracle.numerics import to_f64
from parity import attention_errors, check_hip_stage, to_dev
from synth import decode_case

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


class _Rows:
    """case.q / case.k seen per query-block row: q[r] is the block's rows, k[r] the keys."""

    def __init__(self, fn):
        self.fn = fn

    def __getitem__(self, r):
        return self.fn(r)


def _case(S, H_q, H_kv, D, chunk, keep, n_sink, n_stream, seed, plant="uniform", n_plant=16):
    c = decode_case("pf", B=1, T=S, T_q=1, H_q=H_q, H_kv=H_kv, D=D, dtype="bf16", chunk=chunk,
                    keep=keep, n_sink=n_sink, n_stream=n_stream, seed=seed, plant=plant,
                    n_plant=n_plant)
    # prefill queries: unit-variance rows of their own (the planted keys of the decode
    # generator stay in K)
    rng = np.random.default_rng(seed + 1000)
    from synth import f32_to_bf16_bits
    q = f32_to_bf16_bits(rng.standard_normal((S, H_q, D), dtype=np.float32))
    return c, q


def _run(c, q_bits, debug=True):
    q = to_dev(q_bits[None], "bf16")
    k = to_dev(c.k, "bf16")
    v = to_dev(c.v, "bf16")
    cfg = dsa.HipConfig(c.chunk, c.keep, c.n_sink, c.n_stream)
    res = dsa.hip_prefill_select(q, k, cfg, debug=debug)
    lists = dsa.hip_prefill_lists(q, k, cfg, res[0], res[1])
    out, lse = dsa.sparse_attn_prefill(q, k, v, lists["blk_cnt"], lists["blk_idx"], lists["col_cnt"],
                                       lists["col_idx"])
    torch.cuda.synchronize()
    return res, lists, out, lse


def _check(c, q_bits, res, out, lse, blocks):
    sel_idx, sel_cnt, dbg = res
    S = c.T_max
    view = dataclasses.replace(c, q=_Rows(lambda r: q_bits[64 * r:min(S, 64 * r + 64)]),
                               k=_Rows(lambda r: c.k[0]))
    q64 = to_f64(q_bits, "bf16")
    o = out.float().cpu().numpy()[0]
    lse_g = lse.cpu().numpy()[0]
    stats = {"flips": 0, "band_diffs": 0}
    for m in blocks:
        T_m = hip.prefill_block_len(S, m)
        I = hip.candidate_range(T_m, c.n_sink, c.n_stream)
        for i in range(len(c.chunk)):
            I = check_hip_stage(view, m, dbg, i, I, stats)
        final = sel_idx[m, :int(sel_cnt[m])].cpu().numpy().astype(np.int64)
        assert np.array_equal(final, I), f"block {m}: final selection differs from its replay"
        O64, lse64 = hip.prefill_attention(q64, c.k[0], c.v[0], "bf16", S, {m: final}, c.n_sink,
                                           c.n_stream, c.scale, c.G, blocks=[m])[m]
        r0 = 64 * m
        mx, mn = attention_errors(o[r0:r0 + len(O64)], O64)
        assert mx <= MAX_ABS and mn <= MEAN_ABS, f"block {m}: max {mx:.3e} mean {mn:.3e}"
        fin = np.isfinite(lse64)
        lg = lse_g[:, r0:r0 + len(O64)].T
        assert np.array_equal(fin, np.isfinite(lg))
        assert np.abs(lg[fin] - lse64[fin]).max(initial=0) <= 1e-3
    return stats


@pytest.mark.parametrize("S,D,G", [(1000, 128, 4), (700, 64, 1), (1500, 128, 8)])
def test_small_full_parity(S, D, G):
    H_kv = 2 if G < 8 else 1
    c, q = _case(S, H_kv * G, H_kv, D, chunk=(32, 8), keep=(256, 64), n_sink=16, n_stream=64,
                 seed=80 + S)
    res, lists, out, lse = _run(c, q)
    _check(c, q, res, out, lse, range((S + 63) // 64))


def test_keep_all_is_dense_causal():
    c, q = _case(900, 8, 2, 128, chunk=(16, 4), keep=(4096, 4096), n_sink=4, n_stream=16, seed=83,
                 plant="none")
    res, lists, out, lse = _run(c, q)
    qt = to_dev(q[None], "bf16").float().permute(0, 2, 1, 3)
    kt = to_dev(c.k, "bf16").float().permute(0, 2, 1, 3).repeat_interleave(4, 1)
    vt = to_dev(c.v, "bf16").float().permute(0, 2, 1, 3).repeat_interleave(4, 1)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=True).permute(0, 2, 1, 3)
    assert (out.float() - ref).abs().max().item() <= MAX_ABS


def test_three_stage_8k_sampled_blocks():
    """The pages' stage table (256 -> 32 -> 8 chunks) scaled to S = 8192: 32/8 heads."""
    c, q = _case(8192, 32, 8, 128, chunk=(256, 32, 8), keep=(4096, 1024, 256), n_sink=64,
                 n_stream=256, seed=84, n_plant=32)
    res, lists, out, lse = _run(c, q)
    _check(c, q, res, out, lse, [0, 5, 6, 40, 77, 127])


def test_prefill_128k_config_sampled():
    """S = 131072, 32/8 heads, d = 128, the pages' 3K stage table (chunks 256 / 32 / 8,
    keep 32768 / 8192 / 2048, sink 256, window 1024): sampled query blocks in full."""
    c, q = _case(131072, 32, 8, 128, chunk=(256, 32, 8), keep=(32768, 8192, 2048), n_sink=256,
                 n_stream=1024, seed=85, n_plant=64)
    res, lists, out, lse = _run(c, q)
    # 64 query blocks spread over the sequence (the first and last among them); every
    # block's selection is shared by all 32 heads and its attention is checked for all
    blocks = sorted(set([19, 20, 517] + np.linspace(0, 2047, 64).astype(int).tolist()))
    _check(c, q, res, out, lse, blocks)
