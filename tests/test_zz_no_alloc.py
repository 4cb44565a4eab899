"""sparse_attn_decode_noalloc against sparse_attn_decode and the fp64 oracle (GPU).

The no-allocation variant is for callers that cannot allocate device memory when
they call the decode: a C engine or plug-in with no device allocator of its own,
or a latency-bound loop that must not call cudaMalloc (it can synchronise the
whole device).  Its split-K partials live in a fixed array inside the library
that every call reuses.  The cases here take the split path (more than 16 query
rows per KV head, or fp32 inputs), so the array really holds the partials, and
run back to back with different shapes and lengths: a call whose rows end early
must not merge what the previous call left in the array.  This file is collected
last on purpose.
"""
import numpy as np
import pytest
import torch

import dynamic_sparse_attention_gb300 as dsa
from dynamic_sparse_attention_gb300 import _build
from oracle import hip
from oracle.numerics import to_f64
from parity import attention_errors, to_dev
from synth import decode_case

pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS = 1e-2, 1e-3
SCRATCH_BYTES = 4 << 20


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    _build.build()
    dsa.load()


def _case(seed, B, T_q, dtype, kv_len, H_q=32, H_kv=8, D=128):
    c = decode_case("noalloc", B=B, T=6000, T_q=T_q, H_q=H_q, H_kv=H_kv, D=D, dtype=dtype,
                    chunk=(256, 64, 16), keep=(2048, 1024, 512), n_sink=64, n_stream=256,
                    seed=seed, kv_len=kv_len)
    q, k, v = to_dev(c.q, dtype), to_dev(c.k, dtype), to_dev(c.v, dtype)
    kv = torch.from_numpy(c.kv_len).cuda()
    cfg = dsa.HipConfig(c.chunk, c.keep, c.n_sink, c.n_stream)
    sel_idx, sel_cnt = dsa.hip_select(q, k, kv, cfg)
    return c, q, k, v, kv, sel_idx, sel_cnt


def _check_against_oracle(c, out, lse, sel_idx, sel_cnt):
    o = out.float().cpu().numpy()
    l = lse.cpu().numpy()
    for b in range(c.B):
        T = int(c.kv_len[b])
        I = sel_idx[b, :int(sel_cnt[b])].cpu().numpy()
        A = hip.attended_set(T, c.n_sink, c.n_stream, I)
        O64, lse64 = hip.decode_attention(to_f64(c.q[b], c.dtype), c.k[b], c.v[b], c.dtype, A,
                                          c.scale, c.G)
        mx, mn = attention_errors(o[b], O64)
        assert mx <= MAX_ABS and mn <= MEAN_ABS, f"row {b}: max {mx:.3e} mean {mn:.3e}"
        assert np.abs(l[b] - lse64).max() <= 1e-3


# Back-to-back calls: the first fills all 13 split slots of both rows (3.5 MB of
# partials); in the second, row 1's context (200 tokens) fills 4 of its 13 splits, so
# the other 9 must not merge the first call's leftovers; the third switches to fp32
# and another head layout.
CALLS = [
    dict(seed=61, B=2, T_q=8, dtype="bf16", kv_len=[6000, 5300]),
    dict(seed=62, B=2, T_q=8, dtype="bf16", kv_len=[5999, 200]),
    dict(seed=63, B=2, T_q=4, dtype="f32", kv_len=[4100, 6000], H_q=8, H_kv=2, D=64),
]


def test_noalloc_split_path_matches_workspace_version_and_oracle():
    for kw in CALLS:
        c, q, k, v, kv, sel_idx, sel_cnt = _case(**kw)
        need = dsa.sparse_attn_decode_workspace_bytes(q, k, sel_idx.shape[1], c.n_sink, c.n_stream)
        # the split path: its partials are what the built-in array holds
        assert 0 < need <= SCRATCH_BYTES, need
        ref, ref_lse = dsa.sparse_attn_decode(q, k, v, kv, sel_idx, sel_cnt,
                                              n_sink=c.n_sink, n_stream=c.n_stream)
        got, got_lse = dsa.sparse_attn_decode_noalloc(q, k, v, kv, sel_idx, sel_cnt,
                                                      n_sink=c.n_sink, n_stream=c.n_stream)
        torch.cuda.synchronize()
        d = (got.float() - ref.float()).abs()
        assert d.max().item() <= MAX_ABS and d.mean().item() <= MEAN_ABS, kw
        assert (got_lse - ref_lse).abs().max().item() <= 1e-3, kw
        _check_against_oracle(c, got, got_lse, sel_idx, sel_cnt)


def test_noalloc_rejects_oversized_requests():
    """B=8, T_q=8, 32/8 heads, d=128: 8 * 5 splits * 8 * 32 * 130 * 4 B = 5.3 MB > 4 MiB."""
    dev = torch.device("cuda")
    B, T, T_q = 8, 1024, 8
    q = torch.zeros(B, T_q, 32, 128, dtype=torch.bfloat16, device=dev)
    k = torch.zeros(B, T, 8, 128, dtype=torch.bfloat16, device=dev)
    v = torch.zeros_like(k)
    kv_len = torch.full((B,), T, dtype=torch.int32, device=dev)
    sel_idx = torch.zeros(B, 512, dtype=torch.int32, device=dev)
    sel_cnt = torch.zeros(B, dtype=torch.int32, device=dev)
    need = dsa.sparse_attn_decode_workspace_bytes(q, k, 512, 64, 256)
    assert need > SCRATCH_BYTES
    with pytest.raises(dsa.DsaError) as ei:
        dsa.sparse_attn_decode_noalloc(q, k, v, kv_len, sel_idx, sel_cnt, n_sink=64, n_stream=256)
    assert ei.value.status == -3 and "built-in array" in str(ei.value)
