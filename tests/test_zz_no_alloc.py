"""sparse_attn_decode_noalloc against sparse_attn_decode (GPU).

The no-allocation variant exists for callers that cannot allocate device memory
when they call the decode (a C engine or plug-in without its own allocator, or a
latency-bound loop that must not call cudaMalloc).  Its split-K scratch is a
fixed array inside the library that every call reuses, so the check runs two
calls in a row with different inputs: the second must not see the first call's
leftovers.  This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

import dynamic_sparse_attention_gb300 as dsa
from dynamic_sparse_attention_gb300 import _build
from parity import to_dev
from synth import decode_case

pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS = 1e-2, 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    _build.build()
    dsa.load()


def _case(seed, B):
    c = decode_case("noalloc", B=B, T=6000, T_q=1, H_q=32, H_kv=8, D=128, dtype="bf16",
                    chunk=(256, 64, 16), keep=(2048, 1024, 512), n_sink=64, n_stream=256,
                    seed=seed, kv_len=[6000 - 700 * b for b in range(B)])
    q, k, v = to_dev(c.q, "bf16"), to_dev(c.k, "bf16"), to_dev(c.v, "bf16")
    kv_len = torch.from_numpy(c.kv_len).cuda()
    cfg = dsa.HipConfig(c.chunk, c.keep, c.n_sink, c.n_stream)
    sel_idx, sel_cnt = dsa.hip_select(q, k, kv_len, cfg)
    return c, q, k, v, kv_len, sel_idx, sel_cnt


def test_noalloc_matches_workspace_version_twice():
    for seed, B in ((61, 3), (62, 2)):   # two calls in a row, different inputs and shapes
        c, q, k, v, kv_len, sel_idx, sel_cnt = _case(seed, B)
        ref, ref_lse = dsa.sparse_attn_decode(q, k, v, kv_len, sel_idx, sel_cnt,
                                              n_sink=c.n_sink, n_stream=c.n_stream)
        got, got_lse = dsa.sparse_attn_decode_noalloc(q, k, v, kv_len, sel_idx, sel_cnt,
                                                      n_sink=c.n_sink, n_stream=c.n_stream)
        torch.cuda.synchronize()
        d = (got.float() - ref.float()).abs()
        assert d.max().item() <= MAX_ABS and d.mean().item() <= MEAN_ABS
        assert (got_lse - ref_lse).abs().max().item() <= 1e-3


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
    assert need > 4 << 20
    with pytest.raises(dsa.DsaError) as ei:
        dsa.sparse_attn_decode_noalloc(q, k, v, kv_len, sel_idx, sel_cnt, n_sink=64, n_stream=256)
    assert ei.value.status == -3 and "built-in array" in str(ei.value)
