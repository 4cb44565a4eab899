"""The tensor-core kernels' bounded waits, driven to expiry (GPU).

Every mbarrier wait of the prefill attention and of the two vertical-slash estimate
passes gives up after a limit; a CTA that gives up stops issuing work, drains its copies
and MMAs, frees its tensor memory and sets a device error word.  With the limit set to a
few nanoseconds (dsa_set_wait_limit) a wait that is not satisfied at its first try runs
out, so that path runs without any fault: every CTA either gave up (zero output) or
finished normally (correct output), and afterwards the default limit gives clean,
correct results again.
"""
import math

import numpy as np
import pytest
import torch

import dynamic_sparse_attention_gb300 as dsa
from dynamic_sparse_attention_gb300 import _build
from oracle import vs
from parity import attention_errors, to_dev
from synth import prefill_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    _build.build()
    dsa.load()
    yield
    dsa.set_wait_limit(0)


def _case():
    c = prefill_case("waits", S=4096, H_q=8, H_kv=2, D=128, seed=91, n_vertical=100,
                     n_slash=400)
    return c, to_dev(c.q, "bf16"), to_dev(c.k, "bf16"), to_dev(c.v, "bf16")


def _run(c, q, k, v):
    idx = dsa.vs_index_build(q, k, last_q=c.last_q, n_vertical=c.n_vertical, n_slash=c.n_slash)
    out, lse = dsa.sparse_attn_prefill(q, k, v, idx["blk_cnt"], idx["blk_idx"], idx["col_cnt"],
                                       idx["col_idx"])
    torch.cuda.synchronize()
    return idx, out, lse


def _lists(idx, h, m):
    nb, nc = int(idx["blk_cnt"][0, h, m]), int(idx["col_cnt"][0, h, m])
    return (idx["blk_idx"][0, h, m, :nb].cpu().numpy(), idx["col_idx"][0, h, m, :nc].cpu().numpy())


def test_expired_waits_give_up_cleanly_and_the_next_launch_is_correct():
    c, q, k, v = _case()
    assert dsa.device_error() == 0
    dsa.set_wait_limit(1)   # 1 ns: a wait not satisfied at its first try runs out
    try:
        idx, out, _ = _run(c, q, k, v)
        code = dsa.device_error()
    finally:
        dsa.set_wait_limit(0)
    assert code & 2, "no vertical-slash estimate CTA gave up a wait"
    assert code & 1, "no prefill attention CTA gave up a wait"
    # A CTA that gave up writes zeros for its rows; one whose waits were all satisfied at
    # the first try finished normally.  A CTA's rows are whole 64-row (head, query block)
    # units (two blocks of one head, or one block of two heads whose lists agree), so
    # every unit is one or the other, checked on the lists this run produced.
    o = out.float().cpu().numpy()
    nq = math.ceil(c.S / 64)
    n_zero = 0
    for h in range(c.H_q):
        for m in range(nq):
            rows = o[0, 64 * m:min(c.S, 64 * m + 64), h]
            if not rows.any():
                n_zero += 1
                continue
            blk, col = _lists(idx, h, m)
            O64, _ = vs.prefill_block_attention(c.q[0], c.k[0], c.v[0], h, c.G, m, blk, col,
                                                c.S, c.scale)
            mx, mn = attention_errors(o[0, 64 * m:64 * m + len(O64), h], O64)
            assert mx <= 1e-2 and mn <= 1e-3, (h, m, mx, mn)
    assert n_zero >= 1
    # the default limit: no error word, and the results match the fp64 oracle
    idx, out, lse = _run(c, q, k, v)
    assert dsa.device_error() == 0
    vert = idx["vertical"].cpu().numpy()[0]
    sl = idx["slash"].cpu().numpy()[0]
    o = out.float().cpu().numpy()
    for h in (0, 5):
        blk_o, col_o = vs.vs_convert(vert[h], sl[h], c.S)
        for m in (0, 17, nq - 1):
            blk, col = _lists(idx, h, m)
            assert np.array_equal(blk, blk_o[m]) and np.array_equal(col, col_o[m])
            O64, _ = vs.prefill_block_attention(c.q[0], c.k[0], c.v[0], h, c.G, m, blk, col,
                                                c.S, c.scale)
            mx, mn = attention_errors(o[0, 64 * m:64 * m + len(O64), h], O64)
            assert mx <= 1e-2 and mn <= 1e-3
