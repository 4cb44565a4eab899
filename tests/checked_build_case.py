"""Run by tests/test_gpu_checked_build.py in its own process with DSA_CHECKED=1: the
checked build (device-side input checks compiled in) must run valid inputs without a
report, and report -- while still skipping, not dereferencing -- out-of-range lengths,
counts, selected positions and list entries made on the host."""
import math
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
sys.path.insert(0, os.path.join(ROOT, "tests"))

import numpy as np  # noqa: E402
import torch  # noqa: E402

import dynamic_sparse_attention_gb300 as dsa  # noqa: E402
from dynamic_sparse_attention_gb300 import _build  # noqa: E402
from parity import to_dev  # noqa: E402
from synth import decode_case, prefill_case  # noqa: E402

CHECK = 4   # device_error bit of the checked build


def main():
    assert os.environ.get("DSA_CHECKED") == "1"
    dsa.load()
    assert dsa.library_path() == _build.LIB_CHECKED, dsa.library_path()
    dev = torch.device("cuda")
    assert dsa.device_error() == 0

    # ---- decode: valid selection, then bad positions / count / length
    for dtype, T_q in (("bf16", 1), ("bf16", 8)):   # the cluster kernel and the split path
        c = decode_case("chk", B=2, T=3000, T_q=T_q, H_q=8, H_kv=2, D=128, dtype=dtype,
                        chunk=(64, 16), keep=(512, 128), n_sink=16, n_stream=64, seed=5,
                        kv_len=[3000, 2500])
        q, k, v = to_dev(c.q, dtype), to_dev(c.k, dtype), to_dev(c.v, dtype)
        kv = torch.from_numpy(c.kv_len).to(dev)
        cfg = dsa.HipConfig(c.chunk, c.keep, c.n_sink, c.n_stream)
        sel, cnt = dsa.hip_select(q, k, kv, cfg)
        out, _ = dsa.sparse_attn_decode(q, k, v, kv, sel, cnt, n_sink=c.n_sink, n_stream=c.n_stream)
        torch.cuda.synchronize()
        assert dsa.device_error() == 0, "valid decode reported"
        bad = sel.clone()
        bad[0, 0] = 2999 + 50       # past the row's context
        bad[1, 3] = -7              # negative
        bad[1, 4] = c.n_sink - 1    # inside the sink
        out2, _ = dsa.sparse_attn_decode(q, k, v, kv, bad, cnt, n_sink=c.n_sink, n_stream=c.n_stream)
        torch.cuda.synchronize()
        assert dsa.device_error() & CHECK, "bad selected positions not reported"
        assert torch.isfinite(out2.float()).all()
        cnt_bad = cnt.clone()
        cnt_bad[0] = sel.shape[1] + 9
        dsa.sparse_attn_decode(q, k, v, kv, sel, cnt_bad, n_sink=c.n_sink, n_stream=c.n_stream)
        torch.cuda.synchronize()
        assert dsa.device_error() & CHECK, "bad selection count not reported"
        kv_bad = kv.clone()
        kv_bad[1] = c.T_max + 100
        dsa.hip_select(q, k, kv_bad, cfg)
        torch.cuda.synchronize()
        assert dsa.device_error() & CHECK, "bad kv_len not reported by the selection"

    # ---- prefill: valid lists, then bad block / column entries and counts
    p = prefill_case("chk", S=1000, H_q=4, H_kv=2, D=128, seed=6, n_vertical=40, n_slash=120)
    q, k, v = to_dev(p.q, "bf16"), to_dev(p.k, "bf16"), to_dev(p.v, "bf16")
    idx = dsa.vs_index_build(q, k, last_q=p.last_q, n_vertical=p.n_vertical, n_slash=p.n_slash)
    lists = [idx["blk_cnt"], idx["blk_idx"], idx["col_cnt"], idx["col_idx"]]
    out, _ = dsa.sparse_attn_prefill(q, k, v, *lists)
    torch.cuda.synchronize()
    assert dsa.device_error() == 0, "valid prefill reported"
    nq = math.ceil(p.S / 64)
    blk_idx = lists[1].clone()
    blk_idx[0, 1, 5, 0] = nq + 3                  # a key block past the sequence
    dsa.sparse_attn_prefill(q, k, v, lists[0], blk_idx, lists[2], lists[3])
    torch.cuda.synchronize()
    assert dsa.device_error() & CHECK, "bad block entry not reported"
    col_cnt, col_idx = lists[2].clone(), lists[3].clone()
    col_cnt[0, 2, nq - 1] = 3
    col_idx[0, 2, nq - 1, :3] = torch.tensor([5, p.S + 100, 7], dtype=torch.int32)
    out3, _ = dsa.sparse_attn_prefill(q, k, v, lists[0], lists[1], col_cnt, col_idx)
    torch.cuda.synchronize()
    assert dsa.device_error() & CHECK, "bad column entry not reported"
    assert torch.isfinite(out3.float()).all()
    blk_cnt = lists[0].clone()
    blk_cnt[0, 0, 3] = lists[1].shape[-1] + 1
    dsa.sparse_attn_prefill(q, k, v, blk_cnt, lists[1], lists[2], lists[3])
    torch.cuda.synchronize()
    assert dsa.device_error() & CHECK, "bad block count not reported"
    assert dsa.device_error() == 0   # read and cleared
    print("checked-build ok")


if __name__ == "__main__":
    main()
