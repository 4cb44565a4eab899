"""Run one synthetic workload through the public API a few times (for profilers).

    python -m dynamic_sparse_attention_gb300.run_workload decode_1m --iters 4
    python -m dynamic_sparse_attention_gb300.run_workload prefill_16k --iters 2

Workloads (seeded generators of the `synth` module at the repository root):
  decode_1m    hip_select + sparse_attn_decode, context 1,048,576, 32/8 heads, d=128
  decode_128k  the same at context 131,072
  prefill_128k vs_index_build + sparse_attn_prefill, S=131072, 32/8 heads, d=128
  prefill_16k  the same at S=16384
  prefill_128k_h4  the same at S=131072 with 4 query heads / 1 KV head (the per-CTA tile
               counts of the 128K workload in about 0.3 GB of device memory)
  prefill_bs_32k  block_sparse_index_build (k_b=100) + sparse_attn_prefill at S=32768
  prefill_hip_16k  hip_prefill_select + hip_prefill_lists + sparse_attn_prefill at S=16384
                   (chunks 256 / 32 / 8, keep 4096 / 2048 / 1024, sink 256, window 1024)
  prefill_hip_128k_h4  the same at S=131072 with 4 query heads / 1 KV head and the 128K
                   stage table (keep 32768 / 8192 / 2048): the per-CTA tile counts of the
                   128K InfiniteHiP prefill in well under 1 GB of device memory
Each iteration launches the workload's kernels once on the current stream; nothing is
timed or checked.  The first iteration is a warm-up like any other, so a profiler
that skips the first launches of a kernel sees steady-state ones.
"""
from __future__ import annotations

import argparse
import os
import sys

import numpy as np


def _to_dev(a, torch):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()


def _decode(case, iters):
    import torch

    from . import binding as dsa
    q, k, v = _to_dev(case.q, torch), _to_dev(case.k, torch), _to_dev(case.v, torch)
    kv_len = torch.from_numpy(case.kv_len).cuda()
    cfg = dsa.HipConfig(case.chunk, case.keep, case.n_sink, case.n_stream)
    for _ in range(iters):
        sel, cnt = dsa.hip_select(q, k, kv_len, cfg)
        dsa.sparse_attn_decode(q, k, v, kv_len, sel, cnt, n_sink=case.n_sink, n_stream=case.n_stream)
    torch.cuda.synchronize()


def _prefill(case, iters):
    import torch

    from . import binding as dsa
    q, k, v = _to_dev(case.q, torch), _to_dev(case.k, torch), _to_dev(case.v, torch)
    for _ in range(iters):
        idx = dsa.vs_index_build(q, k, last_q=case.last_q, n_vertical=case.n_vertical,
                                 n_slash=case.n_slash)
        dsa.sparse_attn_prefill(q, k, v, idx["blk_cnt"], idx["blk_idx"], idx["col_cnt"],
                                idx["col_idx"])
    torch.cuda.synchronize()


def _prefill_bs(case, iters, k_b=100):
    import torch

    from . import binding as dsa
    q, k, v = _to_dev(case.q, torch), _to_dev(case.k, torch), _to_dev(case.v, torch)
    for _ in range(iters):
        idx = dsa.block_sparse_index_build(q, k, k_b=k_b)
        dsa.sparse_attn_prefill(q, k, v, idx["blk_cnt"], idx["blk_idx"], idx["col_cnt"], None)
    torch.cuda.synchronize()


def _prefill_hip(case, iters, cfg):
    import torch

    from . import binding as dsa
    q, k, v = _to_dev(case.q, torch), _to_dev(case.k, torch), _to_dev(case.v, torch)
    for _ in range(iters):
        sel, cnt = dsa.hip_prefill_select(q, k, cfg)
        lists = dsa.hip_prefill_lists(q, k, cfg, sel, cnt)
        dsa.sparse_attn_prefill(q, k, v, lists["blk_cnt"], lists["blk_idx"], lists["col_cnt"],
                                lists["col_idx"])
    torch.cuda.synchronize()


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    p.add_argument("workload", choices=["decode_1m", "decode_128k", "prefill_128k", "prefill_16k",
                                        "prefill_128k_h4", "prefill_bs_32k", "prefill_hip_16k",
                                        "prefill_hip_128k_h4"])
    p.add_argument("--iters", type=int, default=4)
    args = p.parse_args(argv)
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import synth

    from . import binding as dsa
    dsa.load()
    if args.workload == "decode_1m":
        _decode(synth.decode_1m(), args.iters)
    elif args.workload == "decode_128k":
        _decode(synth.decode_128k(), args.iters)
    elif args.workload == "prefill_128k":
        _prefill(synth.prefill_128k(), args.iters)
    elif args.workload == "prefill_128k_h4":
        _prefill(synth.prefill_case("prefill_vs_S131072_h4", S=131072, H_q=4, H_kv=1, D=128, seed=4),
                 args.iters)
    elif args.workload == "prefill_hip_16k":
        _prefill_hip(synth.prefill_case("prefill_hip_S16384", S=16384, H_q=32, H_kv=8, D=128, seed=4),
                     args.iters, dsa.HipConfig((256, 32, 8), (4096, 2048, 1024), 256, 1024))
    elif args.workload == "prefill_hip_128k_h4":
        _prefill_hip(synth.prefill_case("prefill_hip_S131072_h4", S=131072, H_q=4, H_kv=1, D=128, seed=4),
                     args.iters, dsa.HipConfig((256, 32, 8), (32768, 8192, 2048), 256, 1024))
    elif args.workload == "prefill_bs_32k":
        _prefill_bs(synth.prefill_case("prefill_bs_S32768", S=32768, H_q=32, H_kv=8, D=128, seed=4),
                    args.iters)
    else:
        _prefill(synth.prefill_case("prefill_vs_S16384", S=16384, H_q=32, H_kv=8, D=128, seed=4),
                 args.iters)
    print(f"{args.workload}: {args.iters} iterations done")


if __name__ == "__main__":
    main()
