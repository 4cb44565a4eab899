#!/usr/bin/env python
"""Benchmark of the sparse-attention hot path on GB300.

One step = one pass of the whole hot path on synthetic input:
  decode : hip_select (4 pruning stages) + sparse_attn_decode at context 1,048,576
           (32 query / 8 KV heads, d=128, bf16, keep 32768/16384/8192/4096, sink 128,
           window 1024, full re-selection every step);
  prefill: vs_index_build + sparse_attn_prefill at S=131072 (32/8 heads, d=128, bf16,
           top 1000 vertical / 6096 slash, 64x64 tiles).
The printed line carries decode us/step (the headline `value`, CUDA-graph replay),
prefill ms, the roofline of each half's dominant kernel (CUDA-event durations of
that kernel inside the run), an end-to-end number through the public API with
host buffers, SM clocks sampled during the timed region, and the fp64 oracle
timed on the host cores.  `--impl reference` times the oracle alone.

Launch: python bench.py [--gpus N --steps K --warmup W]; for N > 1 under
torch.distributed.run every rank runs its own replica (weak scaling).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "sparse-attn decode μs/step @1M ctx; prefill ms @128K; % HBM / TC roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# the nominal denominators the targets are stated against: about 8 TB/s of HBM3e and the
# dense bf16 tensor-core peak of a GB300 (2.25 PFLOP/s)
NOMINAL_HBM_GBS = 8000.0
NOMINAL_BF16_TFLOPS = 2250.0
# DRAM bytes read + written per launch, from ncu captures of the kernels as they are
# now (profiles/hip_stage_score_s0_decode_1m.md, profiles/prefill_attention_tc_S131072.md);
# keyed by (kernel, workload).  Remove an entry when its kernel changes.
# refresh intervals per pruning stage for the mask-caching measurement: the pages' three-stage
# presets (InfiniteHiP section 3.4, default 16/8/4 and "flash" 96/24/8) with the fourth,
# finest stage refreshed together with the third
CACHE_PRESETS = {"default": (16, 8, 4, 4), "flash": (96, 24, 8, 8)}
NCU_TRAFFIC = {
    ("hip_stage_score_s0", "decode_gqa_T1048576"): 201637120 + 3022080,
    ("prefill_attention_tc", "prefill_vs_S131072"): 3470680960 + 1056529664,
}


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=10)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle leg")
    p.add_argument("--small", action="store_true",
                   help="small shapes (context 131072 decode, S=16384 prefill) for a quick check")
    return p.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi sampled every 200 ms while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for name, val in zip(names, parts[5:9]):
                    if val.lower() == "active":
                        reasons.add(name)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ workloads

def workloads(small: bool):
    import synth
    if small:
        dec = synth.decode_case("decode_gqa_T131072", B=1, T=131072, T_q=1, H_q=32, H_kv=8,
                                D=128, dtype="bf16", chunk=(256, 64, 16, 4),
                                keep=(32768, 16384, 8192, 4096), n_sink=128, n_stream=1024,
                                seed=1, plant="uniform", n_plant=64)
        pre = synth.prefill_case("prefill_vs_S16384", S=16384, H_q=32, H_kv=8, D=128, seed=4)
    else:
        dec = synth.decode_1m()
        pre = synth.prefill_128k()
    return dec, pre


def to_dev(a, torch, dev, dtype="bf16"):
    if dtype == "f32":
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev)
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)


def decode_configs():
    """The other decode workloads, each measured on its own (tiny fp32; 128K GQA;
    batch 16 at 32K, which takes the split-K path and its merge across the batch)."""
    import synth
    return [synth.decode_tiny(), synth.decode_128k(), synth.decode_batch16()]


# ------------------------------------------------------------------ oracle leg

def oracle_decode_step(dec):
    """The oracle's full decode step, every batch row (selection + attention); seconds."""
    from oracle import hip
    from oracle.numerics import to_f64
    t0 = time.perf_counter()
    for b in range(dec.B):
        q64 = to_f64(dec.q[b], dec.dtype)
        T = int(dec.kv_len[b])
        _, I = hip.hip_select(q64, dec.k[b], dec.dtype, T, dec.chunk, dec.keep, dec.n_sink,
                              dec.n_stream, dec.G)
        A = hip.attended_set(T, dec.n_sink, dec.n_stream, I)
        hip.decode_attention(q64, dec.k[b], dec.v[b], dec.dtype, A, dec.scale, dec.G)
    return time.perf_counter() - t0


PREFILL_SAMPLE_BUDGET_S = 30.0


def oracle_prefill_sample(pre, budget_s=PREFILL_SAMPLE_BUDGET_S, n_heads=8, blocks_per_head=64):
    """Oracle prefill on a bounded sample, extrapolated to the whole problem; ms.

    Planned sample: the vertical-slash estimate and conversion of `n_heads` heads and,
    for each of them, `blocks_per_head` query blocks spread over the sequence (seeded),
    visited round-robin across the heads; the attention stops once `budget_s` of wall
    time is used, so the blocks actually timed are reported.  The estimate scales by
    heads, the attention by listed tiles (the sampled heads' tile counts stand for the
    average head).
    """
    from oracle import vs
    from oracle.numerics import to_f64
    S, H_q = pre.S, pre.H_q
    t_start = time.perf_counter()
    rows = vs.estimate_rows(S, pre.last_q)
    rng = np.random.default_rng(12345)
    heads = [int(h) for h in rng.permutation(H_q)[:min(n_heads, H_q)]]
    t_est = 0.0
    lists = {}
    for h in heads:
        t0 = time.perf_counter()
        g = h // pre.G
        A = vs.approx_attention(to_f64(pre.q[0, rows, h], "bf16"), rows,
                                to_f64(pre.k[0, :, g], "bf16"), pre.scale)
        v = vs.vertical_sums(A)
        s = vs.slash_sums(A, rows)
        vert = vs.topk_ascending(v, pre.n_vertical)
        sl = vs.topk_ascending(s, pre.n_slash)
        lists[h] = vs.vs_convert(vert, sl, S)
        t_est += time.perf_counter() - t0
    nq = len(lists[heads[0]][0])
    tiles = {h: [len(lists[h][0][m]) + -(-len(lists[h][1][m]) // 64) for m in range(nq)]
             for h in heads}
    # seeded spread of query blocks per head: one per stratum of the sequence
    per = min(blocks_per_head, nq)
    edges = np.linspace(0, nq, per + 1)
    plan = {h: [int(rng.integers(int(edges[i]), max(int(edges[i]) + 1, int(edges[i + 1]))))
                for i in rng.permutation(per)] for h in heads}
    order = [(h, plan[h][i]) for i in range(per) for h in heads]
    t_att, done, sample_tiles = 0.0, 0, 0
    for h, m in order:
        if time.perf_counter() - t_start > budget_s and done > 0:
            break
        blk, col = lists[h]
        t0 = time.perf_counter()
        vs.prefill_block_attention(pre.q[0], pre.k[0], pre.v[0], h, pre.G, m, blk[m], col[m],
                                   S, pre.scale)
        t_att += time.perf_counter() - t0
        done += 1
        sample_tiles += tiles[h][m]
    total_tiles = sum(sum(t) for t in tiles.values()) * H_q / len(heads)
    total_ms = 1e3 * (t_est * H_q / len(heads) + t_att * total_tiles / max(1, sample_tiles))
    desc = (f"estimate+convert of {len(heads)}/{H_q} heads (extrapolated x{H_q / len(heads):g}); "
            f"attention of {done} of the {len(order)} planned (head, query block) pairs "
            f"({blocks_per_head} spread blocks per sampled head, stopped at a {budget_s:g} s wall "
            f"cap), {sample_tiles} of {total_tiles:.0f} tiles, extrapolated by tile count")
    return total_ms, desc


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_model():
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True).stdout
        for line in out.splitlines():
            if line.startswith("Model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def cpu_baseline(dec, pre, configs=()):
    dec_s = oracle_decode_step(dec)
    pre_ms, pre_desc = oracle_prefill_sample(pre)
    per_cfg = {c.name: oracle_decode_step(c) for c in configs}
    return {
        "value": dec_s * 1e6, "unit": "us/step", "cores": host_cores(), "kind": "oracle",
        "cpu": cpu_model(),
        "sample": (f"decode: one full step of {dec.name} (selection + attention, every batch "
                   f"row); the other decode workloads one full step each; prefill: {pre_desc}"),
        "decode_configs_s": per_cfg,
        "prefill_ms_extrapolated": pre_ms,
    }


def max_over_ranks(values, world, device):
    """The per-rank times reduced to their maximum over all ranks (every rank gets it);
    one rank returns them unchanged.  The replicas exchange nothing else."""
    if world <= 1:
        return list(values)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x) for x in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def bench_config(dec, pre, world):
    """The `config` object of the printed line, the same for both arms."""
    return {
        "workload": f"{dec.name} + {pre.name}",
        "decode": {"B": dec.B, "T": dec.T_max, "H_q": dec.H_q, "H_kv": dec.H_kv, "D": dec.D,
                   "chunk": list(dec.chunk), "keep": list(dec.keep), "n_sink": dec.n_sink,
                   "n_stream": dec.n_stream, "selection": "full re-selection every step"},
        "prefill": {"S": pre.S, "H_q": pre.H_q, "H_kv": pre.H_kv, "D": pre.D,
                    "last_q": pre.last_q, "n_vertical": pre.n_vertical, "n_slash": pre.n_slash},
        "l2": ("flushed before each timed decode step and prefill: a 512 MiB write, then a read "
               "of another 512 MiB buffer (leaves L2 clean; the write-only flush is timed beside)"),
        "parallelism": "replicas" if world > 1 else "single GPU",
        "decode_timing": ("the faster of a CUDA-graph replay and eager launches of hip_select + "
                          "sparse_attn_decode, both timed in every step (both under decode)"),
    }


def run_reference(args, rank):
    """The oracle as it stands on the host cores (rank 0 only)."""
    if rank != 0:
        return
    dec, pre = workloads(args.small)
    for _ in range(args.warmup):
        oracle_decode_step(dec)
    times, pre_ms = [], []
    for _ in range(args.steps):
        times.append(oracle_decode_step(dec) * 1e6)
    pre_ms_val, pre_desc = oracle_prefill_sample(pre)
    v = statistics.mean(times)
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "us/step",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        # the timed steps are the decode steps; the prefill is a bounded sample whose
        # extrapolation to the full problem is reported on its own, not added here
        "ms_per_step": v / 1e3, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": bench_config(dec, pre, 1),
        "arm": f"fp64 oracle on {host_cores()} host cores ({cpu_model()})",
        "prefill": {"ms_extrapolated": pre_ms_val, "sample": pre_desc},
        "cpu_baseline": {"value": v, "unit": "us/step", "cores": host_cores(), "kind": "oracle",
                         "cpu": cpu_model(),
                         "sample": (f"decode: {args.steps} full steps of {dec.name} (every batch "
                                    f"row); prefill: {pre_desc}")},
        "e2e": {"value": v, "unit": "us/step", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ decode workloads

def decode_work(dsa, accounting, torch, case, q, kk, kv_len, cfg, elem):
    """Algorithmic work of one decode step over every batch row, from one debug run of
    the same inputs: per-stage bytes (tournament rows + index list + scores + query),
    tournament rows, chunk counts, attention bytes and attended keys.  `elem` is the
    key / value element size (the query keeps its own storage type)."""
    q_elem = 4 if case.dtype == "f32" else 2
    _, cnt2, dbg = dsa.hip_select(q, kk, kv_len, cfg, debug=True)
    torch.cuda.synchronize()
    n = len(case.chunk)
    s_bytes, s_rows, s_chunks = [0] * n, [0] * n, [0] * n
    a_bytes, n_att_total = 0, 0
    qbytes = case.T_q * case.H_q * case.D * q_elem
    for b in range(case.B):
        T = int(case.kv_len[b])
        prev = np.arange(case.n_sink, max(case.n_sink, T - case.n_stream))
        for i, L in enumerate(case.chunk):
            nc = -(-len(prev) // L)
            if nc:
                chunks = [prev[j * L:(j + 1) * L] for j in range(nc)]
                lens = np.array([len(c) for c in chunks], np.int64)
                reps = dbg["rep"][i][b, :, :nc].cpu().numpy().astype(np.int64)
                rows = accounting.stage_rows(reps, None, chunks, lens, case.G)
            else:
                rows = 0
            s_rows[i] += rows
            s_chunks[i] += nc
            idx_bytes = 0 if i == 0 else 4 * len(prev)
            s_bytes[i] += rows * case.D * elem + idx_bytes + 4 * nc + qbytes
            cnt = int(dbg["stage_cnt"][i][b])
            prev = dbg["stage_idx"][i][b, :cnt].cpu().numpy()
        n_att = min(case.n_sink, T) + int(cnt2[b]) + (T - max(case.n_sink, T - case.n_stream))
        n_att_total += n_att
        a_bytes += n_att * case.H_kv * case.D * elem * 2 + 2 * qbytes
    return s_bytes, s_rows, s_chunks, a_bytes, n_att_total


def measure_decode_config(dsa, accounting, torch, dev, case, steps, flush, hbm):
    """One decode workload on its own: CUDA-graph replay of hip_select +
    sparse_attn_decode (L2 flushed before each step), the per-kernel event durations of
    the same steps, and the step's algorithmic bytes against the HBM peak."""
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    q = to_dev(case.q, torch, dev, case.dtype)
    k = to_dev(case.k, torch, dev, case.dtype)
    v = to_dev(case.v, torch, dev, case.dtype)
    kv_len = torch.from_numpy(case.kv_len).to(dev)
    cfg = dsa.HipConfig(case.chunk, case.keep, case.n_sink, case.n_stream)
    sel_idx = torch.empty(case.B, case.keep[-1], dtype=torch.int32, device=dev)
    sel_cnt = torch.empty(case.B, dtype=torch.int32, device=dev)
    ws_sel = torch.empty(dsa.hip_select_workspace_bytes(q, k, cfg), dtype=torch.uint8, device=dev)
    ws_dec = torch.empty(max(1, dsa.sparse_attn_decode_workspace_bytes(
        q, k, case.keep[-1], case.n_sink, case.n_stream)), dtype=torch.uint8, device=dev)
    out = torch.empty_like(q)
    lse = torch.empty(case.B, case.T_q, case.H_q, dtype=torch.float32, device=dev)

    def step():
        dsa.hip_select(q, k, kv_len, cfg, out=(sel_idx, sel_cnt), workspace=ws_sel)
        dsa.sparse_attn_decode(q, k, v, kv_len, sel_idx, sel_cnt, n_sink=case.n_sink,
                               n_stream=case.n_stream, out=out, lse=lse, workspace=ws_dec)

    side = torch.cuda.Stream(device=dev)
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(3):
            step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    times = []
    for _ in range(steps):
        flush()
        e0, e1 = ev(), ev()
        e0.record()
        graph.replay()
        e1.record()
        times.append((e0, e1))
    torch.cuda.synchronize()
    us = 1e3 * statistics.mean(a.elapsed_time(b) for a, b in times)
    dsa.profile_enable(True)
    for _ in range(steps):
        flush()
        step()
    torch.cuda.synchronize()
    dsa.profile_enable(False)
    kern = {name: {"launches": n, "avg_us": 1e3 * t / n} for name, (n, t) in dsa.profile_collect().items()}
    elem = 4 if case.dtype == "f32" else 2
    sb, sr, sc, ab, att = decode_work(dsa, accounting, torch, case, q, k, kv_len, cfg, elem)
    kb = {f"hip_stage_score_s{i}": b_ for i, b_ in enumerate(sb)}
    for name in ("decode_splitk", "decode_cluster_mma"):
        kb[name] = ab
    for name, b_ in kb.items():
        if name in kern:
            kern[name]["algorithmic_bytes"] = b_
            kern[name]["achieved_GBps"] = b_ / (kern[name]["avg_us"] * 1e-6) / 1e9
            kern[name]["hbm_frac"] = kern[name]["achieved_GBps"] / hbm
    step_bytes = sum(r * case.D * elem for r in sr) + ab
    dom = max(kern, key=lambda n_: kern[n_]["avg_us"] * kern[n_]["launches"])
    del q, k, v, graph
    torch.cuda.empty_cache()
    return {
        "us_per_step_graph": us,
        "algorithmic_bytes_per_step": step_bytes,
        "step_hbm_frac": step_bytes / (us * 1e-6) / 1e9 / hbm,
        "dominant_kernel": dom,
        "dominant_kernel_hbm_frac": kern[dom].get("hbm_frac"),
        "tournament_rows_per_stage": sr,
        "chunks_per_stage": sc,
        "attended_keys": att,
        "attention_path": "split-K + merge" if "decode_splitk" in kern else "cluster (DSMEM merge)",
        "shape": {"B": case.B, "T": case.T_max, "T_q": case.T_q, "H_q": case.H_q,
                  "H_kv": case.H_kv, "D": case.D, "dtype": case.dtype, "chunk": list(case.chunk),
                  "keep": list(case.keep), "n_sink": case.n_sink, "n_stream": case.n_stream},
        "kernels": kern,
    }


# ------------------------------------------------------------------ GPU leg

def main():
    args = parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank)
        return

    import torch
    import dynamic_sparse_attention_gb300 as dsa
    from dynamic_sparse_attention_gb300 import accounting
    import torch.distributed as dist

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    dsa.load()
    peaks, peaks_src = load_peaks()

    dec, pre = workloads(args.small)
    # ---------------- decode buffers (resident)
    q = to_dev(dec.q, torch, dev)
    k = to_dev(dec.k, torch, dev)
    v = to_dev(dec.v, torch, dev)
    kv_len = torch.from_numpy(dec.kv_len).to(dev)
    cfg = dsa.HipConfig(dec.chunk, dec.keep, dec.n_sink, dec.n_stream)
    sel_idx = torch.empty(dec.B, dec.keep[-1], dtype=torch.int32, device=dev)
    sel_cnt = torch.empty(dec.B, dtype=torch.int32, device=dev)
    ws_sel = torch.empty(dsa.hip_select_workspace_bytes(q, k, cfg), dtype=torch.uint8, device=dev)
    ws_dec = torch.empty(max(1, dsa.sparse_attn_decode_workspace_bytes(q, k, dec.keep[-1], dec.n_sink,
                                                                       dec.n_stream)),
                         dtype=torch.uint8, device=dev)
    out = torch.empty_like(q)
    lse = torch.empty(dec.B, dec.T_q, dec.H_q, dtype=torch.float32, device=dev)

    def decode_step():
        dsa.hip_select(q, k, kv_len, cfg, out=(sel_idx, sel_cnt), workspace=ws_sel)
        dsa.sparse_attn_decode(q, k, v, kv_len, sel_idx, sel_cnt, n_sink=dec.n_sink,
                               n_stream=dec.n_stream, out=out, lse=lse, workspace=ws_dec)

    # ---------------- prefill buffers (resident)
    pq, pk, pv = to_dev(pre.q, torch, dev), to_dev(pre.k, torch, dev), to_dev(pre.v, torch, dev)
    nq = (pre.S + 63) // 64
    idx = {
        "vertical": torch.empty(1, pre.H_q, pre.n_vertical, dtype=torch.int32, device=dev),
        "slash": torch.empty(1, pre.H_q, pre.n_slash, dtype=torch.int32, device=dev),
        "blk_cnt": torch.empty(1, pre.H_q, nq, dtype=torch.int32, device=dev),
        "blk_idx": torch.empty(1, pre.H_q, nq, nq, dtype=torch.int32, device=dev),
        "col_cnt": torch.empty(1, pre.H_q, nq, dtype=torch.int32, device=dev),
        "col_idx": torch.empty(1, pre.H_q, nq, pre.n_vertical, dtype=torch.int32, device=dev),
    }
    ws_vs = torch.empty(dsa.vs_index_build_workspace_bytes(pq, pk, pre.last_q, pre.n_vertical,
                                                           pre.n_slash), dtype=torch.uint8, device=dev)
    pout = torch.empty_like(pq)
    plse = torch.empty(1, pre.H_q, pre.S, dtype=torch.float32, device=dev)

    def prefill_index():
        dsa.vs_index_build(pq, pk, last_q=pre.last_q, n_vertical=pre.n_vertical,
                           n_slash=pre.n_slash, out=idx, workspace=ws_vs)

    def prefill_attn():
        dsa.sparse_attn_prefill(pq, pk, pv, idx["blk_cnt"], idx["blk_idx"], idx["col_cnt"],
                                idx["col_idx"], out=pout, lse=plse)

    # L2 (129 MB) flush between timed steps: write a 512 MiB buffer, then read a second,
    # never-written 512 MiB buffer.  The write evicts the step's data; the read evicts
    # the write's dirty lines, so that their write-back to HBM (about 129 MB) is not
    # charged to the next timed step.  flush_write_only() is the write alone, timed
    # beside it for comparison.
    flush_buf = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    flush_clean = torch.ones(128 << 20, dtype=torch.int32, device=dev)
    flush_sink = torch.empty((), dtype=torch.int64, device=dev)

    def flush():
        flush_buf.fill_(1)
        torch.sum(flush_clean, dim=0, dtype=torch.int64, out=flush_sink)

    def flush_write_only():
        flush_buf.fill_(1)

    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731

    # ---------------- warm-up (eager), then capture the decode step
    for _ in range(max(3, args.warmup)):
        decode_step()
        prefill_index()
        prefill_attn()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream(device=dev)
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        decode_step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    with torch.cuda.graph(graph):
        decode_step()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()

    # ---------------- timed region
    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    dec_ms, eager, idx_ms, att_ms = [], [], [], []
    barrier()
    with ClockSampler(local_rank) as clocks:
        for _ in range(args.steps):
            # the decode step twice, as a CUDA-graph replay and as eager launches (the
            # plain API calls); the faster is the headline, both are reported
            flush()
            e0, e1 = ev(), ev()
            e0.record()
            graph.replay()
            e1.record()
            flush()
            e5, e6 = ev(), ev()
            e5.record()
            decode_step()
            e6.record()
            eager.append((e5, e6))
            flush()
            e2, e3, e4 = ev(), ev(), ev()
            e2.record()
            prefill_index()
            e3.record()
            prefill_attn()
            e4.record()
            dec_ms.append((e0, e1))
            idx_ms.append((e2, e3))
            att_ms.append((e3, e4))
        barrier()
    dec_ms = [a.elapsed_time(b) for a, b in dec_ms]
    idx_ms = [a.elapsed_time(b) for a, b in idx_ms]
    att_ms = [a.elapsed_time(b) for a, b in att_ms]
    clock_info = clocks.summary()

    # the same graph after a write-only flush (its dirty lines written back inside the step)
    wflush = []
    for _ in range(args.steps):
        flush_write_only()
        e0, e1 = ev(), ev()
        e0.record()
        graph.replay()
        e1.record()
        wflush.append((e0, e1))
    torch.cuda.synchronize()
    wflush = [a.elapsed_time(b) for a, b in wflush]

    eager = [a.elapsed_time(b) for a, b in eager]

    # ---------------- mask caching: amortized decode step over one refresh period
    c_idx, c_cnt = torch.empty_like(sel_idx), torch.empty_like(sel_cnt)
    ws_cache = torch.empty_like(ws_sel)

    def cached_step(mask):
        dsa.hip_select_cached(q, k, kv_len, cfg, mask, out=(c_idx, c_cnt), workspace=ws_cache)
        dsa.sparse_attn_decode(q, k, v, kv_len, c_idx, c_cnt, n_sink=dec.n_sink,
                               n_stream=dec.n_stream, out=out, lse=lse, workspace=ws_dec)

    cached = {}
    cache_graphs = {}
    for name, n_refresh in CACHE_PRESETS.items():
        if len(n_refresh) != len(dec.chunk):
            continue
        period = n_refresh[0]
        masks = [dsa.refresh_mask(s, n_refresh) for s in range(period)]
        for m in sorted(set(masks)):
            if m in cache_graphs:
                continue
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):
                cached_step(m)
            torch.cuda.current_stream().wait_stream(side)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                cached_step(m)
            cache_graphs[m] = g
        by_mask = {}
        reps = max(1, 32 // period)
        for _ in range(reps):
            for m in masks:
                flush()
                e0, e1 = ev(), ev()
                e0.record()
                cache_graphs[m].replay()
                e1.record()
                by_mask.setdefault(m, []).append((e0, e1))
        torch.cuda.synchronize()
        us = {m: [1e3 * a.elapsed_time(b) for a, b in v_] for m, v_ in by_mask.items()}
        total = sum(sum(v_) for v_ in us.values())
        cached[name] = {
            "n_refresh": list(n_refresh), "period_steps": period, "periods_timed": reps,
            "us_per_step_amortized": total / (reps * period),
            "us_by_refreshed_stages": {",".join(str(i) for i in range(len(n_refresh)) if m >> i & 1)
                                       or "none": statistics.mean(v_) for m, v_ in us.items()},
        }

    # ---------------- FP8 E4M3 keys and values: the same step over the cache rounded to
    # E4M3 on the device (torch's float8 conversion: nearest, ties to even)
    k8 = k.to(torch.float8_e4m3fn).view(torch.uint8)
    v8 = v.to(torch.float8_e4m3fn).view(torch.uint8)
    s8_idx, s8_cnt = torch.empty_like(sel_idx), torch.empty_like(sel_cnt)
    ws_sel8 = torch.empty(dsa.hip_select_workspace_bytes(q, k8, cfg), dtype=torch.uint8, device=dev)

    def decode_step_fp8():
        dsa.hip_select(q, k8, kv_len, cfg, out=(s8_idx, s8_cnt), workspace=ws_sel8)
        dsa.sparse_attn_decode(q, k8, v8, kv_len, s8_idx, s8_cnt, n_sink=dec.n_sink,
                               n_stream=dec.n_stream, out=out, lse=lse, workspace=ws_dec)

    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(3):
            decode_step_fp8()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph8 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph8):
        decode_step_fp8()
    fp8_ms = []
    for _ in range(max(3, args.steps)):
        flush()
        e0, e1 = ev(), ev()
        e0.record()
        graph8.replay()
        e1.record()
        fp8_ms.append((e0, e1))
    torch.cuda.synchronize()
    fp8_us = 1e3 * statistics.mean(a.elapsed_time(b_) for a, b_ in fp8_ms)
    dsa.profile_enable(True)
    for _ in range(max(3, args.steps)):
        flush()
        decode_step_fp8()
    torch.cuda.synchronize()
    dsa.profile_enable(False)
    k8stats = dsa.profile_collect()

    # ---------------- per-kernel durations (CUDA events on the launch stream)
    dsa.profile_enable(True)
    for _ in range(args.steps):
        flush()
        decode_step()
        flush()
        prefill_index()
        prefill_attn()
    torch.cuda.synchronize()
    dsa.profile_enable(False)
    kstats = dsa.profile_collect()
    per_step_launches = sum(n for n, _ in kstats.values()) / args.steps
    # each timed step runs the decode twice (graph replay and eager launches)
    per_step_launches += sum(n for name, (n, _) in kstats.items()
                             if name.startswith(("hip_", "decode_"))) / args.steps
    kern = {name: {"launches": n, "avg_us": 1e3 * t / n} for name, (n, t) in kstats.items()}

    # ---------------- algorithmic work (from one debug run of the same inputs)
    elem = 2
    T = int(dec.kv_len[0])
    stage_bytes, stage_rows, stage_chunks, attn_bytes, attended = decode_work(
        dsa, accounting, torch, dec, q, k, kv_len, cfg, elem)
    step_bytes = sum(r * dec.D * elem for r in stage_rows) + attn_bytes
    dec_kernel_bytes = {f"hip_stage_score_s{i}": b for i, b in enumerate(stage_bytes)}
    for name in ("decode_splitk", "decode_cluster_mma"):   # whichever attention kernel ran
        dec_kernel_bytes[name] = attn_bytes
    for name, b in dec_kernel_bytes.items():
        if name in kern:
            kern[name]["algorithmic_bytes"] = b
            kern[name]["achieved_GBps"] = b / (kern[name]["avg_us"] * 1e-6) / 1e9

    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    sb8, sr8, _, ab8, att8 = decode_work(dsa, accounting, torch, dec, q, k8, kv_len, cfg, 1)
    k8b = {f"hip_stage_score_s{i}": b_ for i, b_ in enumerate(sb8)}
    k8b["decode_cluster_mma_fp8"] = ab8
    fp8_kern = {}
    for name, (n_, t_) in k8stats.items():
        e_ = {"launches": n_, "avg_us": 1e3 * t_ / n_}
        if name in k8b:
            e_["algorithmic_bytes"] = k8b[name]
            e_["achieved_GBps"] = k8b[name] / (e_["avg_us"] * 1e-6) / 1e9
            e_["hbm_frac"] = e_["achieved_GBps"] / hbm
        fp8_kern[name] = e_
    step8 = sum(r * dec.D for r in sr8) + ab8
    fp8_line = {"us_per_step_graph": fp8_us, "algorithmic_bytes_per_step": step8,
                "step_hbm_frac": step8 / (fp8_us * 1e-6) / 1e9 / hbm, "attended_keys": att8,
                "tournament_rows_per_stage": sr8, "kernels": fp8_kern,
                "kv": "E4M3 codes rounded on the device from the bf16 cache (torch float8_e4m3fn)"}
    dec_names = [n for n in kern if n.startswith("hip_") or n.startswith("decode_")]
    dom = max(dec_names, key=lambda n: kern[n]["avg_us"] * kern[n]["launches"])
    dom_bytes = dec_kernel_bytes.get(dom)
    achieved = dom_bytes / (kern[dom]["avg_us"] * 1e-6) / 1e9 if dom_bytes else None
    roofline = {"kernel": dom, "bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                "frac": achieved / hbm if achieved else None,
                "traffic": NCU_TRAFFIC.get((dom, dec.name)),
                "peak_source": f"{peaks_src} hbm_gbs",
                "nominal_peak": NOMINAL_HBM_GBS,
                "frac_nominal": achieved / NOMINAL_HBM_GBS if achieved else None,
                "algorithmic_bytes_per_launch": dom_bytes}

    # prefill tiles and FLOPs
    blk_cnt = idx["blk_cnt"].cpu().numpy()
    col_cnt = idx["col_cnt"].cpu().numpy()
    flops = accounting.prefill_tile_flops(blk_cnt, col_cnt, pre.D)
    useful_flops = accounting.prefill_useful_flops(blk_cnt, idx["blk_idx"].cpu().numpy(), col_cnt,
                                                   idx["col_idx"].cpu().numpy(), pre.S, pre.D)
    tiles = int(blk_cnt.sum() + np.ceil(col_cnt / 64.0).sum())
    dense_tiles = accounting.causal_dense_tiles(pre.S) * pre.H_q
    att_name = [n for n in kern if n.startswith("prefill_attention")][0]
    att_us = kern[att_name]["avg_us"]
    # each prefill launch is one kernel of about a hundred milliseconds timed on its own:
    # the burst figure is its denominator (the sustained one is printed beside it)
    tc_peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    tc_sus = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    tflops = flops / (att_us * 1e-6) / 1e12
    kern[att_name]["algorithmic_flops"] = flops
    kern[att_name]["achieved_TFLOPs"] = tflops
    vs_bytes = accounting.vs_index_bytes(1, pre.S, pre.H_q, pre.H_kv, pre.D, pre.n_vertical)
    vs_us = sum(kern[n]["avg_us"] for n in kern if n.startswith("vs_"))
    roofline_prefill = {"kernel": att_name, "bound": "tensor", "achieved": tflops, "peak": tc_peak,
                        "unit": "TFLOP/s", "frac": tflops / tc_peak,
                        "traffic": NCU_TRAFFIC.get((att_name, pre.name)),
                        "peak_source": f"{peaks_src} bf16_tflops (burst: one kernel timed on its own)",
                        "frac_sustained": tflops / tc_sus,
                        "nominal_peak": NOMINAL_BF16_TFLOPS,
                        "frac_nominal": tflops / NOMINAL_BF16_TFLOPS,
                        "algorithmic_flops_per_launch": flops}

    # ---------------- other MInference head patterns on the same prefill kernel
    def time_pattern(build, steps):
        lists = build()
        torch.cuda.synchronize()
        for _ in range(2):
            build()
            dsa.sparse_attn_prefill(pq, pk, pv, lists["blk_cnt"], lists["blk_idx"],
                                    lists["col_cnt"], lists.get("col_idx"), out=pout, lse=plse)
        ib, at = [], []
        for _ in range(steps):
            flush()
            e0, e1, e2 = ev(), ev(), ev()
            e0.record()
            build()
            e1.record()
            dsa.sparse_attn_prefill(pq, pk, pv, lists["blk_cnt"], lists["blk_idx"],
                                    lists["col_cnt"], lists.get("col_idx"), out=pout, lse=plse)
            e2.record()
            ib.append((e0, e1))
            at.append((e1, e2))
        torch.cuda.synchronize()
        ib = statistics.mean(a.elapsed_time(b) for a, b in ib)
        at = statistics.mean(a.elapsed_time(b) for a, b in at)
        bc = lists["blk_cnt"].cpu().numpy()
        cc = lists["col_cnt"].cpu().numpy()
        fl = accounting.prefill_tile_flops(bc, cc, pre.D)
        return {"index_ms": ib, "attention_ms": at, "tiles": int(bc.sum() + np.ceil(cc / 64.0).sum()),
                "tile_density_vs_causal_dense": float(bc.sum()) / dense_tiles,
                "tile_flops": fl, "attention_TFLOPs": fl / (at * 1e-3) / 1e12,
                "attention_tc_frac": fl / (at * 1e-3) / 1e12 / tc_peak}

    n_qb = (pre.S + 63) // 64
    pat_steps = max(2, min(args.steps, 4))
    ash = {"blk_cnt": torch.empty(1, pre.H_q, n_qb, dtype=torch.int32, device=dev),
           "blk_idx": torch.empty(1, pre.H_q, n_qb, 80, dtype=torch.int32, device=dev),
           "col_cnt": torch.empty(1, pre.H_q, n_qb, dtype=torch.int32, device=dev)}
    bsl = {"blk_cnt": torch.empty(1, pre.H_q, n_qb, dtype=torch.int32, device=dev),
           "blk_idx": torch.empty(1, pre.H_q, n_qb, 100, dtype=torch.int32, device=dev),
           "col_cnt": torch.empty(1, pre.H_q, n_qb, dtype=torch.int32, device=dev)}
    ws_bs = torch.empty(dsa.block_sparse_index_build_workspace_bytes(pq, pk), dtype=torch.uint8,
                        device=dev)
    patterns_line = {
        "a_shape": dict(time_pattern(lambda: dsa.ashape_index_build(
            pq, pk, n_global=1024, n_local=4096, out=ash), pat_steps), n_global=1024, n_local=4096),
        "block_sparse": dict(time_pattern(lambda: dsa.block_sparse_index_build(
            pq, pk, k_b=100, out=bsl, workspace=ws_bs), pat_steps), k_b=100),
    }
    mix_pats = [("vertical_slash", "a_shape", "block_sparse")[h % 3] for h in range(pre.H_q)]
    mix_kw = dict(head_pattern=mix_pats, last_q=pre.last_q, n_vertical=pre.n_vertical,
                  n_slash=pre.n_slash, n_global=1024, n_local=4096, k_b=100)
    mix_out = {key: idx[key] for key in ("blk_cnt", "blk_idx", "col_cnt", "col_idx")}
    ws_mix = torch.empty(max(1, dsa.mixed_index_build_workspace_bytes(pq, pk, **mix_kw)),
                         dtype=torch.uint8, device=dev)
    patterns_line["mixed"] = dict(time_pattern(lambda: dsa.mixed_index_build(
        pq, pk, out=mix_out, workspace=ws_mix, **mix_kw), pat_steps),
        heads="h mod 3: vertical-slash, A-shape, Block-Sparse")
    # InfiniteHiP sparse prefill on the same inputs: per-64-row query block pruning with the
    # pages' stage table (chunks 256 / 32 / 8, keep 32768 / 8192 / 2048, sink 256,
    # window 1024), then the prefill kernel over sink + selection + window
    hcfg = dsa.HipConfig((256, 32, 8), (32768, 8192, 2048), 256, 1024)
    n_rows = (pre.S + 63) // 64
    hsel = (torch.empty(n_rows, 2048, dtype=torch.int32, device=dev),
            torch.empty(n_rows, dtype=torch.int32, device=dev))
    ws_h = torch.empty(dsa.hip_prefill_select_workspace_bytes(pq, pk, hcfg), dtype=torch.uint8,
                       device=dev)
    hl = {"blk_cnt": torch.empty(1, pre.H_q, n_rows, dtype=torch.int32, device=dev),
          "blk_idx": torch.empty(1, pre.H_q, n_rows, 22, dtype=torch.int32, device=dev),
          "col_cnt": torch.empty(1, pre.H_q, n_rows, dtype=torch.int32, device=dev),
          "col_idx": torch.empty(1, pre.H_q, n_rows, 2048 + 126, dtype=torch.int32, device=dev)}

    def hip_prefill_index():
        dsa.hip_prefill_select(pq, pk, hcfg, out=hsel, workspace=ws_h)
        dsa.hip_prefill_lists(pq, pk, hcfg, hsel[0], hsel[1], out=hl)
        return hl

    patterns_line["infinitehip"] = dict(time_pattern(hip_prefill_index, pat_steps),
                                        chunk=[256, 32, 8], keep=[32768, 8192, 2048],
                                        n_sink=256, n_stream=1024)
    dsa.profile_enable(True)
    for _ in range(pat_steps):
        flush()
        hip_prefill_index()
    torch.cuda.synchronize()
    dsa.profile_enable(False)
    for name, (n_, t_) in dsa.profile_collect().items():
        patterns_line["infinitehip"][f"{name}_ms"] = t_ / pat_steps
    pool_bytes = accounting.block_sparse_pool_bytes(1, pre.S, pre.H_q, pre.H_kv, pre.D)
    dsa.profile_enable(True)
    for _ in range(pat_steps):
        flush()
        dsa.block_sparse_index_build(pq, pk, k_b=100, out=bsl, workspace=ws_bs)
    torch.cuda.synchronize()
    dsa.profile_enable(False)
    for name, (n, t) in dsa.profile_collect().items():
        patterns_line["block_sparse"][f"{name}_us"] = 1e3 * t / n
        if name == "bs_pool":
            patterns_line["block_sparse"]["bs_pool_GBps"] = pool_bytes / (t / n * 1e-3) / 1e9
            patterns_line["block_sparse"]["bs_pool_hbm_frac"] = pool_bytes / (t / n * 1e-3) / 1e9 / hbm

    # ---------------- end to end through the public API with host buffers
    h_q = torch.empty(q.shape, dtype=q.dtype, pin_memory=True)
    h_q.copy_(q)
    h_kn = torch.empty(k[:, T - 1].shape, dtype=k.dtype, pin_memory=True)
    h_vn = torch.empty_like(h_kn, pin_memory=True)
    h_kn.copy_(k[:, T - 1])
    h_vn.copy_(v[:, T - 1])
    h_out = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    e2e = []
    for _ in range(args.steps):
        flush()
        e0, e1 = ev(), ev()
        e0.record()
        q.copy_(h_q, non_blocking=True)
        k[:, T - 1].copy_(h_kn, non_blocking=True)   # the newest token's key / value row
        v[:, T - 1].copy_(h_vn, non_blocking=True)
        decode_step()
        h_out.copy_(out, non_blocking=True)
        e1.record()
        e2e.append((e0, e1))
    torch.cuda.synchronize()
    e2e = [a.elapsed_time(b) for a, b in e2e]
    h2d = h_q.numel() * 2 + 2 * h_kn.numel() * 2
    d2h = h_out.numel() * 2
    hp = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (pq, pk, pv)]
    for h_, d_ in zip(hp, (pq, pk, pv)):
        h_.copy_(d_)
    h_pout = torch.empty(pout.shape, dtype=pout.dtype, pin_memory=True)
    pe2e = []
    for _ in range(min(args.steps, 3)):
        flush()
        e0, e1 = ev(), ev()
        e0.record()
        for h_, d_ in zip(hp, (pq, pk, pv)):
            d_.copy_(h_, non_blocking=True)
        prefill_index()
        prefill_attn()
        h_pout.copy_(pout, non_blocking=True)
        e1.record()
        pe2e.append((e0, e1))
    torch.cuda.synchronize()
    pe2e = [a.elapsed_time(b) for a, b in pe2e]

    # ---------------- the other decode workloads, each on its own
    del graph8, k8, v8
    torch.cuda.empty_cache()
    configs = [] if args.small else decode_configs()
    config_lines = {c.name: measure_decode_config(dsa, accounting, torch, dev, c, args.steps, flush, hbm)
                    for c in configs}

    # ---------------- max over ranks
    dec_graph_us = 1e3 * statistics.mean(dec_ms)
    dec_eager_us = 1e3 * statistics.mean(eager)
    pre_ms = statistics.mean(idx_ms) + statistics.mean(att_ms)
    dec_graph_us, dec_eager_us, pre_ms = max_over_ranks([dec_graph_us, dec_eager_us, pre_ms], world, dev)
    dec_us = min(dec_graph_us, dec_eager_us)
    if rank != 0:
        dist.destroy_process_group()
        return

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(dec, pre, configs)
        for c in configs:
            config_lines[c.name]["oracle_s_per_step"] = cpu["decode_configs_s"][c.name]

    line = {
        "metric": METRIC,
        "value": dec_us,
        "unit": "us/step",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": dec_us / 1e3 + pre_ms,
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": bench_config(dec, pre, world),
        # the other decode workloads (tiny fp32, 128K GQA, batch 16 at 32K), each its own
        # graph-replayed step with the same accounting
        "decode_configs": config_lines,
        "decode": {
            "us_per_step_graph": dec_graph_us,
            "us_per_step_eager": dec_eager_us,
            "us_per_step_graph_after_write_only_flush": 1e3 * statistics.mean(wflush),
            "algorithmic_bytes_per_step": step_bytes,
            "step_hbm_frac": step_bytes / (dec_us * 1e-6) / 1e9 / hbm,
            "tournament_rows_per_stage": stage_rows,
            "chunks_per_stage": stage_chunks,
            "attended_keys": attended,
        },
        # the same prefill kernel over MInference A-shape (1024 initial + 4096 local tokens),
        # Block-Sparse (k_b = 100), a per-head mix of the three patterns, and InfiniteHiP's
        # per-query-block selection (sink + 2048 selected + 1024 window keys), same inputs
        "prefill_patterns": patterns_line,
        # the same decode step over an FP8 E4M3 copy of the KV cache (bf16 queries)
        "decode_fp8kv": fp8_line,
        # mask caching (InfiniteHiP section 3.4): the same step with stage i recomputed only
        # when step % n_refresh[i] == 0, averaged over whole refresh periods
        "decode_cached": cached,
        "prefill": {
            "ms": pre_ms,
            "vs_index_ms": statistics.mean(idx_ms),
            "attention_ms": statistics.mean(att_ms),
            "tiles": tiles,
            "tile_density_vs_causal_dense": tiles / dense_tiles,
            "tile_flops": flops,
            "vs_index_GBps": vs_bytes / (vs_us * 1e-6) / 1e9,
            "vs_index_hbm_frac": vs_bytes / (vs_us * 1e-6) / 1e9 / hbm,
            # pairs (query row, key) the lists make attended, causal masking subtracted
            "useful_flops": useful_flops,
            "useful_TFLOPs": useful_flops / (att_us * 1e-6) / 1e12,
        },
        # the step's dominant kernel (prefill attention, >99% of a step's GPU time)
        "roofline": roofline_prefill,
        # the decode half's dominant kernel (the headline `value` is decode us/step)
        "roofline_decode": roofline,
        "kernels": kern,
        "gpu_launches": int(round(per_step_launches * args.steps)),
        "e2e": {"value": 1e3 * statistics.mean(e2e), "unit": "us/step",
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "prefill_ms": statistics.mean(pe2e),
                "prefill_h2d_bytes": int(sum(t.numel() * 2 for t in hp)),
                "prefill_d2h_bytes": int(h_pout.numel() * 2)},
        "clocks": clock_info,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
