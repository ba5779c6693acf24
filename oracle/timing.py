"""Times the CPU oracle on a bounded sample of a decode workload (the CPU baseline).

Test infrastructure (see oracle/__init__.py): run only by the benchmark's cpu_baseline
and --impl reference legs.  Inputs come from the seeded generator on the host with the
workload's shapes: each sampled query owns one sequence of N entries, and one "step"
is that query's append (compressor, m = 1) plus the 20-layer decoder schedule.

Usage: python -m oracle.timing --N 131072 --queries 2 [--json]
"""
import argparse
import json
import os
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from fp4_compressed_sparse_02_gb300 import synth  # noqa: E402  (input generator only)
from oracle import compress, formats, schedule  # noqa: E402


def make_query(r, N, cfg):
    d, d_ik, H_i, Hq, W, d_model = (cfg[x] for x in ("d", "d_ik", "H_i", "Hq", "W", "d_model"))
    codes = synth.fp4_codes(r, (N,), d)
    scales = synth.fp4_scales(r, (N,), d)
    K = formats.bf16_value(synth.bf16_normal(r, (N, d_ik)))
    layers = []
    for mode in schedule.decoder_schedule():
        L = dict(mode=mode, q=formats.bf16_value(synth.bf16_normal(r, (Hq, d))),
                 swa_rows=synth.fp8_rows(r, W, d), swa_scale=synth.fp8_row_scales(r, W), swa_start=0, swa_len=W)
        if mode != "reuse":
            L["q_idx"] = formats.bf16_value(synth.bf16_normal(r, (H_i, d_ik)))
            L["w"] = synth.f32_normal(r, (H_i,), 1 / np.sqrt(H_i)).astype(np.float64)
        layers.append(L)
    H = formats.bf16_value(synth.bf16_normal(r, (1, d_model)))
    Wkv = formats.bf16_value(synth.bf16_normal(r, (d_model, d), 1 / np.sqrt(d_model)))
    Wik = formats.bf16_value(synth.bf16_normal(r, (d, d_ik), 1 / np.sqrt(d)))
    cos, sin = synth.rope_tables(N, cfg["d_rope"])
    return dict(codes=codes, scales=scales, K=K, layers=layers, H=H, Wkv=Wkv, Wik=Wik, cos=cos, sin=sin)


def run_query(x, N, cfg):
    """One query-step: append entry N-1 from H, then the 20 decoder layers."""
    app = compress.compress_quant_from_hidden(x["H"], x["Wkv"], None, 1, np.array([N - 1]), x["cos"], x["sin"],
                                              cfg["d_rope"], x["Wik"])
    x["codes"][N - 1] = app["codes"][0]
    x["scales"][N - 1] = app["scales"][0]
    x["K"][N - 1] = formats.bf16_value(app["idx_k"][0])
    return schedule.decode_step(x["layers"], x["K"], x["codes"], x["scales"], cfg["NB"], cfg["P"], cfg["k"],
                                1 / np.sqrt(cfg["d"]))


class LayerSteps:
    """The decode schedule one query-layer at a time, over a small pool of queries: step i runs
    layer i mod 20 of query (i div 20) mod len(pool) (the query's append with its layer 0),
    carrying the layer state (pool, top-k) as the 20-layer step does.  Every 20 steps form
    whole query-steps, so a run of any length times the same mix of layers."""

    def __init__(self, xs, N, cfg):
        self.xs, self.N, self.cfg = xs, N, cfg
        self.i = 0
        self.pool = self.topk = None

    def step(self):
        from oracle import attention, indexer
        nl = len(schedule.decoder_schedule())
        x = self.xs[(self.i // nl) % len(self.xs)]
        li = self.i % nl
        self.i += 1
        cfg, N = self.cfg, self.N
        if li == 0:
            app = compress.compress_quant_from_hidden(x["H"], x["Wkv"], None, 1, np.array([N - 1]), x["cos"],
                                                      x["sin"], cfg["d_rope"], x["Wik"])
            x["codes"][N - 1] = app["codes"][0]
            x["scales"][N - 1] = app["scales"][0]
            x["K"][N - 1] = formats.bf16_value(app["idx_k"][0])
        L = x["layers"][li]
        if L["mode"] == schedule.FULL:
            self.pool, self.topk, _ = indexer.full(L["q_idx"], L["w"], x["K"], cfg["NB"], cfg["P"], cfg["k"])
        elif L["mode"] == schedule.REINDEX:
            self.topk, _ = indexer.reindex(L["q_idx"], L["w"], x["K"], self.pool, cfg["k"])
        else:
            self.topk = indexer.reuse(self.topk)
        return attention.sparse_attention(L["q"], x["codes"], x["scales"], self.topk, L["swa_rows"], L["swa_scale"],
                                          L["swa_start"], L["swa_len"], 1 / np.sqrt(cfg["d"]))


def time_sample(N, queries, cfg, seed=0):
    """Each query is generated, timed through one query-step and dropped, so memory holds
    one sequence at a time; only the query-steps are timed."""
    r = np.random.default_rng(seed)
    dt = 0.0
    for _ in range(queries):
        x = make_query(r, N, cfg)
        t0 = time.perf_counter()
        run_query(x, N, cfg)
        dt += time.perf_counter() - t0
        del x
    layers = len(schedule.decoder_schedule())
    return dict(seconds=dt, query_layers=queries * layers, value=queries * layers / dt)


def _worker(args):
    """One process's share: its own seeded queries, each generated then timed alone."""
    N, queries, cfg, seed = args
    return time_sample(N, queries, cfg, seed)["seconds"]


def time_sample_parallel(N, queries, cfg, procs, seed=0):
    """The same sample spread over `procs` single-threaded processes (spawned, so no state is
    inherited): each process times its own queries, and the rate counts every query-layer
    over the slowest process's timed seconds."""
    import multiprocessing as mp
    per = [queries // procs + (1 if i < queries % procs else 0) for i in range(procs)]
    jobs = [(N, n, cfg, seed * 1000 + i) for i, n in enumerate(per) if n > 0]
    with mp.get_context("spawn").Pool(len(jobs)) as pool:
        secs = pool.map(_worker, jobs)
    layers = len(schedule.decoder_schedule())
    dt = max(secs)
    return dict(seconds=dt, query_layers=queries * layers, value=queries * layers / dt, procs=len(jobs))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--N", type=int, default=131072)
    ap.add_argument("--queries", type=int, default=2)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--config", default="DEC128K")
    ap.add_argument("--procs", type=int, default=1, help="processes (one single-threaded oracle each)")
    a = ap.parse_args()
    cfg = dict(getattr(synth, a.config))
    if a.procs > 1:
        res = time_sample_parallel(a.N, a.queries, cfg, a.procs, a.seed)
    else:
        res = time_sample(a.N, a.queries, cfg, a.seed)
    print(json.dumps(res))


if __name__ == "__main__":
    main()
