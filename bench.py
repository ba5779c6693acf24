"""CSA2 decode benchmark: query-layers/s of the 20-layer decoder step on one GB300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--workload decode1m|decode128k|decode128k_hi32|decode128k_verify6|prefill_compress|prefill|sweep]
               [--impl gb300|reference] [--batch B]

The default workload is decode1m (N = 1,048,576 visible entries, B = 64 sequences), the
1M-context end of the metric's 128K-1M range; decode128k is the 128K end (B = 32).

A step = one decode token for B independent sequences of N visible entries: the new
token's entry is compressed into the cache (m = 1), then the decoder schedule
[Full, Reuse x3] + 4 x [Reindex, Reuse x3] runs, each layer its own index step and
sparse attention.  One query-layer = one query through one attention layer including
its index step.  Under torchrun every rank runs its own batch of sequences (weak
scaling, no collective on the data path).
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from fp4_compressed_sparse_02_gb300 import build as libbuild  # noqa: E402
from fp4_compressed_sparse_02_gb300 import csa2, synth, workload  # noqa: E402
from fp4_compressed_sparse_02_gb300.schedule import FULL, REINDEX, REUSE  # noqa: E402

METRIC = "CSA2 decode query-layers/s at 128K–1M ctx; achieved HBM GB/s vs ~8 TB/s peak"
WORKLOADS = {"decode128k": synth.DEC128K, "decode1m": synth.DEC1M, "decode128k_hi32": synth.DEC128K_HI32,
             "decode128k_ik8": synth.DEC128K_IK8, "decode1m_ik8": synth.DEC1M_IK8,
             "decode128k_verify6": synth.DEC128K_V6, "prefill_compress": synth.PREFILL, "prefill": synth.PREFILL,
             "sweep": synth.DEC1M}
SYNTH_NAME = {"decode128k": "DEC128K", "decode1m": "DEC1M", "decode128k_hi32": "DEC128K_HI32",
              "decode128k_verify6": "DEC128K_V6"}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return j.get("hbm_gbs", 6800.0), "measured"
    return 6800.0, "fallback"


def bf16_peak():
    """Dense bf16 tensor peak (burst) of this GPU, TFLOP/s."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f).get("bf16_tflops", 1900.0), "measured"
    return 1900.0, "fallback"


PROFILES = {("k_attn_tc", "decode128k"): ("k_attn_tc_decode128k.md", "attn.cu"),
            ("k_attn_tc", "decode1m"): ("k_attn_tc_decode1m.md", "attn.cu"),
            ("k_full_scan", "decode1m"): ("k_full_scan_decode1m.md", "index.cu"),
            ("k_full_scan", "decode1m_ik8"): ("k_full_scan_decode1m_ik8.md", "index.cu"),
            ("k_full_scan_short", "decode128k_ik8"): ("k_full_scan_short_decode128k_ik8.md", "index.cu"),
            ("k_full_scan", "decode128k"): ("k_full_scan_decode128k.md", "index.cu"),
            ("k_select_cl_reindex", "decode128k"): ("k_select_cl_reindex_decode128k.md", "index.cu"),
            ("k_proj_tc", "prefill_compress"): ("k_proj_tc_prefill_compress.md", "proj_tc.cu"),
            ("k_score_tc", "decode128k_hi32"): ("k_score_tc_decode128k_hi32.md", "score_tc.cu")}


def profiled_traffic(kernel, workload_name):
    """DRAM bytes per launch from the committed ncu summary of this kernel and workload,
    or None when there is none or the kernel source changed since it was captured."""
    import hashlib
    key = PROFILES.get((kernel, workload_name))
    if key is None:
        return None
    prof = os.path.join(ROOT, "profiles", key[0])
    src = os.path.join(ROOT, "fp4_compressed_sparse_02_gb300", "csrc", key[1])
    if not (os.path.exists(prof) and os.path.exists(src)):
        return None
    fields = {}
    for ln in open(prof):
        if ":" in ln:
            k, v = ln.split(":", 1)
            fields[k.strip()] = v.strip()
    sha = hashlib.sha1(open(src, "rb").read()).hexdigest()
    if fields.get(f"source_sha1 ({key[1]})") != sha:
        return None
    return int(fields["dram_bytes_per_launch"])


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, dev):
        self.dev = dev
        self.proc = None
        self.f = tempfile.TemporaryFile(mode="w+")

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "25", "-i", str(self.dev)], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.seek(0)
        rows = [ln.split(",") for ln in self.f.read().strip().splitlines() if ln.strip()]
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[0]))
                mx = float(r[1])
                for nm, v in zip(names, r[4:8]):
                    if v.strip() == "Active":
                        reasons.add(nm)
            except (ValueError, IndexError):
                continue
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


def host_cpu():
    """Host cores this process may use, all online cores, and the CPU model name (lscpu)."""
    try:
        usable = len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        usable = os.cpu_count() or 1
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.split(":")[0].strip() == "Model name":
                model = ln.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    return usable, os.cpu_count() or usable, model


def mem_available():
    try:
        for ln in open("/proc/meminfo"):
            if ln.startswith("MemAvailable:"):
                return int(ln.split()[1]) * 1024
    except OSError:
        pass
    return None


def cpu_baseline(N, config_name):
    """The oracle on the host's cores, on a bounded sample of the workload: single-threaded,
    and one single-threaded process per usable core (the reported value).  The process count
    is limited only by the cores this process may run on, the sample's queries and the host
    memory one oracle sequence needs (about 2 KB per entry in float64)."""
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1")

    def run(procs, queries):
        r = subprocess.run([sys.executable, "-m", "oracle.timing", "--N", str(N), "--queries", str(queries),
                            "--config", config_name, "--procs", str(procs)], cwd=ROOT, env=env, capture_output=True,
                           text=True, timeout=900)
        if r.returncode != 0:
            return None, (r.stderr.strip().splitlines()[-1] if r.stderr else "failed")
        return json.loads(r.stdout.strip().splitlines()[-1]), None

    usable, online, model = host_cpu()
    per_proc = 2200 * N                            # bytes of one oracle sequence at its peak
    avail = mem_available()
    mem_cap = max(1, int(0.6 * avail) // per_proc) if avail else usable
    procs = max(1, min(usable, mem_cap))
    # about 10-30 s of oracle work: a 1M-entry query-step costs ~8x a 128K one
    q1 = 16 if N <= 262144 else 4
    queries = max(2 * procs, 32) if N <= 262144 else 2 * procs
    host = {"nproc": usable, "online_cpus": online, "model": model,
            "mem_available_gb": round(avail / 1e9, 1) if avail else None}
    one, err = run(1, q1)
    if one is None:
        return {"error": err, "host": host}
    single = {"value": one["value"], "cores": 1, "seconds": one["seconds"], "queries": q1}
    desc = f"query-steps (1 query x 20 layers each, its own sequence of N={N} entries), float64 numpy"
    many, err = run(procs, queries) if procs > 1 else (None, None)
    if many is None:
        return {"value": one["value"], "unit": "query-layers/s", "cores": 1, "kind": "oracle",
                "sample": f"{q1} {desc}, {one['seconds']:.1f} s single-threaded", "host": host}
    cap = "" if procs == usable else f" (memory limits the processes to {procs} of {usable} cores)"
    return {"value": many["value"], "unit": "query-layers/s", "cores": many["procs"], "kind": "oracle",
            "sample": f"{queries} {desc}, spread over {many['procs']} single-threaded processes{cap} "
                      f"(the slowest timed {many['seconds']:.1f} s)",
            "single_thread": single, "host": host}


def run_reference(a):
    """The CPU oracle timed as the reference arm, on the host cores: each step is one
    query-layer of the same workload (the 20-layer decoder schedule walked one layer per
    step, with the append at its first layer, over a pool of two queries that each own a
    sequence of N entries), so a run of K steps is K / 20 query-steps and its memory stays
    bounded whatever K is."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    if a.workload not in SYNTH_NAME:
        print(json.dumps({"impl": "reference", "unavailable": f"the oracle reference arm times decode query-steps; "
                                                               f"{a.workload} has no oracle timing"}), flush=True)
        return
    cfg = WORKLOADS[a.workload]
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1")
    sys.path.insert(0, ROOT)
    os.environ.update(env)
    from oracle import timing
    import numpy as np
    r = np.random.default_rng(0)
    xs = [timing.make_query(r, cfg["N"], dict(cfg)) for _ in range(2)]
    stepper = timing.LayerSteps(xs, cfg["N"], dict(cfg))
    for _ in range(a.warmup):
        stepper.step()
    t0 = time.perf_counter()
    for _ in range(a.steps):
        stepper.step()
    dt = time.perf_counter() - t0
    val = a.steps / dt
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "query-layers/s", "n_gpus": a.gpus,
            "steps": a.steps, "warmup": a.warmup, "ms_per_step": 1000 * dt / a.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{a.workload}: CPU oracle, one query-layer per step (the decoder schedule "
                                   f"walked layer by layer over 2 queries, each its own sequence of N={cfg['N']})"},
            "cpu_baseline": {"value": val, "unit": "query-layers/s", "cores": 1, "kind": "oracle",
                             "sample": f"{a.steps} query-layers = {a.steps / 20:g} query-steps of 20 layers, "
                                       f"N={cfg['N']}, single-threaded float64 numpy"},
            "e2e": {"value": val, "unit": "query-layers/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_prefill_compress(a):
    """The compressor of the encoder prefill chunk alone (65,536 bf16 tokens at m = 2 into
    32,768 FP4 entries with their indexer K): the tensor-bound step, timed on one GPU
    against the measured bf16 tensor peak."""
    import math
    libbuild.build()
    cfg = synth.PREFILL
    T, m, d, d_model, d_ik, d_rope = (cfg[x] for x in ("T", "m", "d", "d_model", "d_ik", "d_rope"))
    G = T // m
    dev = "cuda"
    g = torch.Generator(device=dev).manual_seed(0)
    H = torch.randn((T, d_model), generator=g, device=dev).to(torch.bfloat16)
    Wkv = (torch.randn((d_model, d), generator=g, device=dev) / math.sqrt(d_model)).to(torch.bfloat16)
    Wz = (torch.randn((d_model, d), generator=g, device=dev) / math.sqrt(d_model)).to(torch.bfloat16)
    Wik = (torch.randn((d, d_ik), generator=g, device=dev) / math.sqrt(d)).to(torch.bfloat16)
    pt = torch.randperm(G // 64, generator=torch.Generator().manual_seed(0)).to(torch.int32).reshape(1, -1)
    cache = csa2.PagedCache.allocate(1, G, d, d_ik, dev, pt)
    seq = torch.zeros(G, dtype=torch.int32, device=dev)
    entry = torch.arange(G, dtype=torch.int32, device=dev)
    pos = torch.arange(G, dtype=torch.int32, device=dev) * m + m - 1
    cos, sin = (torch.from_numpy(t).to(dev) for t in synth.rope_tables(T, d_rope))
    ws = csa2.Workspace()
    stream = torch.cuda.Stream()

    def step():
        csa2.compress_quant(cache, seq, entry, m=m, H=H, W_kv=Wkv, W_z=Wz, pos=pos, rope_cos=cos, rope_sin=sin,
                            W_ik=Wik, ws=ws)

    with torch.cuda.stream(stream):
        for _ in range(a.warmup):
            step()
    torch.cuda.synchronize()
    assert csa2.device_error() == 0
    clocks = ClockSampler(0)
    clocks.start()
    time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(a.steps):
            step()
        e1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = e0.elapsed_time(e1) / a.steps
    flops = 2.0 * T * d_model * 2 * d + 2.0 * G * d * d_ik        # the two projections + indexer K
    tflops = flops / (ms / 1000.0) / 1e12
    peak, peak_kind = bf16_peak()
    line = {"metric": "CSA2 compressor of the encoder prefill chunk (tokens/s)", "value": T / (ms / 1000.0),
            "unit": "tokens/s", "n_gpus": 1, "steps": a.steps, "warmup": a.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": f"prefill_compress: T={T} bf16 tokens, m={m}, d_model={d_model}, d={d}, "
                                   f"d_ik={d_ik} -> {G} FP4 entries", "l2": "inputs larger than L2 (671 MB of H)"},
            "roofline": {"bound": "tensor",
                         "kernel": "csa2_compress_quant (k_proj_tc + k_index_k_tc; k_proj_tc is ~94 % of it), "
                                   "timed as the whole call",
                         "achieved": tflops, "peak": peak, "unit": "TFLOP/s", "frac": tflops / peak,
                         "traffic": profiled_traffic("k_proj_tc", "prefill_compress"), "traffic_kernel": "k_proj_tc",
                         "peak_source": peak_kind, "flop_per_step": flops},
            "clocks": clk, "gpu_launches": 2 * a.steps}
    print(json.dumps(line), flush=True)


def max_over_ranks(x, world, device):
    """The largest of every rank's value of x (the slowest rank's time); x itself on one rank."""
    if world <= 1:
        return x
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return t.item()


def whole_job_rate(units_per_rank, world, steps, ms_total):
    """Units all ranks processed per second, over the slowest rank's time (weak scaling: every
    rank processes its own batch)."""
    return units_per_rank * world * steps / (ms_total / 1000.0)


def bf16_peak_sustained():
    """Dense bf16 tensor peak of this GPU held for seconds under the power cap, TFLOP/s."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        if "bf16_tflops_sustained" in j:
            return j["bf16_tflops_sustained"], "measured"
    return 1700.0, "fallback"


def run_prefill(a):
    """The whole encoder prefill chunk: 3 groups x [compress 65,536 tokens at m = 2, Full
    index of the 8,192 causal query tokens, attention of 6 layers (Full + Reuse x 5)] =
    18 query-layers per query token.  Tensor-bound; reported against the sustained bf16
    peak, with the attention (the dominant kernel) timed live by events."""
    libbuild.build()
    cfg = synth.PREFILL
    chunk, info = workload.build_prefill(cfg, seed=0, device="cuda")
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        chunk.run()                                # sizes workspaces, sets kernel attributes
    torch.cuda.synchronize()
    assert csa2.device_error() == 0
    st0 = chunk.steps[0]
    nL = len(st0.layers)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(a.steps)]

    def one(e=None):
        for gi in range(len(chunk.groups)):
            if gi == 0 and e is not None:
                e[0].record(stream)
                chunk.run_compress(0)
                e[1].record(stream)
                st0.run_index(0)
                e[2].record(stream)
                for i in range(nL):
                    st0.run_attn(i)
                e[3].record(stream)
            else:
                chunk.run_group(gi)

    with torch.cuda.stream(stream):
        for _ in range(a.warmup):
            one()
    torch.cuda.synchronize()
    clocks = ClockSampler(0)
    clocks.start()
    time.sleep(0.3)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        t0.record(stream)
        for j in range(a.steps):
            one(evs[j])
        t1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    assert csa2.device_error() == 0
    ms = t0.elapsed_time(t1) / a.steps
    comp_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    idx_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)
    attn_ms = statistics.mean(e[2].elapsed_time(e[3]) for e in evs) / nL
    Q, L = info["Q"], info["layers"]
    fl = info["flops"]
    chunk_flops = info["groups"] * (fl["compress"] + fl["index"]) + L * fl["attn"]
    peak, peak_kind = bf16_peak_sustained()
    attn_tf = fl["attn"] / (attn_ms / 1000.0) / 1e12
    chunk_tf = chunk_flops / (ms / 1000.0) / 1e12
    # end to end: every chunk's inputs (hidden states, Main Q, indexer Q and weights, window
    # rows) copied from pinned host memory, the chunk, the last layer's output read back.
    # Double-buffered: chunk s's inputs are copied (copy stream) into device set s % 2 while
    # chunk s - 1 runs on the other set; each output is read back on a third stream.  (Four copy
    # streams sharing the inputs measured slower than one.)
    host_in = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True).copy_(t) for t in chunk.inputs]
    chunk2, _ = workload.build_prefill(cfg, seed=1, device="cuda")
    with torch.cuda.stream(stream):
        chunk2.run()                               # sizes its workspaces
    torch.cuda.synchronize()
    sets = [chunk, chunk2]
    out_last = chunk.steps[-1].out[-1]
    host_out = torch.empty(out_last.shape, dtype=out_last.dtype, pin_memory=True)
    h2d = sum(h.numel() * h.element_size() for h in host_in)
    d2h = host_out.numel() * host_out.element_size()
    e2e_steps = max(2, a.steps // 4)
    copy_st, read_st = torch.cuda.Stream(), torch.cuda.Stream()
    copied = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]
    torch.cuda.synchronize()
    u0, u1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    u0.record(copy_st)
    for s_ in range(e2e_steps):
        c = sets[s_ % 2]
        with torch.cuda.stream(copy_st):
            if s_ >= 2:
                copy_st.wait_event(done[s_ % 2])   # chunk s - 2 has finished with this set
            for dev_t, host_t in zip(c.inputs, host_in):
                dev_t.copy_(host_t, non_blocking=True)
            copied[s_ % 2].record(copy_st)
        with torch.cuda.stream(stream):
            stream.wait_event(copied[s_ % 2])
            for gi in range(len(c.groups)):
                c.run_group(gi)
            done[s_ % 2].record(stream)
        with torch.cuda.stream(read_st):
            read_st.wait_event(done[s_ % 2])
            host_out.copy_(c.steps[-1].out[-1], non_blocking=True)
    u1.record(read_st)
    torch.cuda.synchronize()
    e2e_ms = u0.elapsed_time(u1) / e2e_steps
    del chunk2, sets
    line = {"metric": "CSA2 encoder prefill chunk query-layers/s (8,192 causal queries x 18 layers)",
            "value": Q * L / (ms / 1000.0), "unit": "query-layers/s", "n_gpus": 1, "steps": a.steps,
            "warmup": a.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"prefill: T={info['T']} tokens at m={info['m']} ({info['NE']} entries) per "
                                   f"group, {info['groups']} groups x [compress, Full index, attention x "
                                   f"{nL}] for Q={Q} causal query tokens, d_kv={info['d']}, Hq={info['Hq']}, "
                                   f"indexer {info['H_i']}x{info['d_ik']}, Top-{info['k']}, SWA {info['W']}",
                       "l2": "inputs larger than L2 (671 MB of H and 537 MB of Main Q per layer)"},
            "roofline": {"bound": "tensor", "kernel": "k_attn_tc (csa2_sparse_attn, one layer of 8,192 queries; "
                                                      "mean of the 6 layers of group 0)",
                         "achieved": attn_tf, "peak": peak, "unit": "TFLOP/s", "frac": attn_tf / peak,
                         "traffic": None, "peak_source": peak_kind + " (sustained)", "flop_per_launch": fl["attn"],
                         "ms": attn_ms},
            "chunk": {"flop": chunk_flops, "achieved_tflops": chunk_tf, "frac": chunk_tf / peak,
                      "ms_compress": comp_ms, "ms_index_full": idx_ms, "ms_attn_layer": attn_ms},
            "clocks": clk, "gpu_launches": a.steps * info["groups"] * (2 + 3 + nL),
            "e2e": {"value": Q * L / (e2e_ms / 1000.0), "unit": "query-layers/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h}}
    print(json.dumps(line), flush=True)


def run_sweep(a):
    """The batched paged decode sweep: batch B in 1, 2, 4, ..., 256 sequences, each context
    drawn uniformly from {4K, 64K, 256K, 1M} entries, one 20-layer decoder step (with the
    append) per timed iteration.  Every iteration is timed alone by events after a write
    of a buffer twice the L2 size, so small batches are not served from L2."""
    import numpy as np
    libbuild.build()
    ctx = [4096, 65536, 262144, 1048576]
    peak, peak_kind = peaks()
    flush = torch.empty(2 * 129 * 2 ** 20 // 4, dtype=torch.float32, device="cuda")
    stream = torch.cuda.Stream()
    rows = []
    clocks = ClockSampler(0)
    clocks.start()
    launches = 0
    for B in (1, 2, 4, 8, 16, 32, 64, 128, 256):
        r = np.random.default_rng(1000 + B)
        Ns = r.choice(ctx, size=B)
        step, info = workload.build_decode(synth.DEC1M, Ns=Ns, seed=2000 + B)
        nbytes = workload.algorithmic_bytes(info)["total"]
        with torch.cuda.stream(stream):
            step.run()
        torch.cuda.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            step.run()
        with torch.cuda.stream(stream):
            for _ in range(a.warmup):
                gr.replay()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(a.steps)]
        with torch.cuda.stream(stream):
            for e0, e1 in evs:
                flush.fill_(1.0)
                e0.record(stream)
                gr.replay()
                e1.record(stream)
        torch.cuda.synchronize()
        assert csa2.device_error() == 0
        ms = statistics.mean(e0.elapsed_time(e1) for e0, e1 in evs)
        modes = info["schedule"]
        launches += a.steps * (2 + 2 * list(modes).count(FULL) + list(modes).count(REINDEX) + len(modes))
        gbs = nbytes / (ms / 1000.0) / 1e9
        rows.append({"B": B, "contexts": {str(c): int((Ns == c).sum()) for c in ctx}, "ms_per_step": ms,
                     "query_layers_per_s": B * info["layers"] / (ms / 1000.0), "algorithmic_bytes": nbytes,
                     "achieved_gbs": gbs, "frac": gbs / peak})
        del step, gr
        torch.cuda.empty_cache()
    clk = clocks.stop()
    last = rows[-1]
    line = {"metric": METRIC, "value": last["query_layers_per_s"], "unit": "query-layers/s", "n_gpus": 1,
            "steps": a.steps, "warmup": a.warmup, "ms_per_step": last["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "sweep: batched paged 20-layer decode step, contexts drawn from {4K, 64K, 256K, 1M} "
                                   "entries, batch 1..256 (value, ms_per_step: batch 256)",
                       "l2": "a 258 MB buffer written before every timed step"},
            "roofline": {"bound": "hbm", "kernel": "whole 20-layer step (all kernels), batch 256",
                         "achieved": last["achieved_gbs"], "peak": peak, "unit": "GB/s", "frac": last["frac"],
                         "traffic": None, "peak_source": peak_kind},
            "sweep": rows, "clocks": clk, "gpu_launches": launches}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="decode1m", choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--batch", type=int, default=None, help="sequences per GPU (default: the workload's)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    a = ap.parse_args()
    a.steps_default = a.steps is None
    if a.steps is None:
        a.steps = 2000
    a.warmup = max(a.warmup, 3)
    if a.impl == "reference":
        run_reference(a)
        return

    if a.workload == "prefill_compress":
        run_prefill_compress(a)
        return
    if a.workload == "sweep":
        if a.steps_default:
            a.steps = 20
        run_sweep(a)
        return
    if a.workload == "prefill":
        if a.steps_default:
            a.steps = 10
        run_prefill(a)
        return

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    libbuild.build()
    cfg = WORKLOADS[a.workload]
    step, info = workload.build_decode(cfg, B=a.batch, seed=1000 + rank, device=f"cuda:{local}")
    nbytes = workload.algorithmic_bytes(info)
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()

    # eager warm-up sizes the workspace and sets kernel attributes before capture
    with torch.cuda.stream(stream):
        step.run()
    torch.cuda.synchronize()
    # The timed loop replays graphs that each hold S consecutive steps (few launch gaps).
    # In the first captured step of each graph, external event-record nodes bracket the
    # layer-0 Full indexer call (scan + select), the three back-to-back Reuse-layer attention
    # calls (layers 1..3) and the layer-4 Reindex call.  NG such graphs, each with its own
    # events, are replayed in turn, so the timed region gives up to NG samples of each.  (An
    # event node between two kernels turns their programmatic launch edge into a full one, so
    # the other S - 1 steps of a graph carry none.)
    modes = info["schedule"]
    assert modes[0] == FULL and list(modes[1:4]) == [REUSE] * 3 and modes[4] == REINDEX
    S = next(d for d in (10, 5, 4, 2, 1) if a.steps % d == 0)
    NG = max(1, min(5, a.steps // S))
    evs = [[torch.cuda.Event(enable_timing=True, external=True) for _ in range(6)] for _ in range(NG)]

    def one_step(e):
        step.run_append()
        e[0].record(stream)
        step.run_index(0)
        e[1].record(stream)
        step.run_attn(0)
        e[2].record(stream)
        for i in (1, 2, 3):
            step.run_layer(i)
        e[3].record(stream)
        step.run_index(4)
        e[4].record(stream)
        step.run_attn(4)
        e[5].record(stream)
        for i in range(5, len(step.layers)):
            step.run_layer(i)

    g_multi = []
    for gi in range(NG):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for j in range(S):
                if j == 0:
                    one_step(evs[gi])
                else:
                    step.run()
        g_multi.append(g)
    g_one = torch.cuda.CUDAGraph()                 # one step, for the end-to-end loop
    with torch.cuda.graph(g_one, stream=stream):
        step.run()

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    with torch.cuda.stream(stream):
        for r_ in range((a.warmup + S - 1) // S):
            g_multi[r_ % NG].replay()
    torch.cuda.synchronize()

    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    with torch.cuda.stream(stream):
        t_start.record(stream)
        for r_ in range(a.steps // S):
            g_multi[r_ % NG].replay()
        t_end.record(stream)
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop()
    ms_total = t_start.elapsed_time(t_end)
    full_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    attn_ms = statistics.mean(e[2].elapsed_time(e[3]) for e in evs) / 3.0
    reindex_ms = statistics.mean(e[3].elapsed_time(e[4]) for e in evs)
    ms_total = max_over_ranks(ms_total, world, f"cuda:{local}")
    ms_step = ms_total / a.steps
    B = info["B"]
    ql = B * info["layers"] * world
    value = whole_job_rate(B * info["layers"], world, a.steps, ms_total)

    # end to end: per step, copy the step's inputs from pinned host memory, run the step,
    # read the last layer's output back.  The device inputs and outputs are double-buffered:
    # step s+1's inputs are uploaded on a copy stream while step s runs (set s % 2 is
    # reused once step s - 2 has finished), and each result is read back on a third stream.
    keys = [(i, key) for i, L in enumerate(step.layers) for key in ("q", "q_idx", "w") if key in L]
    def dev_inputs():
        return [step.layers[i][key] for i, key in keys] + [step.append["H"]]
    def set_inputs(ts):
        for (i, key), t in zip(keys, ts):
            step.layers[i][key] = t
        step.append["H"] = ts[-1]
    set0 = dev_inputs()
    set1 = [t.clone() for t in set0]
    host_in = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True).copy_(t) for t in set0]
    outs = [step.out[-1], step.out[-1].clone()]
    host_out = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in outs]
    h2d = sum(h.numel() * h.element_size() for h in host_in)
    d2h = host_out[0].numel() * host_out[0].element_size()
    g_e2e = [g_one, torch.cuda.CUDAGraph()]
    set_inputs(set1)
    step.out[-1] = outs[1]
    with torch.cuda.stream(stream):                # sizes nothing new; the workspace is allocated
        step.run()
    torch.cuda.synchronize()
    with torch.cuda.graph(g_e2e[1], stream=stream):
        step.run()
    set_inputs(set0)
    step.out[-1] = outs[0]
    sets = [set0, set1]
    copy_st, d2h_st = torch.cuda.Stream(), torch.cuda.Stream()
    ready = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]
    read = [torch.cuda.Event() for _ in range(2)]   # output set b read back
    e2e_steps = max(10, a.steps // 10)
    barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(copy_st)
    for s_ in range(e2e_steps):
        b_ = s_ % 2
        with torch.cuda.stream(copy_st):
            if s_ >= 2:
                copy_st.wait_event(done[b_])
            for dev_t, host_t in zip(sets[b_], host_in):
                dev_t.copy_(host_t, non_blocking=True)
            ready[b_].record(copy_st)
        stream.wait_event(ready[b_])
        if s_ >= 2:
            stream.wait_event(read[b_])
        with torch.cuda.stream(stream):
            g_e2e[b_].replay()
            done[b_].record(stream)
        d2h_st.wait_event(done[b_])
        with torch.cuda.stream(d2h_st):
            host_out[b_].copy_(outs[b_], non_blocking=True)
            read[b_].record(d2h_st)
    e1.record(d2h_st)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    e2e_ms = max_over_ranks(e2e_ms, world, f"cuda:{local}")
    e2e_val = whole_job_rate(B * info["layers"], world, 1, e2e_ms)

    if rank == 0:
        peak, peak_kind = peaks()
        attn_bytes = B * nbytes["per_query"]["attn"]
        attn_gbs = attn_bytes / (attn_ms / 1000.0) / 1e9
        full_bytes = B * nbytes["per_query"]["full"]
        full_gbs = full_bytes / (full_ms / 1000.0) / 1e9
        reindex_bytes = B * nbytes["per_query"]["reindex"]
        reindex_gbs = reindex_bytes / (reindex_ms / 1000.0) / 1e9
        step_gbs = nbytes["total"] / (ms_step / 1000.0) / 1e9
        # the Full call scores on the tensor cores when a group's heads fill >= 16 columns
        ik8 = bool(info.get("ik8"))
        tc_full = (not ik8 and info["d_ik"] == 128 and info["H_i"] in (8, 16, 32) and
                   info["H_i"] * info.get("G", 1) >= 16)
        # the FP8 form scans blocks of at most 64 entries (one head group, P = 8) with k_full_scan_short
        short_scan = (ik8 and info["d_ik"] == 128 and info["H_i"] <= 8 and info.get("G", 1) == 1 and
                      info["P"] == 8 and -(-info["N"] // info["NB"]) <= 64)
        scan_kernel = "k_full_scan_short" if short_scan else "k_full_scan"
        full_kernels = ("k_score_tc + k_block_topp + k_select_cl" if tc_full else
                        scan_kernel + " + k_select_cl" + (" (+ k_quant_q8, FP8 indexer)" if ik8 else ""))
        # kernels per step: compressor append 2 (projection; quantisation + indexer K), Full
        # indexer 2 (scan, select) or 3 (score, block top-P, select; or FP8: Q quantisation,
        # scan, select), Reindex 1 (FP8: 2), attention 1 per layer
        launches = (2 + (3 if (tc_full or ik8) else 2) * list(modes).count(FULL) +
                    (2 if ik8 else 1) * list(modes).count(REINDEX) + len(modes))
        n_full = list(modes).count(FULL)
        n_reindex = list(modes).count(REINDEX)
        roof = {
            "attn": {"bound": "hbm", "kernel": "k_attn_tc (csa2_sparse_attn, one layer; mean of 3 back-to-back)",
                     "achieved": attn_gbs, "peak": peak, "unit": "GB/s", "frac": attn_gbs / peak,
                     "traffic": profiled_traffic("k_attn_tc", a.workload), "peak_source": peak_kind,
                     "algorithmic_bytes": attn_bytes, "ms": attn_ms, "launches_per_step": len(modes),
                     "share_of_step": len(modes) * attn_ms / ms_step},
            "index_full": {"bound": "hbm", "kernel": full_kernels + " (csa2_index_full)",
                           "achieved": full_gbs, "peak": peak, "unit": "GB/s", "frac": full_gbs / peak,
                           "traffic": profiled_traffic(full_kernels.split(" ")[0], a.workload),
                           "traffic_kernel": full_kernels.split(" ")[0], "peak_source": peak_kind,
                           "algorithmic_bytes": full_bytes, "ms": full_ms, "launches_per_step": n_full,
                           "share_of_step": n_full * full_ms / ms_step},
            "index_reindex": {"bound": "hbm", "kernel": "k_select_cl (csa2_index_reindex, scoring fused in)",
                              "achieved": reindex_gbs, "peak": peak, "unit": "GB/s", "frac": reindex_gbs / peak,
                              "traffic": profiled_traffic("k_select_cl_reindex", a.workload),
                              "traffic_kernel": "k_select_cl", "peak_source": peak_kind,
                              "algorithmic_bytes": reindex_bytes, "ms": reindex_ms, "launches_per_step": n_reindex,
                              "share_of_step": n_reindex * reindex_ms / ms_step},
        }
        dominant = max(roof, key=lambda k_: roof[k_]["share_of_step"])
        line = {
            "metric": METRIC, "value": value, "unit": "query-layers/s", "n_gpus": world, "steps": a.steps,
            "warmup": a.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"{a.workload}: 20-layer CSA2 decoder step, N={info['N']} visible entries, "
                                   + (f"B={B} sequences per GPU" if info.get("G", 1) == 1 else
                                      f"B={info['seqs']} sequences x {info['G']} verification positions = {B} "
                                      f"queries per GPU (Full scan of a sequence shared by its {info['G']} queries)")
                                   + f", Top-{info['k']}, SWA {info['W']}, pool {info['NB']}x{info['P']}",
                       "N": info["N"], "B": B, "layers": info["layers"], "d_kv": info["d"], "Hq": info["Hq"],
                       "indexer": f"{info['H_i']}x{info['d_ik']}" + (", FP8 E4M3 indexer K and Q" if ik8 else
                                                                      ", bf16 indexer K"),
                       "parallelism": f"replicas x{world}",
                       "l2": f"inputs larger than L2: {nbytes['total'] / 1e9:.2f} GB algorithmic bytes per step"},
            "roofline": dict(roof[dominant], dominant_of=sorted(roof), event_samples=len(evs)),
            "roofline_attn": roof["attn"],
            "roofline_index_full": roof["index_full"],
            "roofline_index_reindex": roof["index_reindex"],
            "step_hbm": {"algorithmic_bytes": nbytes["total"], "achieved_gbs": step_gbs, "frac": step_gbs / peak,
                         "peak": peak, "peak_source": peak_kind},
            "clocks": clk,
            "gpu_launches": a.steps * launches,
            "e2e": {"value": e2e_val, "unit": "query-layers/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
        }
        if not a.no_cpu_baseline and a.workload in SYNTH_NAME:
            line["cpu_baseline"] = cpu_baseline(info["N"], SYNTH_NAME[a.workload])
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
