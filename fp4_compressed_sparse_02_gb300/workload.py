"""Seeded synthetic decode workloads built directly on the device (for sizes where a host
round trip would dominate set-up).  Same recipes as synth.py (random bytes for FP4
codes, E4M3 scale bytes in [0x20, 0x3F], N(0,1) bf16 for indexer K / queries / hidden
states, weights N(0, 1/fan_in), E4M3 SWA rows with exponent field 3..13 and row scales
in [0.005, 0.02]); no arithmetic of the method happens here."""
import math

import numpy as np
import torch

from . import csa2, synth
from .schedule import FULL, REINDEX, REUSE, DecodeStep, decoder_schedule


def _randn_bf16(shape, g, device, sigma=1.0):
    return (torch.randn(shape, generator=g, device=device, dtype=torch.float32) * sigma).to(torch.bfloat16)


def _fp8_rows(rows, d, g, device):
    sign = torch.randint(0, 2, (rows, d), generator=g, device=device, dtype=torch.int32) << 7
    expo = torch.randint(3, 14, (rows, d), generator=g, device=device, dtype=torch.int32) << 3
    man = torch.randint(0, 8, (rows, d), generator=g, device=device, dtype=torch.int32)
    return (sign | expo | man).to(torch.uint8)


def build_decode(cfg, B=None, N=None, seed=0, device="cuda", append=True, schedule=None, chunk_pages=32768,
                 Ns=None, G=None):
    """A decode step of B independent sequences with N visible entries each (or Ns[b]
    entries for sequence b when Ns is given; N is then max(Ns)).

    G > 1 (cfg["G"] by default): G consecutive queries per sequence, the positions of a
    speculative-decoding verification step: query (b, t) sees Ns[b] - G + 1 + t entries,
    appends its own entry, and the Full scan runs the G queries of a sequence together.

    The cache holds N (Ns[b]) entries per sequence (the last one is rewritten by the
    step's append when append=True).  Pages are a random permutation; page-table slots
    past a sequence's length point at page 0 and are never read.  Returns (DecodeStep,
    info)."""
    if Ns is not None:
        Ns = [int(x) for x in Ns]
        B = len(Ns)
        N = max(Ns)
    B = B or cfg["B"]
    N = N or cfg["N"]
    Ns = Ns or [N] * B
    G = G or cfg.get("G", 1)
    Q = B * G                                    # queries
    d, d_ik, H_i, Hq, W, k = cfg["d"], cfg["d_ik"], cfg["H_i"], cfg["Hq"], cfg["W"], cfg["k"]
    NB, P, d_model, d_rope = cfg["NB"], cfg["P"], cfg["d_model"], cfg["d_rope"]
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    gc = torch.Generator()
    gc.manual_seed(seed)
    mp = (N + 63) // 64
    used = [(n + 63) // 64 for n in Ns]
    num_pages = sum(used)
    perm = torch.randperm(num_pages, generator=gc).to(torch.int32)
    page_table = torch.zeros((B, mp), dtype=torch.int32)
    o = 0
    for b, u in enumerate(used):
        page_table[b, :u] = perm[o:o + u]
        o += u
    page_table = page_table.to(device)
    ik8 = bool(cfg.get("ik8"))
    cache = csa2.PagedCache(
        codes=torch.empty((num_pages, 64, d // 2), dtype=torch.uint8, device=device),
        scales=torch.empty((num_pages, 64, d // 16), dtype=torch.uint8, device=device),
        idx_k=None if ik8 else torch.empty((num_pages, 64, d_ik), dtype=torch.bfloat16, device=device),
        page_table=page_table,
        idx_k8=torch.empty((num_pages, 64, d_ik), dtype=torch.uint8, device=device) if ik8 else None,
        idx_k8_scale=torch.empty((num_pages, 64), dtype=torch.float32, device=device) if ik8 else None)
    for p0 in range(0, num_pages, chunk_pages):
        p1 = min(num_pages, p0 + chunk_pages)
        cache.codes[p0:p1] = torch.randint(0, 256, (p1 - p0, 64, d // 2), generator=g, device=device,
                                           dtype=torch.uint8)
        cache.scales[p0:p1] = torch.randint(0x20, 0x40, (p1 - p0, 64, d // 16), generator=g, device=device,
                                            dtype=torch.uint8)
        if ik8:
            cache.idx_k8[p0:p1] = _fp8_rows((p1 - p0) * 64, d_ik, g, device).view(p1 - p0, 64, d_ik)
            cache.idx_k8_scale[p0:p1] = torch.rand((p1 - p0, 64), generator=g, device=device) * 0.015 + 0.005
        else:
            cache.idx_k[p0:p1] = _randn_bf16((p1 - p0, 64, d_ik), g, device)
    seq_of = torch.arange(B, dtype=torch.int32, device=device).repeat_interleave(G)
    nq = [n - G + 1 + t for n in Ns for t in range(G)]
    n_vis = torch.tensor(nq, dtype=torch.int32, device=device)
    sched = schedule or decoder_schedule()
    layers = []
    for mode in sched:
        L = dict(mode=mode, q=_randn_bf16((Q, Hq, d), g, device),
                 swa=_fp8_rows(Q * W, d, g, device),
                 swa_scale=(torch.rand(Q * W, generator=g, device=device) * 0.015 + 0.005).float(),
                 swa_start=torch.arange(Q, dtype=torch.int32, device=device) * W,
                 swa_len=torch.full((Q,), W, dtype=torch.int32, device=device))
        if mode in (FULL, REINDEX):
            L["q_idx"] = _randn_bf16((Q, H_i, d_ik), g, device)
            L["w"] = torch.randn((Q, H_i), generator=g, device=device) / math.sqrt(H_i)
        layers.append(L)
    app = None
    rope = None
    if append:
        app = dict(H=_randn_bf16((Q, d_model), g, device),
                   W_kv=_randn_bf16((d_model, d), g, device, 1 / math.sqrt(d_model)),
                   W_ik=_randn_bf16((d, d_ik), g, device, 1 / math.sqrt(d)),
                   pos=n_vis - 1,
                   seq=seq_of.clone(),
                   entry=n_vis - 1)
        cos, sin = synth.rope_tables(N, d_rope)
        rope = (torch.from_numpy(cos).to(device), torch.from_numpy(sin).to(device))
    step = DecodeStep(cache, seq_of, n_vis, N, layers, NB, P, k, W, append=app, rope=rope, group=G)
    info = dict(B=Q, G=G, seqs=B, N=N, Ns=Ns, layers=len(sched), schedule=sched, d=d, d_ik=d_ik, H_i=H_i, Hq=Hq,
                W=W, k=k, NB=NB, P=P, d_model=d_model, d_rope=d_rope, ik8=ik8)
    return step, info


class PrefillChunk:
    """The encoder prefill chunk: T tokens of one sequence at compression ratio m, then
    3 groups [Full, Reuse x 5] for the last Q tokens as causal queries.  Each group has its
    own hidden states, compressor weights and Main KV cache (T / m entries): the group's
    first layer compresses its chunk, its Full index step scores the causal range of every
    query (the Q queries form one group: one tensor-core product), and its six layers
    attend with their own Main Q over the group's Top-k and their own FP8 window (the
    query's last W tokens)."""

    def __init__(self, groups, steps, inputs):
        self.groups = groups          # per group: dict(cache, H, W_kv, W_z, W_ik)
        self.steps = steps            # per group: DecodeStep over the group's cache
        self.inputs = inputs          # the device tensors a chunk reads from the host

    def run_compress(self, gi):
        G = self.groups[gi]
        csa2.compress_quant(G["cache"], G["seq"], G["entry"], m=G["m"], H=G["H"], W_kv=G["W_kv"], W_z=G["W_z"],
                            pos=G["pos"], rope_cos=G["cos"], rope_sin=G["sin"], W_ik=G["W_ik"], ws=G["ws"])

    def run_group(self, gi):
        self.run_compress(gi)
        st = self.steps[gi]
        for i in range(len(st.layers)):
            st.run_layer(i)

    def run(self):
        for gi in range(len(self.groups)):
            self.run_group(gi)


def build_prefill(cfg, seed=0, device="cuda", n_groups=3, reuse=5):
    """The encoder prefill chunk of cfg (T, m, Q, ...).  Inputs follow the recipes of the
    module docstring; the query tokens are the last Q of the chunk, token t seeing the
    (t + 1) // m entries complete at t.  Returns (PrefillChunk, info)."""
    T, m, d, d_model, d_ik, d_rope = (cfg[x] for x in ("T", "m", "d", "d_model", "d_ik", "d_rope"))
    Hq, H_i, Q, W, k, NB, P = (cfg[x] for x in ("Hq", "H_i", "Q", "W", "k", "NB", "P"))
    NE = T // m
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    gc = torch.Generator()
    gc.manual_seed(seed)
    cos, sin = (torch.from_numpy(t).to(device) for t in synth.rope_tables(T, d_rope))
    tq = torch.arange(T - Q, T, dtype=torch.int32, device=device)
    n_vis = ((tq + 1) // m).to(torch.int32)
    seq_q = torch.zeros(Q, dtype=torch.int32, device=device)
    schedule = [FULL] + [REUSE] * reuse
    # Main Q and the FP8 window rows of the group's layers (one set, shared by the groups:
    # every tensor is larger than L2, so sharing changes no traffic)
    lay = []
    for mode in schedule:
        lay.append(dict(mode=mode, q=_randn_bf16((Q, Hq, d), g, device), swa=_fp8_rows(T, d, g, device),
                        swa_scale=(torch.rand(T, generator=g, device=device) * 0.015 + 0.005).float(),
                        swa_start=(tq - (W - 1)).to(torch.int32),
                        swa_len=torch.full((Q,), W, dtype=torch.int32, device=device)))
    groups, steps = [], []
    inputs = [L["q"] for L in lay] + [L["swa"] for L in lay]
    for _ in range(n_groups):
        pt = torch.randperm(NE // 64, generator=gc).to(torch.int32).reshape(1, -1)
        cache = csa2.PagedCache.allocate(1, NE, d, d_ik, device, pt)
        G = dict(cache=cache, m=m, H=_randn_bf16((T, d_model), g, device),
                 W_kv=_randn_bf16((d_model, d), g, device, 1 / math.sqrt(d_model)),
                 W_z=_randn_bf16((d_model, d), g, device, 1 / math.sqrt(d_model)),
                 W_ik=_randn_bf16((d, d_ik), g, device, 1 / math.sqrt(d)),
                 seq=torch.zeros(NE, dtype=torch.int32, device=device),
                 entry=torch.arange(NE, dtype=torch.int32, device=device),
                 pos=torch.arange(NE, dtype=torch.int32, device=device) * m + m - 1,
                 cos=cos, sin=sin, ws=csa2.Workspace(device))
        layers = [dict(L) for L in lay]
        layers[0]["q_idx"] = _randn_bf16((Q, H_i, d_ik), g, device)
        layers[0]["w"] = torch.randn((Q, H_i), generator=g, device=device) / math.sqrt(H_i)
        steps.append(DecodeStep(cache, seq_q, n_vis, NE, layers, NB, P, k, W, group=Q))
        groups.append(G)
        inputs += [G["H"], layers[0]["q_idx"], layers[0]["w"]]
    n_sum = int(n_vis.sum().item())
    info = dict(T=T, m=m, NE=NE, Q=Q, groups=n_groups, layers=n_groups * len(schedule), d=d, d_model=d_model,
                d_ik=d_ik, H_i=H_i, Hq=Hq, W=W, k=k, NB=NB, P=P, n_vis_sum=n_sum,
                flops=dict(compress=2.0 * T * d_model * 2 * d + 2.0 * NE * d * d_ik,
                           index=2.0 * H_i * d_ik * n_sum,
                           attn=4.0 * Q * Hq * (k + W) * d))
    return PrefillChunk(groups, steps, inputs), info


def algorithmic_bytes(info):
    """Bytes a decode step must move at minimum (each byte read or written once):

    append     : H row (d_model*2) + W_kv + W_ik once (shared by the batch) + the new
                 entry (d/2 + d/16 + ik) per query
    Full       : n*ik of indexer K (once per group of G queries of a sequence) + q_idx
                 + w + pool (4*NB*P) + topk (4k) per query
    Reindex    : pool*ik gathered indexer K + pool ids (4*NB*P) + q_idx + w + topk
    (ik = the bytes of one entry's indexer K: 2*d_ik in bf16, d_ik + 4 in the FP8 form)
    attention  : k*(d/2 + d/16) FP4 rows + W*(d + 4) SWA rows + q (2*Hq*d)
                 + out (2*Hq*d) + topk ids (4k) per query-layer
    """
    B, N, d, d_ik, H_i, Hq, W, k = (info[x] for x in ("B", "N", "d", "d_ik", "H_i", "Hq", "W", "k"))
    pool = info["NB"] * info["P"]
    G = info.get("G", 1)
    ik = d_ik + 4 if info.get("ik8") else 2 * d_ik

    def per_query(n):
        q = {}
        q["full"] = n * ik // G + 2 * H_i * d_ik + 4 * H_i + 4 * pool + 4 * k
        q["reindex"] = min(n, pool) * ik + 4 * pool + 2 * H_i * d_ik + 4 * H_i + 4 * k
        q["attn"] = k * (d // 2 + d // 16) + W * (d + 4) + 2 * Hq * d * 2 + 4 * k
        return q

    per_q = per_query(N)
    tot = 0
    for n in info.get("Ns") or [N] * (B // G):      # each sequence at its own length
        q = per_query(n)
        for mode in info["schedule"]:
            if mode == FULL:
                tot += G * q["full"]
            elif mode == REINDEX:
                tot += G * q["reindex"]
            tot += G * q["attn"]
    app = 0
    if info.get("append", True):
        app = B * (info["d_model"] * 2 + d // 2 + d // 16 + ik) + info["d_model"] * d * 2 + d * d_ik * 2
    return dict(total=tot + app, per_query=per_q, append=app)


def host_sequence(step, b, n):
    """Entries [0, n) of query b's sequence copied to the host: (codes, scales, indexer K),
    the indexer K as bf16 bits, or as (E4M3 bytes, float32 scales) in the FP8 form."""
    pt = step.cache.page_table[int(step.seq_of[b].item())].cpu().numpy()
    e = np.arange(n)
    pages = torch.from_numpy(pt[e // 64].astype(np.int64)).to(step.cache.codes.device)
    slots = torch.from_numpy(e % 64).to(step.cache.codes.device)
    codes = step.cache.codes[pages, slots].cpu().numpy()
    scales = step.cache.scales[pages, slots].cpu().numpy()
    if step.cache.idx_k8 is not None:
        idxk = (step.cache.idx_k8[pages, slots].cpu().numpy(), step.cache.idx_k8_scale[pages, slots].cpu().numpy())
    else:
        idxk = step.cache.idx_k[pages, slots].view(torch.int16).cpu().numpy().view(np.uint16)
    return codes, scales, idxk
