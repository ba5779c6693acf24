"""Layer schedule driver: one decode step of the 20-layer CSA2 decoder through the C ABI.

"DeepSeek-V4.1-Flash deep dive", section 3.2: decoder group 1 = [Full x1 + Reuse x3],
groups 2-5 = [Reindex x1 + Reuse x3]; section 3.3: the pool is built by the decoder's
first Full layer and shared by the Reindex layers; Reuse layers use the most recent
Top-512.  Each layer keeps its own Main Q and SWA window (section 3.1).

Layers run in order as separate library calls (a layer's Q depends on the previous
layer's output in a real model, so nothing is fused across layers).  All outputs are
preallocated so that a whole step can be captured in CUDA graphs.
"""
import torch

from . import csa2

FULL, REINDEX, REUSE = "full", "reindex", "reuse"


def decoder_schedule():
    return [FULL, REUSE, REUSE, REUSE] + [REINDEX, REUSE, REUSE, REUSE] * 4


class DecodeStep:
    """Holds the per-step buffers of B decode queries over a paged cache.

    append: optional dict(H, W_kv, W_ik, pos, seq, entry) -- compress the new token's
            hidden state into the cache (m = 1) before the layers run.
    layers: list of dict(mode, q_idx, w, q, swa, swa_scale, swa_start, swa_len) in
            schedule order (q_idx / w only for Full / Reindex layers).
    """

    def __init__(self, cache, seq_of, n_vis, max_n, layers, num_blocks, per_block, k, swa_max,
                 append=None, rope=None, out_dtype=torch.bfloat16, group=1):
        self.cache = cache
        self.group = group                        # queries per sequence scanned together by Full
        self.seq_of = seq_of
        self.n_vis = n_vis
        self.max_n = max_n
        self.layers = layers
        self.NB, self.P, self.k, self.swa_max = num_blocks, per_block, k, swa_max
        self.append = append
        self.rope = rope
        dev = seq_of.device
        B = seq_of.shape[0]
        self.pool = torch.full((B, num_blocks * per_block), -1, dtype=torch.int32, device=dev)
        self.pool_len = torch.zeros(B, dtype=torch.int32, device=dev)
        self.topk = [torch.full((B, k), -1, dtype=torch.int32, device=dev) for _ in layers]
        self.topk_len = [torch.zeros(B, dtype=torch.int32, device=dev) for _ in layers]
        Hq, d = layers[0]["q"].shape[1:]
        self.out = [torch.empty((B, Hq, d), dtype=out_dtype, device=dev) for _ in layers]
        self.lse = [torch.empty((B, Hq), dtype=torch.float32, device=dev) for _ in layers]
        self.ws = csa2.Workspace(dev)

    def run_append(self):
        if self.append is None:
            return
        a = self.append
        cos, sin = self.rope if self.rope is not None else (None, None)
        csa2.compress_quant(self.cache, a["seq"], a["entry"], m=1, H=a["H"], W_kv=a["W_kv"], pos=a["pos"],
                            rope_cos=cos, rope_sin=sin, W_ik=a["W_ik"], ws=self.ws)

    def run_layer(self, i):
        self.run_index(i)
        self.run_attn(i)

    def run_index(self, i):
        """The index step of layer i (nothing for a Reuse layer)."""
        L = self.layers[i]
        mode = L["mode"]
        if mode == FULL:
            csa2.index_full(self.cache, L["q_idx"], L["w"], self.seq_of, self.n_vis, self.max_n, self.NB,
                            self.P, self.k, out=(self.pool, self.pool_len, self.topk[i], self.topk_len[i]),
                            ws=self.ws, group=self.group)
        elif mode == REINDEX:
            csa2.index_reindex(self.cache, L["q_idx"], L["w"], self.seq_of, self.pool, self.pool_len, self.k,
                               out=(self.topk[i], self.topk_len[i]), ws=self.ws)

    def run_attn(self, i, after_attn=None):
        """The sparse attention of layer i over its own (or the reused) index set.  A Reuse
        layer runs right after the previous layer's attention, which writes none of its
        inputs, so it may start reading them before that kernel completes (after_attn: whether
        the kernel just before on the stream is that attention; by default, for Reuse layers)."""
        L = self.layers[i]
        tk, tl = self.result_topk(i)
        if after_attn is None:
            after_attn = L["mode"] == REUSE and i > 0
        csa2.sparse_attn(self.cache, L["q"], self.seq_of, tk, tl, L["swa"], L["swa_scale"], L["swa_start"],
                         L["swa_len"], self.swa_max, out=self.out[i], lse=self.lse[i], ws=self.ws,
                         inputs_ready=after_attn)

    def _last_topk(self, i):
        for j in range(i - 1, -1, -1):
            if self.layers[j]["mode"] != REUSE:
                return self.topk[j], self.topk_len[j]
        raise ValueError("a Reuse layer needs an earlier Full or Reindex layer")

    def run(self):
        self.run_append()
        for i in range(len(self.layers)):
            self.run_layer(i)

    def result_topk(self, i):
        """Index set used by layer i (its own for Full/Reindex, the reused one otherwise)."""
        if self.layers[i]["mode"] == REUSE:
            return self._last_topk(i)
        return self.topk[i], self.topk_len[i]
