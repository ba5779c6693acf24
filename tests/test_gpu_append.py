"""GPU parity of csa2_compress_append, the decode-time cache append: every call brings one
new token of each sequence; at m > 1 a token that does not complete its group waits in the
caller's pending buffer, and the completing token writes the group's entry.  Compared with
the oracle's token-by-token append (which pins to compressing the whole sequence at once)."""
import math

import numpy as np
import pytest
import torch

from fp4_compressed_sparse_02_gb300 import csa2, synth
from oracle import compress, formats
from parity_utils import bf16_dev, bf16_host_bits, check_index_k, fp4_mismatch_is_tolerated, to_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("m,h_dtype,B,d_model", [(2, "bf16", 6, 5120), (4, "bf16", 3, 512), (2, "f32", 5, 1024),
                                                 (1, "bf16", 4, 512), (2, "bf16", 80, 512)])
def test_append_token_by_token(m, h_dtype, B, d_model):
    r = np.random.default_rng(1100 + 10 * m + B)
    d, d_ik, d_rope = 512, 128, 64
    T = 2 * m + 1                                   # the last group stays incomplete
    if h_dtype == "bf16":
        Hb = synth.bf16_normal(r, (T, B, d_model))
        H_host = formats.bf16_value(Hb)
        H_dev = [bf16_dev(Hb[t]) for t in range(T)]
    else:
        H_host = synth.f32_normal(r, (T, B, d_model)).astype(np.float64)
        H_dev = [to_dev(H_host[t].astype(np.float32)) for t in range(T)]
    Wkv = synth.bf16_normal(r, (d_model, d), 1 / math.sqrt(d_model))
    Wz = synth.bf16_normal(r, (d_model, d), 1 / math.sqrt(d_model))
    Wik = synth.bf16_normal(r, (d, d_ik), 1 / math.sqrt(d))
    Wkv_h, Wz_h, Wik_h = (formats.bf16_value(w) for w in (Wkv, Wz, Wik))
    cos, sin = synth.rope_tables(64, d_rope)
    G = T // m + 1
    pt = synth.page_table(r, B, 1)
    cache = csa2.PagedCache.allocate(B, G, d, d_ik, "cuda", torch.from_numpy(pt))
    cache.codes.fill_(0xEE)
    cache.scales.fill_(0xEE)
    pend = torch.full((B, 2, m, d), float("nan"), dtype=torch.float32, device="cuda") if m > 1 else None
    seq = to_dev(np.arange(B, dtype=np.int32))
    pending = [[] for _ in range(B)]
    want = {}                                       # (b, g) -> oracle entry
    ys = {}                                         # (b, g) -> the GPU's pre-quantisation row
    for t in range(T):
        y = torch.full((B, d), float("nan"), dtype=torch.float32, device="cuda")
        csa2.compress_append(cache, H_dev[t], seq, to_dev(np.full(B, t, np.int32)), bf16_dev(Wkv), m=m,
                             W_z=bf16_dev(Wz) if m > 1 else None, pend=pend, rope_cos=to_dev(cos), rope_sin=to_dev(sin),
                             W_ik=bf16_dev(Wik), y_out=y)
        assert csa2.device_error() == 0
        yg = y.cpu().numpy()
        done = t % m == m - 1
        assert np.isnan(yg).all() != done             # rows only for tokens that complete a group
        for b in range(B):
            res = compress.append_token(pending[b], H_host[t, b], t, Wkv_h, Wz_h, m, cos, sin, d_rope, Wik_h)
            if res is not None:
                want[b, res[0]] = res[1]
                ys[b, res[0]] = yg[b]
        codes = cache.codes.cpu().numpy()[pt[:, 0]]
        # the group still waiting has no entry yet
        g_open = t // m if not done else None
        if g_open is not None:
            assert (codes[:, g_open] == 0xEE).all()
    codes = cache.codes.cpu().numpy()[pt[:, 0]]
    scales = cache.scales.cpu().numpy()[pt[:, 0]]
    ik = bf16_host_bits(cache.idx_k)[pt[:, 0]]
    assert len(want) == B * (T // m)
    yg = np.stack([ys[key] for key in sorted(want)])
    yo = np.stack([want[key]["y"][0] for key in sorted(want)])
    cg = np.stack([codes[b, g] for b, g in sorted(want)])
    sg = np.stack([scales[b, g] for b, g in sorted(want)])
    co = np.stack([want[key]["codes"][0] for key in sorted(want)])
    so = np.stack([want[key]["scales"][0] for key in sorted(want)])
    err = np.abs(yg.astype(np.float64) - yo)
    assert err.max() <= 1e-5 * np.abs(yo).max(), err.max()
    c_own, s_own = formats.fp4_quantize(yg)                 # the quantiser rule on the GPU's own rows
    np.testing.assert_array_equal(sg, s_own)
    np.testing.assert_array_equal(cg, c_own)
    bad, tol = fp4_mismatch_is_tolerated(yo, cg, sg, co, so, err)
    assert bad == tol
    same = (cg == co).all(1) & (sg == so).all(1)
    ikg = np.stack([ik[b, g] for b, g in sorted(want)])
    iko = np.stack([want[key]["idx_k"][0] for key in sorted(want)])
    check_index_k(ikg[same], iko[same], co[same], so[same], Wik)
    assert (codes[:, T // m] == 0xEE).all()                  # the last, incomplete group: no entry


def test_append_flags_bad_sequence_and_position():
    r = np.random.default_rng(1200)
    B, d_model, d = 3, 256, 128
    H = synth.bf16_normal(r, (B, d_model))
    Wkv = synth.bf16_normal(r, (d_model, d), 1 / 16)
    pt = synth.page_table(r, 2, 1)
    cache = csa2.PagedCache.allocate(2, 64, d, 0, "cuda", torch.from_numpy(pt))
    cache.codes.fill_(0xEE)
    csa2.compress_append(cache, bf16_dev(H), to_dev(np.array([0, 5, 1], np.int32)), to_dev(np.array([3, 0, -2], np.int32)),
                         bf16_dev(Wkv))
    err = csa2.device_error()
    assert err & 0x10 and err & 0x40                           # sequence 5 does not exist; position -2
    codes = cache.codes.cpu().numpy()
    assert (codes[pt[0, 0], 3] != 0xEE).any()                  # the valid token was written
    assert (codes[pt[1, 0]] == 0xEE).all()                     # the token at position -2 was not
