"""GPU parity of csa2_sparse_attn against the oracle attention, on identical FP4 caches,
SWA rows and index sets (drawn by the input generator)."""
import numpy as np
import pytest
import torch

from fp4_compressed_sparse_02_gb300 import csa2, synth
from oracle import attention, formats
from parity_utils import ATTN_MAX_ABS, ATTN_REL_L2, bf16_dev, logical_to_paged, rel_l2, to_dev

pytestmark = pytest.mark.gpu


def _case(r, B, Hq, d, k, W, n, ns=2, fill=0.9):
    mp = (n + 63) // 64
    pt = synth.page_table(r, ns, mp)
    codes = [synth.fp4_codes(r, (n,), d) for _ in range(ns)]
    scales = [synth.fp4_scales(r, (n,), d) for _ in range(ns)]
    cache = csa2.PagedCache.allocate(ns, n, d, 0, "cuda", torch.from_numpy(pt))
    cache.codes.copy_(to_dev(logical_to_paged(codes, pt, ns * mp, d // 2, np.uint8)))
    cache.scales.copy_(to_dev(logical_to_paged(scales, pt, ns * mp, d // 16, np.uint8)))
    seq_of = (np.arange(B) % ns).astype(np.int32)
    topk = np.full((B, k), -1, dtype=np.int32)
    tlen = np.zeros(B, dtype=np.int32)
    for b in range(B):
        cnt = min(n, max(0, int(k * fill) if b % 3 else k))
        sel = synth.sorted_distinct(r, n, cnt)
        topk[b, :len(sel)] = sel
        tlen[b] = len(sel)
    rows = B * W + 7
    swa = synth.fp8_rows(r, rows, d)
    swa_scale = synth.fp8_row_scales(r, rows)
    swa_start = (np.arange(B) * W + 3).astype(np.int32)
    swa_len = np.full(B, W, dtype=np.int32)
    q = synth.bf16_normal(r, (B, Hq, d))
    return dict(cache=cache, codes=codes, scales=scales, seq_of=seq_of, topk=topk, tlen=tlen, swa=swa,
                swa_scale=swa_scale, swa_start=swa_start, swa_len=swa_len, q=q, W=W)


def _run(c, out_dtype=torch.float32, use_tlen=True):
    out, lse = csa2.sparse_attn(c["cache"], bf16_dev(c["q"]), to_dev(c["seq_of"]), to_dev(c["topk"]),
                                to_dev(c["tlen"]) if use_tlen else None, to_dev(c["swa"]), to_dev(c["swa_scale"]),
                                to_dev(c["swa_start"]), to_dev(c["swa_len"]), c["W"], out_dtype=out_dtype)
    assert csa2.device_error() == 0
    return out.float().cpu().numpy(), lse.cpu().numpy()


def _oracle(c):
    B, Hq, d = c["q"].shape
    outs, lses = [], []
    for b in range(B):
        s = c["seq_of"][b]
        o, l = attention.sparse_attention(formats.bf16_value(c["q"][b]), c["codes"][s], c["scales"][s],
                                          c["topk"][b, :c["tlen"][b]], c["swa"], c["swa_scale"],
                                          int(c["swa_start"][b]), int(c["swa_len"][b]), 1 / np.sqrt(d))
        outs.append(o)
        lses.append(l)
    return np.stack(outs), np.stack(lses)


def _assert_close(got, ref):
    assert rel_l2(got, ref) <= ATTN_REL_L2, rel_l2(got, ref)
    assert np.abs(got - ref).max() <= ATTN_MAX_ABS


@pytest.mark.parametrize("B,Hq,d,k,W", [(5, 64, 512, 512, 128), (7, 8, 128, 64, 32), (3, 16, 512, 256, 64),
                                        (4, 32, 128, 200, 100), (2, 64, 128, 512, 128)])
def test_attn_parity(B, Hq, d, k, W):
    r = np.random.default_rng(B * 1000 + Hq + d + k + W)
    c = _case(r, B, Hq, d, k, W, n=3000)
    out, lse = _run(c)
    ref, rlse = _oracle(c)
    _assert_close(out, ref)
    np.testing.assert_allclose(lse, rlse, rtol=1e-4, atol=1e-4)


def _offset16(t):
    """A copy of t whose data starts 16 bytes past a 256-byte boundary (16-byte aligned,
    not 32-byte aligned)."""
    n = t.numel() * t.element_size()
    buf = torch.zeros(n + 256, dtype=torch.uint8, device=t.device)
    v = buf[16:16 + n].view(t.dtype).view(t.shape)
    v.copy_(t)
    assert v.data_ptr() % 32 == 16
    return v


def test_attn_many_queries():
    # many more queries than one wave of clusters: against the oracle, and bit for bit
    # against the same queries in batches of one wave; some queries have no selected slot,
    # no window row, or neither.
    r = np.random.default_rng(4242)
    B = 640
    c = _case(r, B, 64, 512, 512, 128, n=3000)
    c["tlen"][5] = 0
    c["topk"][5] = -1
    c["swa_len"][5] = 0
    c["tlen"][6] = 0
    c["topk"][6] = -1
    c["swa_len"][7] = 0
    c["swa_len"][8] = 77
    got, lse = _run(c)
    ref, rlse = _oracle(c)
    _assert_close(got, ref)
    fin = np.isfinite(rlse)
    np.testing.assert_allclose(lse[fin], rlse[fin], rtol=1e-4, atol=1e-4)
    assert (~np.isfinite(lse[~fin])).all() and (got[5] == 0).all()
    for lo in range(0, B, 30):
        hi = min(B, lo + 30)
        part = {key: (v[lo:hi] if isinstance(v, np.ndarray) and v.ndim >= 1 and v.shape[0] == B else v)
                for key, v in c.items()}
        g2, l2 = _run(part)
        np.testing.assert_array_equal(g2, got[lo:hi])
        np.testing.assert_array_equal(l2, lse[lo:hi])


def test_attn_16_byte_aligned_arrays():
    # codes and window rows that are only 16-byte aligned take the 16-byte gather loads
    r = np.random.default_rng(77)
    c = _case(r, 5, 64, 512, 512, 128, n=3000)
    ref, rlse = _oracle(c)
    cache = c["cache"]
    c["cache"] = csa2.PagedCache(_offset16(cache.codes), cache.scales, cache.idx_k, cache.page_table)
    swa = _offset16(to_dev(c["swa"]))
    out, lse = csa2.sparse_attn(c["cache"], bf16_dev(c["q"]), to_dev(c["seq_of"]), to_dev(c["topk"]),
                                to_dev(c["tlen"]), swa, to_dev(c["swa_scale"]), to_dev(c["swa_start"]),
                                to_dev(c["swa_len"]), c["W"], out_dtype=torch.float32)
    assert csa2.device_error() == 0
    _assert_close(out.cpu().numpy(), ref)
    np.testing.assert_allclose(lse.cpu().numpy(), rlse, rtol=1e-4, atol=1e-4)


def test_attn_bf16_output_and_determinism():
    r = np.random.default_rng(50)
    c = _case(r, 4, 64, 512, 512, 128, n=5000)
    o1, _ = _run(c, torch.bfloat16)
    o2, _ = _run(c, torch.bfloat16)
    np.testing.assert_array_equal(o1, o2)          # Reuse = the same call again: identical
    ref, _ = _oracle(c)
    # bf16 output: add the output rounding, half a bf16 ulp (2^-9 relative), on top
    assert rel_l2(o1, ref) <= ATTN_REL_L2 + 2.0 ** -9
    assert (np.abs(o1 - ref) <= ATTN_MAX_ABS + 2.0 ** -8 * np.abs(ref)).all()


def test_attn_empty_and_one_sided():
    r = np.random.default_rng(51)
    c = _case(r, 4, 64, 512, 512, 128, n=2000)
    c["tlen"][0] = 0
    c["swa_len"][0] = 0            # nothing to attend: out 0, lse -inf
    c["tlen"][1] = 0               # window only
    c["swa_len"][2] = 0            # selection only
    c["topk"][3, ::3] = -1         # holes inside the valid prefix are skipped
    out, lse = _run(c)
    ref, rlse = _oracle(c)
    assert (out[0] == 0).all() and np.isneginf(lse[0]).all()
    _assert_close(out[1:], ref[1:])
    np.testing.assert_allclose(lse[1:], rlse[1:], rtol=1e-4, atol=1e-4)


def test_attn_window_only_layer():
    # an SWA-only layer (the encoder's first two layers): k = 0, no selection at all
    r = np.random.default_rng(52)
    c = _case(r, 6, 64, 512, 0, 128, n=500)
    empty = torch.empty((6, 0), dtype=torch.int32, device="cuda")
    out, lse = csa2.sparse_attn(c["cache"], bf16_dev(c["q"]), to_dev(c["seq_of"]), empty, None, to_dev(c["swa"]),
                                to_dev(c["swa_scale"]), to_dev(c["swa_start"]), to_dev(c["swa_len"]), c["W"],
                                out_dtype=torch.float32)
    assert csa2.device_error() == 0
    ref, rlse = _oracle(c)
    _assert_close(out.cpu().numpy(), ref)
    np.testing.assert_allclose(lse.cpu().numpy(), rlse, rtol=1e-4, atol=1e-4)


def test_attn_without_topk_len_reads_all_slots():
    r = np.random.default_rng(52)
    c = _case(r, 3, 64, 512, 512, 128, n=4000, fill=0.5)
    out, _ = _run(c, use_tlen=False)
    ref, _ = _oracle(c)
    _assert_close(out, ref)


def test_attn_single_key_returns_its_row():
    r = np.random.default_rng(53)
    c = _case(r, 2, 64, 512, 512, 128, n=1000)
    c["topk"][:] = -1
    c["topk"][:, 0] = [17, 900]
    c["tlen"][:] = 1
    c["swa_len"][:] = 0
    out, lse = _run(c)
    for b in range(2):
        row = formats.fp4_dequantize(c["codes"][c["seq_of"][b]][c["topk"][b, 0]],
                                     c["scales"][c["seq_of"][b]][c["topk"][b, 0]])
        np.testing.assert_allclose(out[b], np.tile(row, (64, 1)), rtol=1e-6, atol=1e-6)


def test_swa_window_outside_rows_is_flagged():
    r = np.random.default_rng(54)
    c = _case(r, 2, 8, 128, 64, 32, n=500)
    c["swa_start"][1] = c["swa"].shape[0] - 5       # window runs past the last row
    _run_noerr = csa2.sparse_attn(c["cache"], bf16_dev(c["q"]), to_dev(c["seq_of"]), to_dev(c["topk"]),
                                  to_dev(c["tlen"]), to_dev(c["swa"]), to_dev(c["swa_scale"]),
                                  to_dev(c["swa_start"]), to_dev(c["swa_len"]), c["W"])
    assert csa2.device_error() & 0x20


def test_bounded_wait_times_out_reports_and_context_survives():
    # a wait that nothing satisfies gives up, sets the timeout bit and returns
    csa2.selftest_wait_timeout(1000)
    import ctypes
    from fp4_compressed_sparse_02_gb300 import _lib
    word = ctypes.c_uint32(0)
    assert _lib.lib().csa2_get_device_error(ctypes.byref(word)) == 6      # CSA2_ERR_TIMEOUT
    assert word.value & 0x80
    assert csa2.device_error() == 0                 # the word was cleared by the read
    # the context is still usable: a normal call right after runs and agrees
    r = np.random.default_rng(55)
    c = _case(r, 3, 64, 512, 512, 128, n=2000)
    out, _ = _run(c)
    ref, _ = _oracle(c)
    _assert_close(out, ref)


# ---- the whole input range ------------------------------------------------------------
# The default generator keeps every input in a moderate range.  These cases sweep what the
# formats allow: every finite E4M3 byte in the window rows (subnormals and 128..448 among
# them), row scales from 2^-24 to 2^7, every FP4 scale byte 0x00..0x7E (0 included) and bf16
# Q whose magnitudes span 2^-30..2^15 (and a query far beyond the fp16 range).  The outputs
# then span many orders of magnitude, so the comparison is per query head: relative L2
# <= 2e-3, and max-abs <= 1e-2 x max(1, max |o_ref|) of that head (the 1e-2 is an absolute
# bound for outputs of unit scale, relative above it).

_E4M3_FINITE = np.array([v for v in range(256) if (v & 0x7F) != 0x7F], dtype=np.uint8)


def _assert_close_per_head(got, ref, what=""):
    B, H, _ = ref.shape
    for b in range(B):
        for h in range(H):
            g, o = got[b, h].astype(np.float64), ref[b, h]
            no = np.linalg.norm(o)
            if no == 0:
                assert not g.any(), f"{what} b={b} h={h}: expected zeros"
                continue
            e = np.linalg.norm(g - o) / no
            assert e <= ATTN_REL_L2, f"{what} b={b} h={h}: rel-L2 {e:.3g} (|o| ~ {np.abs(o).max():.3g})"
            assert np.abs(g - o).max() <= ATTN_MAX_ABS * max(1.0, np.abs(o).max()), f"{what} b={b} h={h}: max-abs"


def _lse_close(lse, rlse):
    fin = np.isfinite(rlse)
    np.testing.assert_allclose(lse[fin], rlse[fin], rtol=1e-4, atol=1e-4)
    assert np.isneginf(lse[~fin]).all()


def _q_log_uniform(r, shape, lo, hi):
    """bf16 values with random signs and magnitudes 2^u, u uniform in [lo, hi]."""
    mag = np.exp2(r.uniform(lo, hi, size=shape))
    sgn = np.where(r.random(shape) < 0.5, -1.0, 1.0)
    return synth.bf16_bits_from_f32((sgn * mag).astype(np.float32))


SHAPES = [(5, 64, 512, 512, 128), (6, 8, 128, 64, 32)]   # tensor-core kernel; general-shape kernel


@pytest.mark.parametrize("B,Hq,d,k,W", SHAPES)
def test_attn_window_rows_full_range(B, Hq, d, k, W):
    r = np.random.default_rng(600 + d)
    c = _case(r, B, Hq, d, k, W, n=3000)
    rows = c["swa"].shape[0]
    c["swa"] = r.choice(_E4M3_FINITE, size=(rows, d))
    c["swa_scale"] = np.exp2(r.uniform(-24, 7, size=rows)).astype(np.float32)
    # queries 1 and 3 attend to their window only; query 3's window is quiet (every row
    # scale in 2^-24 .. 2^-20), query 4's the loudest the range allows (2^6 .. 2^7)
    for b in (1, 3):
        c["tlen"][b] = 0
        c["topk"][b] = -1
    s3, s4 = int(c["swa_start"][3]), int(c["swa_start"][4])
    c["swa_scale"][s3:s3 + W] = np.exp2(r.uniform(-24, -20, size=W))
    c["swa_scale"][s4:s4 + W] = np.exp2(r.uniform(6, 7, size=W))
    out, lse = _run(c)
    ref, rlse = _oracle(c)
    _assert_close_per_head(out, ref, "window rows")
    _lse_close(lse, rlse)


@pytest.mark.parametrize("B,Hq,d,k,W", SHAPES)
def test_attn_fp4_scale_bytes_full_range(B, Hq, d, k, W):
    r = np.random.default_rng(700 + d)
    c = _case(r, B, Hq, d, k, W, n=3000)
    for s in range(len(c["scales"])):
        c["scales"][s] = r.integers(0, 0x7F, size=c["scales"][s].shape, dtype=np.uint8)   # 0x00..0x7E
        c["scales"][s][::7] = 0                                                          # all-zero groups
    # sequence 1's entries are all tiny (scale bytes 0x00..0x08: scales 0 .. 2^-6); its
    # queries 1 and 3 see no window
    c["scales"][1] = r.integers(0, 9, size=c["scales"][1].shape, dtype=np.uint8)
    c["swa_len"][1] = 0
    c["swa_len"][3] = 0
    pt = c["cache"].page_table.cpu().numpy()
    c["cache"].scales.copy_(to_dev(logical_to_paged(c["scales"], pt, c["cache"].num_pages, d // 16, np.uint8)))
    out, lse = _run(c)
    ref, rlse = _oracle(c)
    _assert_close_per_head(out, ref, "FP4 scales")
    _lse_close(lse, rlse)


@pytest.mark.parametrize("B,Hq,d,k,W", SHAPES)
def test_attn_q_full_range(B, Hq, d, k, W):
    r = np.random.default_rng(800 + d)
    c = _case(r, B, Hq, d, k, W, n=3000)
    # query 0: every element's magnitude log-uniform in 2^-30 .. 2^15; query 1: each head
    # scaled as a whole by 2^e, e uniform in -30 .. 15; query 2: tiny heads only
    # (2^-30 .. 2^-20); query 3: beyond the fp16 range (2^16 .. 2^40)
    c["q"][0] = _q_log_uniform(r, (Hq, d), -30, 15)
    base = formats.bf16_value(synth.bf16_normal(r, (Hq, d)))
    e = r.uniform(-30, 15, size=(Hq, 1))
    c["q"][1] = synth.bf16_bits_from_f32((base * np.exp2(np.floor(e))).astype(np.float32))
    c["q"][2] = _q_log_uniform(r, (Hq, d), -30, -20)
    c["q"][3] = _q_log_uniform(r, (Hq, d), 16, 40)
    out, lse = _run(c)
    ref, rlse = _oracle(c)
    _assert_close_per_head(out, ref, "Q range")
    _lse_close(lse, rlse)


@pytest.mark.parametrize("shape", [(40, 64, 512, 512, 128), (6, 8, 128, 64, 32)])
def test_attn_inputs_ready_matches_the_ordered_call(shape):
    # Reuse layers: calls after an attention call that writes none of their inputs start
    # before it completes; their results equal the ordinary calls' bit for bit, eagerly and
    # replayed from a CUDA graph, and their outputs are written after the previous call's
    B, Hq, d, k, W = shape
    r = np.random.default_rng(990 + d)
    c = _case(r, B, Hq, d, k, W, n=3000)
    args = [c["cache"], bf16_dev(c["q"]), to_dev(c["seq_of"]), to_dev(c["topk"]), to_dev(c["tlen"]),
            to_dev(c["swa"]), to_dev(c["swa_scale"]), to_dev(c["swa_start"]), to_dev(c["swa_len"]), W]
    ref, rlse = csa2.sparse_attn(*args, out_dtype=torch.float32)
    outs = [torch.full((B, Hq, d), float("nan"), device="cuda") for _ in range(3)]
    lses = [torch.empty((B, Hq), device="cuda") for _ in range(3)]
    ws = csa2.Workspace()

    def chain():
        for i in range(3):
            csa2.sparse_attn(*args, out_dtype=torch.float32, out=outs[i], lse=lses[i], ws=ws, inputs_ready=i > 0)

    chain()
    torch.cuda.synchronize()
    assert csa2.device_error() == 0
    for o, l in zip(outs, lses):
        assert torch.equal(o, ref) and torch.equal(l, rlse)
    g = torch.cuda.CUDAGraph()
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        chain()
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=st):
        chain()
    for o in outs:
        o.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    for o, l in zip(outs, lses):
        assert torch.equal(o, ref) and torch.equal(l, rlse)
