"""The algorithmic bytes behind every achieved-bandwidth figure, pinned to the per-unit sums
written out from the layouts (d = 512, d_ik = 128, H_i = 8, Hq = 64, k = 512, W = 128, pool
2,048 x 8)."""
from fp4_compressed_sparse_02_gb300 import workload
from fp4_compressed_sparse_02_gb300.schedule import decoder_schedule


def _info(**kw):
    info = dict(B=32, G=1, seqs=32, N=131072, layers=20, schedule=decoder_schedule(), d=512, d_ik=128, H_i=8,
                Hq=64, W=128, k=512, NB=2048, P=8, d_model=5120)
    info.update(kw)
    return info


def test_per_query_units():
    q = workload.algorithmic_bytes(_info())["per_query"]
    # indexer K of every visible entry + q_idx + w + pool ids + top-k ids
    assert q["full"] == 131072 * 256 + 8 * 128 * 2 + 8 * 4 + 16384 * 4 + 512 * 4 == 33_624_096
    # the pool's gathered indexer-K rows + pool ids + q_idx + w + top-k ids
    assert q["reindex"] == 16384 * 256 + 16384 * 4 + 8 * 128 * 2 + 8 * 4 + 512 * 4 == 4_263_968
    # FP4 rows (codes + scales) + FP8 window rows with their scales + Q and out (bf16) + ids
    assert q["attn"] == 512 * (256 + 32) + 128 * (512 + 4) + 2 * 64 * 512 * 2 + 512 * 4 == 346_624


def test_step_total_sums_the_schedule():
    info = _info(B=2, seqs=2)
    nb = workload.algorithmic_bytes(info)
    q = nb["per_query"]
    # decoder schedule: 1 Full, 4 Reindex, 20 attention layers per query, plus the append
    assert nb["total"] == 2 * (q["full"] + 4 * q["reindex"] + 20 * q["attn"]) + nb["append"]
    assert nb["append"] == 2 * (5120 * 2 + 256 + 32 + 2 * 128) + 5120 * 512 * 2 + 512 * 128 * 2


def test_short_contexts_and_verification_groups():
    # a context shorter than the pool: the pool is the whole range; a group of G queries reads
    # its sequence's indexer K once
    short = workload.algorithmic_bytes(_info(N=4096, Ns=[4096]))["per_query"]
    assert short["reindex"] == 4096 * 256 + 16384 * 4 + 8 * 128 * 2 + 8 * 4 + 512 * 4
    g6 = workload.algorithmic_bytes(_info(B=12, G=6, seqs=2, Ns=[131072, 131072]))
    one = workload.algorithmic_bytes(_info(B=2, seqs=2, Ns=[131072, 131072]))
    scan = 131072 * 256
    assert g6["per_query"]["full"] == scan // 6 + 8 * 128 * 2 + 8 * 4 + 16384 * 4 + 512 * 4
    # (each of the 6 queries counts a sixth of the scan, rounded down)
    assert g6["total"] - g6["append"] == 6 * (one["total"] - one["append"]) - 2 * 6 * scan + 2 * 6 * (scan // 6)
