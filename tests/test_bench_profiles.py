"""bench.py's `traffic` figures come from the committed ncu summaries: every summary the bench
maps a (kernel, workload) to must exist, carry the fields the bench reads, and state a traffic
close to its algorithmic bytes (a summary whose DRAM bytes were far above them would flag
re-reads).  The per-launch figure is reported only while the kernel's source still has the
summary's hash, which this test checks the bench does.  No GPU is involved."""
import hashlib
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _fields(path):
    out = {}
    for ln in open(path):
        if ":" in ln:
            k, v = ln.split(":", 1)
            out[k.strip()] = v.strip()
    return out


@pytest.mark.parametrize("key", sorted(bench.PROFILES))
def test_profile_summary_is_complete(key):
    name, src = bench.PROFILES[key]
    path = os.path.join(ROOT, "profiles", name)
    assert os.path.exists(path), path
    f = _fields(path)
    traffic = int(f["dram_bytes_per_launch"])
    alg = int(f["algorithmic_bytes_per_launch"])
    assert 0.9 * alg <= traffic <= 1.1 * alg, (name, traffic, alg)
    assert f"source_sha1 ({src})" in f
    assert os.path.exists(os.path.join(ROOT, "fp4_compressed_sparse_02_gb300", "csrc", src))
    text = open(path).read()
    assert "--clock-control none" in text and "ncu " in text       # the command that made it


def test_traffic_is_reported_only_for_the_captured_source(tmp_path, monkeypatch):
    kernel, workload = ("k_full_scan", "decode1m")
    name, src = bench.PROFILES[(kernel, workload)]
    real = open(os.path.join(ROOT, "profiles", name)).read()
    sha = hashlib.sha1(open(os.path.join(ROOT, "fp4_compressed_sparse_02_gb300", "csrc", src), "rb").read()).hexdigest()
    root = tmp_path / "repo"
    (root / "profiles").mkdir(parents=True)
    (root / "fp4_compressed_sparse_02_gb300" / "csrc").mkdir(parents=True)
    (root / "fp4_compressed_sparse_02_gb300" / "csrc" / src).write_bytes(
        open(os.path.join(ROOT, "fp4_compressed_sparse_02_gb300", "csrc", src), "rb").read())
    monkeypatch.setattr(bench, "ROOT", str(root))
    # a summary whose hash matches the source: its figure is reported
    (root / "profiles" / name).write_text(real.replace(
        [ln for ln in real.splitlines() if ln.startswith(f"source_sha1 ({src})")][0], f"source_sha1 ({src}): {sha}"))
    assert bench.profiled_traffic(kernel, workload) == int(_fields(root / "profiles" / name)["dram_bytes_per_launch"])
    # the source changed since the capture: nothing is reported
    (root / "fp4_compressed_sparse_02_gb300" / "csrc" / src).write_bytes(b"// changed\n")
    assert bench.profiled_traffic(kernel, workload) is None
    # no summary for this kernel and workload
    assert bench.profiled_traffic("k_attn_tc", "no_such_workload") is None
