"""bench.py's recorded DRAM traffic (host logic, CPU): a figure from the
committed ncu summary is reported only while the source file of every kernel
it covers still hashes to the value recorded beside it, and the summary holds
a figure for every kernel and workload the default bench line reports."""
import hashlib
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

CSRC = os.path.join("gated_deltanet_verification_gb300", "csrc")


def _tree(tmp_path, records):
    """A minimal copy of the repository layout recorded_traffic reads."""
    os.makedirs(tmp_path / CSRC)
    os.makedirs(tmp_path / "profiles")
    for f in ("tc_verify.cu", "tc_big.cu"):
        (tmp_path / CSRC / f).write_bytes(f"// {f}\n".encode())
    shas = {f: hashlib.sha256((tmp_path / CSRC / f).read_bytes()).hexdigest()
            for f in ("tc_verify.cu", "tc_big.cu")}
    lines = ["# comment"] + [f"source {f} {s}" for f, s in shas.items()] + records
    (tmp_path / "profiles" / "traffic.txt").write_text("\n".join(lines) + "\n")


def test_recorded_traffic_follows_the_source_hash(tmp_path, monkeypatch):
    _tree(tmp_path, ["tc_verify_kernel 3 1000", "tc_commit_kernel 3 500",
                     "tc_big_fused_kernel 4chain 700", "tc_commit_kernel 4chain 300"])
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.recorded_traffic(["tc_verify_kernel", "tc_commit_kernel"], "3") == 1500
    assert bench.recorded_traffic(["tc_big_fused_kernel", "tc_commit_kernel"], "4chain") == 1000
    assert bench.recorded_traffic(["tc_verify_kernel"], "2") is None      # no capture
    assert bench.recorded_traffic([], "3") is None
    # an edit to one source voids every figure of the kernels it holds
    with open(tmp_path / CSRC / "tc_verify.cu", "a") as fh:
        fh.write("// edited\n")
    assert bench.recorded_traffic(["tc_verify_kernel"], "3") is None
    assert bench.recorded_traffic(["tc_big_fused_kernel", "tc_commit_kernel"], "4chain") is None
    assert bench.recorded_traffic(["tc_big_fused_kernel"], "4chain") == 700


def test_workload_keys():
    assert bench.workload_key(3, "chain") == "3"
    assert bench.workload_key(4, "4ary") == "44ary"
    assert bench.workload_key(2, "chain", "f32") == "2f32"
    assert bench.workload_key(0, "chain", "f32") == "0"


def test_committed_summary_covers_the_bench_lines():
    """Every (kernel, workload) the bench reports a dominant-kernel traffic
    for has a record in the committed summary, and every kernel's source file
    is named there."""
    lines = [ln.split() for ln in open(os.path.join(ROOT, "profiles", "traffic.txt"))
             if ln.strip() and not ln.startswith("#")]
    sources = {ln[1] for ln in lines if ln[0] == "source"}
    assert set(bench.KERNEL_SOURCES.values()) <= sources
    have = {(ln[0], ln[1]) for ln in lines if ln[0] != "source"}
    for wl in ("3", "2", "1"):
        assert ("tc_commit_verify", wl) in have
    for wl in ("3", "2"):
        assert ("tc_verify_kernel", wl) in have and ("tc_commit_kernel", wl) in have
    for sh in ("chain", "star", "4ary"):
        assert ("tc_big_fused_kernel", "4" + sh) in have and ("tc_commit_kernel", "4" + sh) in have
