"""The benchmark's host-side bookkeeping on CPU: workload shapes, the algorithmic bytes
the grouped rooflines divide by, and the traffic records' source-hash gate."""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_grouped_workloads_share_shapes():
    fp8, bf16 = bench.workload_spec("grouped_fp8"), bench.workload_spec("grouped_bf16")
    assert len(fp8) == len(bf16) == 9
    for a, b in zip(fp8, bf16):
        assert (a["T"], a["N"], a["K"], a["case"]) == (b["T"], b["N"], b["K"], b["case"])
        assert a["kind"] == "grouped" and b["kind"] == "grouped_bf16"
    assert {(g["T"], g["N"], g["K"]) for g in bf16} == {
        (t, n, k) for t in (128, 1024, 16384) for (n, k) in ((2048, 7168), (7168, 2304), (16384, 6656))}


def test_grouped_algorithmic_bytes():
    ms = np.array([5, 0, 3, 0], dtype=np.int64)            # two live groups of four
    g8 = dict(kind="grouped", T=8, N=256, K=384)
    g16 = dict(kind="grouped_bf16", T=8, N=256, K=384)
    # FP8: W codes + FP32 128x128 scales of the live groups, X codes + FP32 1x128 scales,
    # BF16 D, int64 m_sizes
    assert bench.grouped_bytes(g8, ms) == (2 * (256 * 384 + 4 * 2 * 3) + 8 * 384 + 4 * 8 * 3
                                           + 2 * 8 * 256 + 8 * 4)
    # BF16: two bytes per X and W element, no scales
    assert bench.grouped_bytes(g16, ms) == 2 * 256 * 384 * 2 + 8 * 384 * 2 + 2 * 8 * 256 + 8 * 4


def test_flops_and_descriptions():
    g = dict(kind="grouped_bf16", T=128, N=2048, K=7168)
    assert bench.flops_of(g) == 2.0 * 128 * 2048 * 7168
    assert bench.describe(g) == "grouped_bf16 G=8 totM=128 N=2048 K=7168"


def test_traffic_record_requires_matching_sources(tmp_path, monkeypatch):
    """A traffic record counts only while its hash matches the kernel sources."""
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "traffic_grouped_bf16.txt").write_text(
        "kernel_sources_sha256_16: 0000000000000000\ndram_bytes_per_launch: 123\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda w: "0000000000000000")
    assert bench.recorded_traffic("grouped_bf16") == 123.0
    monkeypatch.setattr(bench, "kernel_source_hash", lambda w: "ffffffffffffffff")
    assert bench.recorded_traffic("grouped_bf16") is None


def test_source_hash_ignores_comments_only():
    code = "int f(int x) {  // doubles\n  return 2 * x; /* no overflow check */\n}\n"
    same = "// a comment line added\nint f(int x) {\n  return 2 * x;\n}\n"
    other = "int f(int x) {\n  return 3 * x;\n}\n"
    assert bench._code_only(code) == bench._code_only(same)
    assert bench._code_only(code) != bench._code_only(other)


def test_kernel_sources_cover_their_includes():
    """Every header that a hashed kernel source includes from the library's own sources is
    hashed too, so a change anywhere in a kernel's code invalidates its traffic record."""
    import re
    csrc = os.path.join(ROOT, "block_scaled_precision_mma_gb300", "csrc")
    local = set(os.listdir(csrc))
    for workload, files in bench.KERNEL_SOURCES.items():
        todo, seen = list(files), set()
        while todo:
            f = todo.pop()
            if f in seen:
                continue
            seen.add(f)
            with open(os.path.join(csrc, f), encoding="utf-8") as fh:
                todo += [h for h in re.findall(r'#include "([^"]+)"', fh.read()) if h in local]
        assert seen <= set(files), (workload, sorted(seen - set(files)))
