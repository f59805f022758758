"""The DRAM-traffic records bench.py reports as roofline.traffic (CPU only):
a record counts only while the kernel's source and every local header it
includes are unchanged since the capture."""
import os
import shutil

import bench


def _copy_tree(tmp_path):
    root = tmp_path / "repo"
    shutil.copytree(os.path.join(bench.ROOT, "block_sparse_paged_score_gb300", "csrc"),
                    root / "block_sparse_paged_score_gb300" / "csrc")
    shutil.copytree(os.path.join(bench.ROOT, "include"), root / "include")
    shutil.copytree(os.path.join(bench.ROOT, "profiles"), root / "profiles")
    return root


def test_include_closure_reaches_nested_headers():
    srcs = bench.kernel_sources(["index_score.cu"])
    names = {os.path.basename(f) for f in srcs}
    # directly included, included through another header, and the ABI header
    assert {"index_score.cu", "common.cuh", "kernels.h", "topk_row.cuh", "bsp.h"} <= names
    assert "sparse_pa.cu" not in names


def test_record_follows_every_header(tmp_path, monkeypatch):
    root = _copy_tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(root))
    h = bench.kernel_source_hash(["index_score.cu"])
    (root / "profiles" / "dram_traffic.txt").write_text(f"index_score_kernel wl {h} 123\n")
    assert bench.recorded_traffic("index_score_kernel", "wl", ["index_score.cu"]) == 123.0
    assert bench.recorded_traffic("index_score_kernel", "other-wl", ["index_score.cu"]) is None
    assert bench.recorded_traffic("sparse_pa_kernel", "wl", ["sparse_pa.cu"]) is None
    # a header two includes deep changes: the record no longer counts
    hdr = root / "block_sparse_paged_score_gb300" / "csrc" / "topk_row.cuh"
    hdr.write_text(hdr.read_text() + "\n// changed\n")
    assert bench.kernel_source_hash(["index_score.cu"]) != h
    assert bench.recorded_traffic("index_score_kernel", "wl", ["index_score.cu"]) is None


def test_committed_records_name_known_kernels():
    kernels = {"index_score_kernel": "index_score.cu", "sparse_pa_kernel": "sparse_pa.cu",
               "index_score_mx_tc_kernel": "index_score_mx_tc.cu"}
    for line in open(os.path.join(bench.ROOT, "profiles", "dram_traffic.txt")):
        if line.startswith("#") or not line.strip():
            continue
        k, wl, h, nbytes = line.split()
        assert k in kernels and len(h) == 16 and float(nbytes) > 0
