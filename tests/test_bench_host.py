"""bench.py's host-side bookkeeping, on CPU: the per-launch DRAM counters are used only while
the files that decide a stage's kernel hash as they did when the counters were taken."""
import os

import bench


def test_stage_hash_depends_on_that_stage_files_only(tmp_path):
    files = {"quant.cu": b"q", "gemm.cu": b"g", "cast.cuh": b"c", "ptx.cuh": b"p", "kernels.h": b"k", "api.cu": b"a"}
    read = lambda f: files[f]
    cast0 = bench.source_hash(bench.STAGE_SOURCES["quant_x"], read)
    gemm0 = bench.source_hash(bench.STAGE_SOURCES["gemm_fwd"], read)
    files["gemm.cu"] = b"g2"  # a GEMM change leaves the casts' key alone
    assert bench.source_hash(bench.STAGE_SOURCES["quant_x"], read) == cast0
    assert bench.source_hash(bench.STAGE_SOURCES["gemm_fwd"], read) != gemm0
    files["cast.cuh"] = b"c2"  # a shared header changes both
    assert bench.source_hash(bench.STAGE_SOURCES["quant_x"], read) != cast0
    # file names are part of the hash: moving bytes between files changes it
    a = bench.source_hash(("quant.cu", "api.cu"), lambda f: {"quant.cu": b"xy", "api.cu": b""}[f])
    b = bench.source_hash(("quant.cu", "api.cu"), lambda f: {"quant.cu": b"x", "api.cu": b"y"}[f])
    assert a != b


def test_traffic_table_keeps_only_current_keys(tmp_path, monkeypatch):
    root = tmp_path
    (root / "profiles").mkdir()
    csrc = root / "fp8_mixed_precision_saturating_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for f in ("quant.cu", "gemm.cu", "cast.cuh", "ptx.cuh", "kernels.h", "api.cu"):
        (csrc / f).write_bytes(f.encode())
    monkeypatch.setattr(bench, "ROOT", str(root))
    hc = bench.source_hash(bench.STAGE_SOURCES["quant_dy"])
    hg = bench.source_hash(bench.STAGE_SOURCES["gemm_bwd"])
    (root / "profiles" / "traffic_per_launch.txt").write_text(
        "# comment\nquant_dy 100 %s\ngemm_bwd 200 %s\ngemm_fwd 300 deadbeefdeadbeef\nunknown 5 %s\n" % (hc, hg, hc))
    t = bench.traffic_table()
    assert t == {"quant_dy": 100.0, "gemm_bwd": 200.0}
    (csrc / "gemm.cu").write_bytes(b"changed")
    assert bench.traffic_table() == {"quant_dy": 100.0}
    os.remove(root / "profiles" / "traffic_per_launch.txt")
    assert bench.traffic_table() == {}
