"""Host-side pieces of bench.py that the reported numbers rest on, checked
without a GPU: the metric's compulsory bytes against the byte counts of the
five workloads worked out by hand (8 B per nonzero, 12 B per row, 4 B per
column), the algorithmic bytes of the conversions, and the rule that a
committed DRAM-traffic record is dropped once its kernel's source changes."""
import hashlib
import json

import pytest

import bench


@pytest.mark.parametrize("R, C, Z, want", [
    (4_096, 4_096, 32_768, 327_680),                        # 4096², 8 per row
    (4_194_304, 4_194_304, 20_963_328, 234_815_488),        # 5-point Laplacian, 2048²
    (1_000_000, 1_000_000, 5_000_000, 56_000_000),          # uniform random, 5 per row
    (4_096_000, 4_096_000, 109_215_352, 939_258_816),       # 27-point stencil, 160³
])
def test_compulsory_bytes(R, C, Z, want):
    assert bench.compulsory_bytes(R, C, Z) == want == 8 * Z + 12 * R + 4 * C


def test_compulsory_bytes_eight_byte_values():
    # value 8 B + column 4 B per nonzero; rowPtrs 4 B and y in and out 16 B per row; x 8 B
    assert bench.compulsory_bytes(10, 7, 30, vb=8) == 12 * 30 + 20 * 10 + 8 * 7


def test_call_bytes_laplace2d():
    R = C = 4_194_304
    Z = 20_963_328
    cb = lambda name, K=5: bench.call_bytes(name, R, C, Z, K, K, 0)  # noqa: E731
    assert cb("create") == cb("convert_coo") == 4 * (R + 1) + 4 * Z
    # ELL of width 5: read rowPtrs, colIdx and value; write 5 slots of column
    # and value per row and nnzPerRow
    assert cb("convert_ell") == 4 * (R + 1) + 8 * Z + 8 * R * 5 + 4 * R == 369_033_220
    assert cb("convert_jds") == 4 * (R + 1) + 4 * R + 16 * Z
    for f in ("CSR", "COO", "ELL", "HYB", "JDS"):
        assert cb("spmv_" + f) == 234_815_488


def test_convert_bytes_agree_with_the_step_calls():
    """The per-format conversion bytes of --mode kernels: the step's own
    figures for COO, ELL, HYB and JDS with 4-byte values, and the arrays
    each format reads and writes by hand for SELL and XBLOCK."""
    R, C, Z, K, tail = 1000, 900, 7000, 9, 55
    for f, name in (("COO", "convert_coo"), ("ELL", "convert_ell"), ("JDS", "convert_jds")):
        assert bench.convert_bytes(f, R, C, Z, 4, width=K) == \
            bench.call_bytes(name, R, C, Z, K, K, 0)
    assert bench.convert_bytes("HYB", R, C, Z, 4, width=K, tail=tail) == \
        bench.call_bytes("convert_hyb", R, C, Z, K, K, tail)
    slots = 7300
    # SELL: rowPtrs, perm, CSR entries read, column + value per slot written
    assert bench.convert_bytes("SELL", R, C, Z, 8, slots=slots) == \
        4 * (R + 1) + 4 * R + 12 * Z + 12 * slots
    # XBLOCK: columns twice, values once; row + 16-bit column + value per slot
    assert bench.convert_bytes("XBLOCK", R, C, Z, 4, slots=slots) == 4 * Z + 8 * Z + 10 * slots


def test_traffic_record_follows_its_source(tmp_path, monkeypatch):
    src = tmp_path / "kernel.cu"
    src.write_text("// kernel source\n")
    (tmp_path / "profiles").mkdir()
    rec = {"kernel": "k_demo", "source": "kernel.cu",
           "source_sha256": hashlib.sha256(src.read_bytes()).hexdigest(),
           "dram_bytes_per_launch": 123456}
    (tmp_path / "profiles" / "traffic_demo.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_record("demo", "k_demo") == 123456
    assert bench.traffic_record("demo", "k_other") is None      # another kernel
    assert bench.traffic_record("absent", "k_demo") is None     # no capture
    src.write_text("// kernel source, changed\n")
    assert bench.traffic_record("demo", "k_demo") is None       # stale capture


def test_sample_bytes_count_only_referenced_columns():
    """A row sample reads x only at the columns its nonzeros reference."""
    import numpy as np
    import synth
    rp = np.array([0, 2, 3, 3], np.int32)           # rows of 2, 1 and 0 entries
    ci = np.array([5, 9, 5], np.int32)              # columns 5 and 9, 5 twice
    va = np.ones(3, np.float32)
    s = synth.CSRInput("t", 3, 100, rp, ci, va, np.zeros(100, np.float32),
                       np.zeros(3, np.float32))
    assert bench.sample_bytes(s) == 8 * 3 + 12 * 3 + 4 * 2


def test_dominant_kernels_name_single_kernel_calls():
    """The roofline's kernel is timed by the CUDA events of a call that
    launches that kernel alone."""
    for call, kernel in bench.DOMINANT.values():
        assert kernel.startswith(bench.SINGLE_KERNEL_CALLS[call])
    assert bench.DEFAULT_WORKLOAD == "stencil27"
    assert bench.DEFAULT_WORKLOAD in bench.DOMINANT
    assert set(bench.CONFIG_ORDER) == set(bench.WORKLOAD_DESC)
