"""Host logic of the benchmark's bookkeeping (CPU only): the algorithmic bytes and
flops every fraction is built on, the reading of ncu CSVs into the committed
records, and the source digest that decides whether a record still applies."""
import os
import shutil
from types import SimpleNamespace

import pytest

import bench
from tensor_core_matrix_02_gb300 import workloads as W


def problem(name, shape=None):
    r = W.RECIPES[name]
    M, N, K = shape if shape else (r.M, r.N, r.K)
    return W.Problem(name, M, N, K, r.ta, r.tb, r.tacc, None, None, None, r.sparse, None)


# The configurations' algorithmic bytes, counted by hand from their definitions: A (or
# the compressed values, K/2 per row, plus the 2-bit index, K/8 bytes per row), B, C
# and D each once (8-bit inputs 1 byte, 16-bit 2, C and D of f32 or i32 4 bytes).
BYTES = {
    "dense_f16_128": 128 * 256 * 2 + 256 * 128 * 2 + 2 * 128 * 128 * 4,                    # 262,144
    "dense_i8_4096": 2 * 4096 * 4096 + 2 * 4096 * 4096 * 4,                                # 167.8 MB
    "dense_bf16_8192": 2 * 8192 * 8192 * 2 + 2 * 8192 * 8192 * 4,                          # 805.3 MB
    "dense_bf16_skinny": 2 * 1024 * 65536 * 2 + 2 * 1024 * 1024 * 4,                       # 276.8 MB
    "sparse_f16_random": 8192 * 4096 * 2 + 8192 * 1024 + 8192 * 8192 * 2 + 2 * 8192 * 8192 * 4,   # 746.6 MB
    "sparse_f16_keep02": 8192 * 4096 * 2 + 8192 * 1024 + 8192 * 8192 * 2 + 2 * 8192 * 8192 * 4,
    "sparse_e4m3_e5m2": 16384 * 8192 + 16384 * 2048 + 16384 * 16384 + 2 * 16384 * 16384 * 4,  # 2583.7 MB
    "dense_e4m3_16384": 2 * 16384 * 16384 + 2 * 16384 * 16384 * 4,                         # 2684.4 MB
}


@pytest.mark.parametrize("name", sorted(BYTES))
def test_algorithmic_bytes_match_the_configurations(name):
    assert bench.algorithmic_bytes(problem(name)) == BYTES[name]


def test_flops_count_the_uncompressed_K():
    # the pages' ops column: a 16 x 16 x 64 sparse product is 32768 ops
    p = W.Problem("x", 16, 16, 64, "f16", "f16", "f32", None, None, None, "random", None)
    assert p.flops == 32768
    assert problem("sparse_e4m3_e5m2").flops == 2 * 16384 ** 3


# each suite GEMM's peak as a multiple of the bf16 one: FP8 twice the 16-bit rate, 4:2
# twice the dense rate of its type (the tcgen05 ceilings: 8192, 16384, 16384 and ~32k
# ops per SM clock for bf16, E4M3, 4:2 f16 and 4:2 FP8); i8 runs on the bf16 path
PEAK_RATIO = {"dense_i8_4096": 1.0, "dense_bf16_8192": 1.0, "dense_bf16_skinny": 1.0,
              "sparse_f16_keep02": 2.0, "sparse_f16_random": 2.0, "sparse_e4m3_e5m2": 4.0,
              "dense_e4m3_16384": 2.0}


def test_every_suite_workload_has_a_kernel_and_a_peak():
    assert sorted(PEAK_RATIO) == sorted(bench.SUITE)
    pk = dict(bench.FALLBACK_PEAKS)
    for name in bench.SUITE:
        p = problem(name)
        kernel, pattern = bench.kernel_of(p)
        assert pattern in kernel
        assert bench.tensor_peak(p, pk) == pytest.approx(PEAK_RATIO[name] * pk["bf16_tflops"])
        assert bench.tensor_peak(p, pk, sustained=True) == pytest.approx(
            PEAK_RATIO[name] * pk["bf16_tflops_sustained"])


HEADER = '"ID","Process ID","Process Name","Host Name","Kernel Name","Context","Stream","Block Size",' \
         '"Grid Size","Device","CC","Section Name","Metric Name","Metric Unit","Metric Value"\n'


def csv_rows(kernel, metrics, launch_id="0"):
    out = ""
    for name, unit, value in metrics:
        out += (f'"{launch_id}","1","python3","127.0.0.1","void {kernel}(CUtensorMap_st, GemmArgs)","1","7",'
                f'"(384, 1, 1)","(152, 1, 1)","0","10.3","Command line profiler metrics","{name}","{unit}","{value}"\n')
    return out


def write_csv(tmp_path, body):
    path = tmp_path / "capture.csv"
    path.write_text("==PROF== Connected to process 1\n" + HEADER + body)
    return str(path)


def test_ncu_values_are_brought_to_base_units(tmp_path):
    body = csv_rows("gemm_pair_kernel<0, 0, 0>", [
        ("dram__bytes_read.sum", "Gbyte", "1.5"), ("dram__bytes_write.sum", "Kbyte", "2,048"),
        ("gpu__time_duration.sum", "usecond", "175.5"), ("sm__cycles_elapsed.avg.per_second", "Ghz", "1.8"),
        ("sm__pipe_tensor_cycles_active.avg.pct_of_peak_sustained_elapsed", "%", "70.5")])
    body += csv_rows("other_kernel", [("dram__bytes_read.sum", "byte", "7")], launch_id="1")
    got = bench._ncu_launches(write_csv(tmp_path, body), "gemm_pair_kernel")
    assert len(got) == 1
    m = got[0]
    assert m["dram__bytes_read.sum"] == pytest.approx(1.5e9)
    assert m["dram__bytes_write.sum"] == pytest.approx(2.048e6)
    assert m["gpu__time_duration.sum"] == pytest.approx(175.5e3)      # nanoseconds
    assert m["sm__cycles_elapsed.avg.per_second"] == pytest.approx(1.8e9)
    assert m["sm__pipe_tensor_cycles_active.avg.pct_of_peak_sustained_elapsed"] == pytest.approx(70.5)


def test_an_unknown_ncu_unit_is_an_error(tmp_path):
    body = csv_rows("gemm_pair_kernel<0, 0, 0>", [("dram__bytes_read.sum", "furlong", "3")])
    with pytest.raises(SystemExit):
        bench._ncu_launches(write_csv(tmp_path, body), "gemm_pair_kernel")


def full_metrics(read, write, ns, hz, tensor_pct, dram_pct):
    return [("gpu__time_duration.sum", "ns", str(ns)), ("dram__bytes_read.sum", "byte", str(read)),
            ("dram__bytes_write.sum", "byte", str(write)),
            ("sm__pipe_tensor_cycles_active.avg.pct_of_peak_sustained_elapsed", "%", str(tensor_pct)),
            ("gpu__dram_throughput.avg.pct_of_peak_sustained_elapsed", "%", str(dram_pct)),
            ("sm__cycles_elapsed.avg.per_second", "hz", str(hz))]


def test_ncu_record_round_trip_and_digest(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "NCU_PATH", str(tmp_path / "ncu.json"))
    monkeypatch.setattr(bench, "peaks", lambda: ({"hbm_gbs": 8000.0, "bf16_tflops": 2000.0,
                                                   "bf16_tflops_sustained": 1800.0}, "measured"))
    # two launches of the kernel: the record keeps their means
    body = csv_rows("gemm_pair_kernel<0, 0, 0>", full_metrics(4e8, 2e8, 200_000, 1.8e9, 70, 40), "0")
    body += csv_rows("gemm_pair_kernel<0, 0, 0>", full_metrics(6e8, 2e8, 300_000, 1.6e9, 60, 50), "1")
    shape = [8192, 8192, 2048]
    bench.record_ncu(SimpleNamespace(workloads=["dense_bf16_8192"], shape=shape,
                                     record_ncu=write_csv(tmp_path, body)))
    rec = bench.recorded_ncu("gemm_pair_kernel<f16>", "dense_bf16_8192")
    assert rec is not None
    assert rec["shape"] == shape and rec["launches"] == 2
    assert rec["ncu_duration_us"] == pytest.approx(250.0)
    assert rec["dram_read"] == 500_000_000 and rec["dram_write"] == 200_000_000
    assert rec["dram_gbs"] == pytest.approx(7e8 / 250e-6 / 1e9, rel=1e-3)
    assert rec["dram_frac_of_hbm"] == pytest.approx(7e8 / 250e-6 / 1e9 / 8000.0, rel=1e-3)
    assert rec["sm_mhz"] == pytest.approx(1700.0)
    assert rec["tensor_pipe_active_pct"] == pytest.approx(65.0)
    assert rec["algorithmic_bytes"] == bench.algorithmic_bytes(problem("dense_bf16_8192", shape))
    assert rec["tflops_under_ncu"] == pytest.approx(2 * 8192 * 8192 * 2048 / 250e-6 / 1e12, rel=1e-3)
    # a record taken on other kernel sources no longer applies
    monkeypatch.setattr(bench, "source_digest", lambda kernel: "0" * 16)
    assert bench.recorded_ncu("gemm_pair_kernel<f16>", "dense_bf16_8192") is None


def test_traffic_record_round_trip_and_digest(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "TRAFFIC_PATH", str(tmp_path / "traffic.json"))
    body = csv_rows("gemm_pair_kernel<1, 0, 0>", [("dram__bytes_read.sum", "Gbyte", "8.49"),
                                                  ("dram__bytes_write.sum", "Gbyte", "1.07"),
                                                  ("gpu__time_duration.sum", "msecond", "2.5")])
    bench.record_traffic(SimpleNamespace(workloads=["dense_e4m3_16384"], record_traffic=write_csv(tmp_path, body)))
    assert bench.recorded_traffic("gemm_pair_kernel<f8f6f4>", "dense_e4m3_16384") == 9_560_000_000
    monkeypatch.setattr(bench, "source_digest", lambda kernel: "0" * 16)
    assert bench.recorded_traffic("gemm_pair_kernel<f8f6f4>", "dense_e4m3_16384") is None


def test_source_digest_follows_the_kernels_files(tmp_path, monkeypatch):
    src = os.path.join(bench.ROOT, "tensor_core_matrix_02_gb300", "csrc")
    dst = tmp_path / "tensor_core_matrix_02_gb300" / "csrc"
    dst.mkdir(parents=True)
    for f in set(sum(bench.KERNEL_SOURCES.values(), [])) | set(bench.COMMON_SOURCES):
        shutil.copy(os.path.join(src, f), dst / f)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    pair0 = bench.source_digest("gemm_pair_kernel<f16>")
    sparse0 = bench.source_digest("gemm_sparse_pair_kernel<f16>")
    assert pair0 == bench.source_digest("gemm_pair_kernel<f8f6f4>")   # one family, one digest
    with open(dst / "gemm_pair_kernel.cuh", "a") as f:
        f.write("\n")
    assert bench.source_digest("gemm_pair_kernel<f16>") != pair0
    assert bench.source_digest("gemm_sparse_pair_kernel<f16>") == sparse0
    with open(dst / "api.cu", "a") as f:                              # the launch code is common
        f.write("\n")
    assert bench.source_digest("gemm_sparse_pair_kernel<f16>") != sparse0
