"""CPU tests of bench.py's host logic: the launch order the traffic records follow, the ncu CSV
ingestion that writes them (a split tail's fixup folded into its GEMM, the record keyed to the
sources' hash), and the freshness rule that reports no traffic once the sources change."""
import csv
import json
import os

import pytest

import bench
from megatron_tensor_transformer_tcgen05_gb300 import build as build_mod
from megatron_tensor_transformer_tcgen05_gb300.inputs import ATTN_WORKLOADS, WORKLOADS

COLS = ["ID", "Process ID", "Process Name", "Kernel Name", "Block Size", "Grid Size", "Section Name", "Metric Name",
        "Metric Unit", "Metric Value"]


def test_kernel_sequences():
    assert bench.kernel_sequence(WORKLOADS["gpt3-175b"]) == list(range(8))
    assert bench.kernel_sequence(WORKLOADS["gpt3-175b-swiglu"]) == [0, 1, 2, 3, 4, 4, 5]
    assert bench.kernel_sequence(ATTN_WORKLOADS["gpt3-175b-attn"]) == list(range(9, 19))


def _write_csv(path, launches):
    """launches: (kernel name, {metric: (unit, value)}) in launch order, ncu's --csv layout,
    after a line of ncu's own output."""
    with open(path, "w", newline="") as fh:
        fh.write("==PROF== Connected to process 1234\n")
        w = csv.writer(fh, quoting=csv.QUOTE_ALL)
        w.writerow(COLS)
        for i, (name, metrics) in enumerate(launches):
            for m, (unit, value) in metrics.items():
                w.writerow([i, 1234, "python", name, "(320, 1, 1)", "(144, 1, 1)", "Command line profiler metrics", m,
                            unit, f"{value:,}"])


def _launch(name, rd_mb, wr_mb, ms):
    return (name, {"dram__bytes_read.sum": ("Mbyte", rd_mb), "dram__bytes_write.sum": ("Mbyte", wr_mb),
                   "gpu__time_duration.sum": ("msecond", ms)})


@pytest.fixture(scope="module")
def built():
    build_mod.build()  # ingestion names kernels through the library (loads without a GPU)


def test_ingest_folds_fixups_and_keys_the_sources(tmp_path, built):
    gemm = "void mlp::umma_gemm_kernel<512, 0, 1, 2, 2>(mlp::GemmArgs)"
    fix = "void mlp::splitk_fixup_kernel<2>(mlp::GemmArgs, int, int)"
    launches = [_launch(gemm, 1000.0, 100.0, 2.5), _launch(fix, 40.0, 1.0, 0.02),  # fwd_up + its fixup
                _launch(gemm, 2000.0, 10.0, 2.4),                                     # fwd_down, whole tiles only
                _launch(gemm, 3000.0, 400.0, 2.6), _launch(fix, 44.0, 0.0, 0.03),
                _launch(gemm, 4000.0, 10.0, 2.4), _launch(gemm, 5000.0, 1200.0, 2.5), _launch(gemm, 6000.0, 1200.0, 2.5),
                _launch("colsum_partial_kernel", 100.0, 0.1, 0.02), _launch("bias_grad_finalize_kernel", 25.0, 0.0, 0.01)]
    src, out = tmp_path / "m.csv", tmp_path / "traffic.json"
    _write_csv(src, launches)
    bench.ingest_ncu(WORKLOADS["gpt3-175b"], "gpt3-175b", str(src), str(out))
    rec = json.loads(out.read_text())
    assert rec["workload"] == "gpt3-175b"
    assert rec["source_sha256"] == bench._source_sha256("mlp")
    got = {int(k): v for k, v in rec["bytes_per_launch"].items()}
    want = {0: 1141e6, 1: 2010e6, 2: 3444e6, 3: 4010e6, 4: 6200e6, 5: 7200e6, 6: 100.1e6, 7: 25e6}
    assert got.keys() == want.keys()
    for k in want:
        assert got[k] == pytest.approx(want[k], rel=1e-9), k


def test_ingest_rejects_a_capture_of_the_wrong_length(tmp_path, built):
    src, out = tmp_path / "m.csv", tmp_path / "traffic.json"
    _write_csv(src, [_launch("void mlp::umma_gemm_kernel<512, 0, 1, 2, 2>(mlp::GemmArgs)", 1.0, 1.0, 1.0)] * 5)
    with pytest.raises(SystemExit, match="5 launches"):
        bench.ingest_ncu(WORKLOADS["gpt3-175b"], "gpt3-175b", str(src), str(out))
    assert not out.exists()


def test_traffic_is_reported_only_for_the_sources_it_was_captured_on(tmp_path, monkeypatch):
    (tmp_path / "profiles").mkdir()
    rec = {"workload": "w", "source_sha256": "captured-on", "bytes_per_launch": {"2": 4.5e9}}
    (tmp_path / "profiles" / "traffic_w.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "_source_sha256", lambda kind="attention": "captured-on")
    assert bench._ncu_traffic("w", 2, "gelu") == 4.5e9
    assert bench._ncu_traffic("w", 3, "gelu") is None          # no figure for that kernel
    assert bench._ncu_traffic("other", 2, "gelu") is None      # no record for that workload
    monkeypatch.setattr(bench, "_source_sha256", lambda kind="attention": "changed-since")
    assert bench._ncu_traffic("w", 2, "gelu") is None


def test_mlp_hash_ignores_the_attention_sources():
    """An MLP workload's record stays valid across edits to the attention core alone."""
    files = sorted(os.listdir(os.path.join(bench.ROOT, "megatron_tensor_transformer_tcgen05_gb300", "csrc")))
    assert any(f in bench.ATTN_ONLY_SOURCES for f in files)
    assert bench._source_sha256("mlp") != bench._source_sha256("attention")
