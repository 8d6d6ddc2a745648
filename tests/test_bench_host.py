"""Host-side logic of bench.py that feeds the reported roofline: the FLOP each
profiled kernel kind is credited with, the per-kind DRAM traffic summary read
from an ncu CSV, the source-hash gate on that summary, and the peak fallback.
No GPU needed."""
import importlib.util
import os
import types

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


class FakeLib:
    """Stands in for the binding: the chunk width a call of this shape uses."""
    def __init__(self, chunk):
        self.chunk = chunk

    def flce_vocab_chunk(self, N, H, V):
        return min(self.chunk, V)


def args(shards=0):
    return types.SimpleNamespace(vocab_shards=shards)


def test_kind_flops_three_launches(bench):
    N, H, V = 8192, 4096, 128256
    f = bench.kind_flops(FakeLib(14592), N, H, V, args(), merged=False)
    full = 2.0 * N * V * H
    assert f["fwd_logits_lse"] == f["bwd_dz_recompute"] == f["bwd_dw_gemm"] == f["bwd_dx_gemm"] == full
    assert f["bwd_merged"] == 0.0
    # the four kinds add up to the step's 8NVH
    assert sum(v for k, v in f.items()) == pytest.approx(8.0 * N * V * H)


def test_kind_flops_merged(bench):
    N, H, V, cv = 8192, 4096, 128256, 8192
    f = bench.kind_flops(FakeLib(cv), N, H, V, args(), merged=True)
    full = 2.0 * N * V * H
    assert f["bwd_dz_recompute"] == pytest.approx(2.0 * N * cv * H)       # chunk 0 alone
    assert f["bwd_merged"] == pytest.approx(3.0 * full - 2.0 * N * cv * H)
    assert sum(f.values()) - f["bwd_dw_gemm"] - f["bwd_dx_gemm"] == pytest.approx(4.0 * full)


def test_kind_flops_merged_dw_dx(bench):
    N, H, V = 8192, 4096, 128256
    f = bench.kind_flops(FakeLib(14592), N, H, V, args(), merged=2)
    full = 2.0 * N * V * H
    assert f["bwd_dz_recompute"] == f["fwd_logits_lse"] == full
    assert f["bwd_merged"] == 2.0 * full


def test_kind_flops_merged_vocab_shards(bench):
    """Each shard's backward runs its own chunk 0 alone."""
    N, H, V, cv = 1024, 512, 10000, 1024
    f = bench.kind_flops(FakeLib(cv), N, H, V, args(shards=4), merged=True)
    P = 4
    bounds = [round(V * i / P / 256) * 256 for i in range(P)] + [V]
    dz0 = sum(2.0 * N * min(cv, b1 - b0) * H for b0, b1 in zip(bounds, bounds[1:]))
    assert f["bwd_dz_recompute"] == pytest.approx(dz0)
    assert f["bwd_merged"] + f["bwd_dz_recompute"] == pytest.approx(3.0 * 2.0 * N * V * H)


CSV_HEADER = '"ID","Kernel Name","Metric Name","Metric Unit","Metric Value"\n'


def _row(i, name, metric, unit, value):
    return f'"{i}","{name}","{metric}","{unit}","{value}"\n'


def test_traffic_summary_and_source_gate(bench, tmp_path, monkeypatch):
    names = {
        0: "_ZN4flce16gemm_pair_kernelILNS_3EpiE0ELb0ELb0ELi6ELb0EEEv14CUtensorMap_st",  # forward
        1: "_ZN4flce16gemm_pair_kernelILNS_3EpiE1ELb0ELb0ELi6ELb0EEEv14CUtensorMap_st",  # dZ
        2: "_ZN4flce16gemm_pair_kernelILNS_3EpiE2ELb1ELb1ELi6ELb0EEEv14CUtensorMap_st",  # dW
        3: "_ZN4flce16gemm_pair_kernelILNS_3EpiE2ELb0ELb1ELi6ELb0EEEv14CUtensorMap_st",  # dX
        4: "_ZN4flce16gemm_pair_kernelILNS_3EpiE2ELb1ELb1ELi6ELb0EEEv14CUtensorMap_st",  # dW again
        5: "_ZN4flce16bwd_fused_kernelILi6EEEvNS_9FusedMapsENS_11FusedParamsE",          # merged
        6: "_ZN4flce16lse_merge_kernelEPK6float4",                                       # not a GEMM
    }
    text = CSV_HEADER
    for i, n in names.items():
        text += _row(i, n, "dram__bytes_read.sum", "Mbyte", f"{100 * (i + 1):,}")
        text += _row(i, n, "dram__bytes_write.sum", "Kbyte", "500")
        text += _row(i, n, "gpu__time_duration.sum", "usecond", "10")
    csv_path = tmp_path / "cap.csv"
    csv_path.write_text("==PROF== a profiler line\n" + text)
    out = tmp_path / "traffic.txt"
    monkeypatch.setattr(bench, "traffic_path", lambda w: str(out))
    bench.summarize_traffic(str(csv_path), "wl")
    got = bench.load_traffic("wl")
    assert got["fwd_logits_lse"] == pytest.approx(100e6 + 500e3)
    assert got["bwd_dz_recompute"] == pytest.approx(200e6 + 500e3)
    assert got["bwd_dw_gemm"] == pytest.approx(500e6 + 500e3)   # the last of two launches
    assert got["bwd_dx_gemm"] == pytest.approx(400e6 + 500e3)
    assert got["bwd_merged"] == pytest.approx(600e6 + 500e3)
    assert "lse_merge" not in " ".join(got)
    # a summary taken on other kernel source is not used
    lines = out.read_text().splitlines()
    lines = [("# source_sha256 " + "0" * 64) if l.startswith("# source_sha256") else l
             for l in lines]
    out.write_text("\n".join(lines) + "\n")
    assert bench.load_traffic("wl") is None
    # a capture at reduced V (same N and H) scales the forward by V_full / V
    bench.summarize_traffic(str(csv_path), "llama3_n8192", shape=(8192, 4096, 32064))
    got = bench.load_traffic("llama3_n8192")
    assert got["fwd_logits_lse"] == pytest.approx((100e6 + 500e3) * 128256 / 32064)
    assert got["bwd_dx_gemm"] == pytest.approx(400e6 + 500e3)
    with pytest.raises(ValueError):
        bench.summarize_traffic(str(csv_path), "llama3_n8192", shape=(4096, 4096, 32064))


def test_peaks_measured_and_fallback(bench, tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    p = bench.peaks()
    assert p["source"] == "fallback" and p["bf16_sustained"] > 0
    (tmp_path / "MEASURED_PEAKS.json").write_text(
        '{"bf16_tflops": 1899.8, "bf16_tflops_sustained": 1728.5, "hbm_gbs": 6695.5}')
    p = bench.peaks()
    assert p == {"bf16_burst": 1899.8, "bf16_sustained": 1728.5, "hbm_gbs": 6695.5,
                 "source": "measured"}


def test_peak_choice_follows_the_timed_loop(bench):
    pk = {"bf16_burst": 1900.0, "bf16_sustained": 1700.0, "hbm_gbs": 6800.0}
    name, val, why = bench.peak_choice(pk, 0.4)
    assert (name, val) == ("burst", 1900.0) and why
    name, val, why = bench.peak_choice(pk, bench.SUSTAINED_LOOP_S)
    assert (name, val) == ("sustained", 1700.0) and why
    name, _, _ = bench.peak_choice(pk, 3.0)
    assert name == "sustained"


def test_reference_arm_prints_the_same_config(bench, capsys):
    """The reference arm's `config` is built by the same function as ours: the
    workload alone, no engine settings."""
    import json
    a = types.SimpleNamespace(workload="llama3_n8192", shape="64,32,256", seed=0, steps=1,
                              warmup=0, reference_rows=8, gpus=1, z_loss=0.0)
    bench.run_reference(a, 0)
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    want = bench.line_config(bench.workload_spec(a), a, 1)
    assert line["config"] == want
    assert line["impl"] == "reference" and line["steps"] == 1
    for k in ("vocab_chunk", "tiles", "cluster_multicast", "backward"):
        assert k not in line["config"]
    assert want["workload"].startswith("llama3_n8192") and want["N"] == 64
