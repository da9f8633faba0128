"""CPU tests of bench.py's host logic behind the roofline fields: the peak
denominators, the source-hash gate on the committed DRAM-traffic table, the
nvidia-smi clock summary and the FLOP count of a step."""
import json
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    import bench as b
    return b


def test_flops_per_step_of_the_bench_workload(bench):
    cfg = bench.workload()
    assert (cfg.M, cfg.d, cfg.F, cfg.P, cfg.chunks) == (8192, 4096, 14336, 2, 8)
    # gate/up 4*M*d*F plus down 2*M*F*d, independent of P and the chunking
    assert bench.flops_per_step(cfg) == 6.0 * 8192 * 4096 * 14336


def test_peaks_come_from_the_measured_file(bench):
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if not os.path.exists(path):
        pytest.skip("no measured peaks in this checkout")
    j = json.load(open(path))
    pk = bench.peaks()
    assert pk["source"] == "measured"
    assert (pk["bf16_burst"], pk["bf16_sustained"], pk["hbm"]) == (j["bf16_tflops"], j["bf16_tflops_sustained"],
                                                                  j["hbm_gbs"])


def test_traffic_table_is_gated_on_the_kernel_sources(bench, monkeypatch):
    table = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
    entries = {k: v for k, v in table.items() if not k.startswith("_")}
    assert entries
    for name, e in entries.items():
        assert e["bytes_per_launch"] > 0
        for src in e["sources"]:
            assert os.path.exists(os.path.join(ROOT, "sequence_tensor_transformer_gb300", "csrc", src)), src
        # the value is reported exactly when the hash matches the current sources
        expect = e["bytes_per_launch"] if bench.sources_sha(e["sources"]) == e["sources_sha"] else None
        assert bench.kernel_traffic(name) == expect
    # any change to a listed source withdraws the number
    monkeypatch.setattr(bench, "sources_sha", lambda names: "0" * 16)
    assert all(bench.kernel_traffic(name) is None for name in entries)
    assert bench.kernel_traffic("no_such_kernel") is None


def test_clock_summary(bench):
    cs = bench.ClockSampler(0)
    row = lambda sm, mx, pw, hw="Not Active", cap="Not Active": [sm, mx, pw, "0x0", hw, "Not Active", "Not Active",
                                                                  cap]
    cs.samples = [row("1500", "2070", "950.5"), row("1600", "2070", "1001.0", cap="Active"),
                  row("1550", "2070", "980.0"), row("[N/A]", "2070", "[N/A]")]
    s = cs.summary()
    assert s["sm_mhz"] == 1550.0 and s["sm_max_mhz"] == 2070.0 and s["power_w_median"] == 980.0
    assert s["samples"] == 4 and s["reasons"] == ["sw_power_cap"]
    cs.samples.append(row("900", "2070", "700", hw="Active"))
    assert cs.summary()["reasons"] == ["hw_slowdown", "sw_power_cap"]
    empty = bench.ClockSampler(0)
    assert empty.summary() is None


def test_config_index_selects_the_workload(bench, monkeypatch):
    """--config N names the five workloads in their listed order; without it
    the boundary (the headline line) runs."""
    import sys
    expect = ["tiny", "boundary", "qwen2", "msweep", "dtp"]
    assert list(bench.CONFIG_WORKLOADS) == expect
    for i, w in enumerate(expect):
        monkeypatch.setattr(sys, "argv", ["bench.py", "--config", str(i)])
        assert bench.parse().workload == w
    monkeypatch.setattr(sys, "argv", ["bench.py"])
    a = bench.parse()
    assert a.workload == "boundary" and a.config is None
    monkeypatch.setattr(sys, "argv", ["bench.py", "--config", "5"])
    with pytest.raises(SystemExit):
        bench.parse()
