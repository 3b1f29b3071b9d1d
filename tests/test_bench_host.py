"""Host-side pieces of bench.py that need no GPU: the sampled, extrapolated
timing of the wgrad oracle, and the rotation of the next rows whose inputs fit
in L2."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import dgr_inputs as gi  # noqa: E402

L2_BYTES = 129e6


def test_wgrad_oracle_sample_extrapolates():
    wi = gi.wgrad_input(2, 300, 128, 256, seed=3)
    r = bench.wgrad_oracle_sample([wi.G, wi.X, wi.offs, wi.main_grad], budget_s=0.2)
    assert r["elements_timed"] >= 16
    assert r["tflops_extrapolated"] > 0
    assert r["full_seconds_extrapolated"] > 0
    assert "E2 N128 K256" in r["sample"]


def test_rotated_next_rows_stream_more_than_twice_l2_between_uses():
    # between two uses of one input copy, the other copies' calls stream their
    # algorithmic bytes: that must exceed twice L2 so no timed call hits in L2
    for name, copies in bench.ROTATE.items():
        assert name in bench.EXTRAS
        assert (copies - 1) * bench.ALGO[name] > 2 * L2_BYTES, name


def test_clock_window_reports_each_window_and_its_reasons():
    c = bench.ClockSampler(0)
    c.proc = object()  # samples are injected; no nvidia-smi here
    t = 1000.0
    c.samples = [(t, "2070, 2070, 900.5, 0x0, Not Active, Not Active, Not Active, Not Active"),
                 (t + 1, "1800, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active")]
    step = c.window(t - 0.1, t + 0.05)
    assert step["sm_mhz"] == 2070.0 and step["reasons"] == [] and step["samples"] == 1
    extra = c.window(t + 0.5, t + 1.2)
    assert extra["sm_mhz"] == 1800.0 and extra["reasons"] == ["sw_power_cap"]
    empty = c.window(t + 5, t + 6)
    assert empty["sm_mhz"] is None and empty["samples"] == 0
    assert c.window(t + 5, t + 6, fallback=True)["samples"] == 2


def test_host_cpu_names_a_model_and_counts_cores():
    h = bench.host_cpu()
    assert isinstance(h["cpu_model"], str) and h["cpu_model"]
    assert h["host_cores"] >= 1


def test_tensor_peak_follows_the_clock_record():
    peaks = {"bf16": 1916.5, "bf16_sus": 1702.9}
    # a short window at full clock, no reason active: the burst figure
    assert bench.tensor_peak(peaks, {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []}) == (1916.5,
                                                                                              "bf16 burst")
    # the power cap, or clocks held well below maximum: the sustained figure
    assert bench.tensor_peak(peaks, {"sm_mhz": 1950.0, "sm_max_mhz": 2070.0,
                                     "reasons": ["sw_power_cap"]})[1] == "bf16 sustained"
    assert bench.tensor_peak(peaks, {"sm_mhz": 1700.0, "sm_max_mhz": 2070.0, "reasons": []})[0] == 1702.9
    assert bench.tensor_peak(peaks, None) == (1916.5, "bf16 burst")


def test_traffic_kept_only_while_the_kernel_sources_match(tmp_path, monkeypatch):
    # a summary's DRAM bytes count only while its `source:` digest matches the
    # kernel's sources; after a change to them the figure is dropped (null)
    csrc = tmp_path / "deterministic_gradient_reduction_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "wgrad.cu").write_text("kernel v1\n")
    (csrc / "tc_common.cuh").write_text("helpers\n")
    (csrc / "dgr_common.cuh").write_text("common\n")
    prof = tmp_path / "profiles"
    prof.mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    digest = bench.source_digest("wgrad")
    assert digest is not None and len(digest) == 64
    (prof / "wgrad.md").write_text(f"text\n\nsource: wgrad {digest}\ntraffic: wgrad 1234\n")
    (prof / "other.md").write_text("traffic: dprob 99\n")  # no source line: not kept
    assert bench.load_traffic() == {"wgrad": 1234}
    (csrc / "tc_common.cuh").write_text("helpers, changed\n")
    assert bench.source_digest("wgrad") != digest
    assert bench.load_traffic() == {}
