"""Host logic of bench.py that needs no GPU: the clock sampler's summary of
nvidia-smi rows (throttle reasons that reject a run), the peak fallback, the
rule that recorded ncu traffic is used only for the kernel source it was
captured on, and the step's launch shape on each benchmark workload."""

import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _row(sm, mx, hw="Not Active", hw_th="Not Active", sw_th="Not Active", cap="Not Active"):
    return ["0", str(sm), str(mx), "900.5", "0x0", hw, hw_th, sw_th, cap]


def test_clock_summary_reports_median_max_and_active_reasons():
    s = bench.ClockSampler(0)
    s.rows = [_row(2070, 2070), _row(1980, 2070, cap="Active"), _row(2040, 2070)]
    out = s.summary()
    assert out["sm_mhz"] == 2040 and out["sm_max_mhz"] == 2070 and out["samples"] == 3
    assert out["reasons"] == ["sw_power_cap"]
    s.rows = [_row(1500, 2070, hw="Active", sw_th="Active")]
    assert s.summary()["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]


def test_clock_summary_without_samples():
    out = bench.ClockSampler(0).summary()
    assert out["samples"] == 0 and out["reasons"] == ["unsampled"] and out["sm_mhz"] is None


def test_clock_summary_skips_unreadable_clock_fields():
    s = bench.ClockSampler(0)
    s.rows = [_row("[N/A]", "[N/A]"), _row(2070, 2070)]
    out = s.summary()
    assert out["sm_mhz"] == 2070 and out["sm_max_mhz"] == 2070 and out["samples"] == 2


def test_measured_peak_and_fallback(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_peaks() == (6800.0, "fallback")
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 6795.5}))
    assert bench.measured_peaks() == (6795.5, "measured")


def test_recorded_traffic_only_for_the_captured_source(tmp_path, monkeypatch):
    csrc = tmp_path / "hierarchical_speculative_decoding_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    src = csrc / "verify_attn.cu"
    src.write_text("// kernel v1\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h = bench.kernel_source_hash("verify_attn.cu")
    (tmp_path / "profiles" / "traffic.txt").write_text(
        "# kernel-file source-hash workload bytes\n"
        f"verify_attn.cu {h} llama2-7b-128k-32layer 2149004288\n")
    assert bench.recorded_traffic("verify_attn.cu", "llama2-7b-128k-32layer") == 2149004288.0
    assert bench.recorded_traffic("verify_attn.cu", "llama3-8b-gqa-128k-b4") is None  # other workload
    src.write_text("// kernel v2\n")  # the kernel changed since the capture
    assert bench.recorded_traffic("verify_attn.cu", "llama2-7b-128k-32layer") is None


def test_committed_traffic_lines_name_existing_kernels():
    with open(os.path.join(ROOT, "profiles", "traffic.txt")) as f:
        lines = [l.split() for l in f if l.strip() and not l.startswith("#")]
    assert lines
    for parts in lines:
        assert len(parts) == 4 and len(parts[1]) == 16 and float(parts[3]) > 0
        assert os.path.exists(os.path.join(ROOT, "hierarchical_speculative_decoding_gb300", "csrc", parts[0]))


def test_every_benchmark_workload_runs_two_launches_per_layer():
    """The step's launch shape per workload: the window rows ride in the verify
    launch where they fit (Llama2-7B: one query head per KV head), else in the
    fused draft (GQA groups of two to four heads); either way a layer is two
    launches.  Groups beyond four heads keep the separate window launch."""
    from types import SimpleNamespace

    from hierarchical_speculative_decoding_gb300 import synth

    names = ["llama2-7b-128k-32layer", "llama3-8b-gqa-128k-b4", "mixed-b8-gqa-16k-128k"]
    assert bench.parse([]).workload == names[0]
    assert bench.parse([]).extra_workloads.split(",") == names[1:]
    expect = {names[0]: (1, False), names[1]: (2, True), names[2]: (2, True)}
    for name in names:
        w = synth.WORKLOADS[name]
        G = w.Hq // w.Hkv
        st = SimpleNamespace(vw_launches=bench.window_launches(G, w.T), window_in_draft=bench.window_in_draft(G, w.T))
        assert (st.vw_launches, st.window_in_draft) == expect[name], name
        assert bench.launches_per_layer(st, two_call=False) == 2, name
    for G, T in ((1, 6), (8, 6), (5, 3)):
        assert not bench.window_in_draft(G, T)
    for G in (2, 3, 4):
        for T in range(1, 17):
            assert bench.window_in_draft(G, T) == (bench.window_launches(G, T) == 2), (G, T)


def test_algorithmic_bytes_match_hand_counts():
    """The byte counts behind the roofline's `achieved`, on the two full-length
    128K workloads with kc full chunks selected per (b, g), against counts done
    by hand from the cache sizes:
    - Llama2-7B verify: K + V of one layer, 32 heads x 131072 x 128 x 2 B x 2
      = 2 GiB, + the 6 verify queries in (bf16) and out (fp32) per head
      (32 x 6 x 128 x 6 B = 147456), + the window row's query and output that
      ride in the launch (32 x 128 x 6 B = 24576);
    - Llama2-7B draft: the chunk means (32 x 16384 x 256 B = 128 MiB), the ids
      (32 x 512 x 4 B), the selected K + V (32 x 512 x 8 rows x 512 B = 64 MiB),
      the query in and the output out (24576);
    - GQA batch 4 verify: 2 GiB + 4 x 32 x 6 x 128 x 6 B (589824);
    - GQA batch 4 draft with the window rows: 128 MiB + 4 x 8 x 512 x 4 B +
      64 MiB + 4 x 32 x 128 x 6 B, + the 256 sink and window keys' K + V
      (4 x 8 x 256 x 512 B = 4 MiB) and the window output (4 x 32 x 128 x 4 B)."""
    import torch

    from hierarchical_speculative_decoding_gb300 import synth

    expect = {
        "llama2-7b-128k-32layer": {"verify": 2**31 + 147456 + 24576,
                                   "draft": 2**27 + 65536 + 2**26 + 24576},
        "llama3-8b-gqa-128k-b4": {"verify": 2**31 + 589824,
                                  "draft": 2**27 + 65536 + 2**26 + 98304 + 2**22 + 65536},
    }
    for name, want in expect.items():
        w = synth.WORKLOADS[name]
        G = w.Hq // w.Hkv
        st = object.__new__(bench.StepState)  # the byte count needs no device state
        st.w = w
        st.seq_cpu = synth.seq_lens_for(w)
        st.vw_launches = bench.window_launches(G, w.T)
        st.window_in_draft = bench.window_in_draft(G, w.T)
        st.idx = torch.arange(w.kc, dtype=torch.int32).expand(1, w.B, w.Hkv, w.kc).clone()
        st.nsel = torch.full((1, w.B, w.Hkv), w.kc, dtype=torch.int32)
        nb = st.bytes_per_launch()
        assert nb["verify"] == want["verify"], name
        assert nb["draft"] == want["draft"], name
