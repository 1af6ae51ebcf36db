"""Host-side logic of bench.py that needs no GPU: the DRAM-traffic figure is taken from a committed
ncu summary only while that summary was captured on the current kernel and host sources, and the
peak denominators come from the measured-peaks file when present, else the stated fallback."""
import json
import os

import pytest

import bench


def _write_profile(dirpath, workload, sha, traffic):
    p = dirpath / f"chain_kernel_{workload}.md"
    p.write_text(f"# summary\n\n- kernel_source_sha256: `{sha}`\n- traffic_bytes_per_launch: {traffic}\n\n| a | b |\n")
    return p


def test_every_hashed_source_exists():
    for f in bench.KERNEL_SOURCES:
        assert os.path.exists(os.path.join(bench.ROOT, f)), f
    h = bench.kernel_source_hash()
    assert len(h) == 16 and int(h, 16) >= 0


def test_traffic_only_from_a_summary_of_this_kernel(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "PROFILE_DIR", str(tmp_path))
    assert bench.recorded_traffic("decode_m128_d4096") is None            # no summary
    _write_profile(tmp_path, "decode_m128_d4096", bench.kernel_source_hash(), 69006848)
    assert bench.recorded_traffic("decode_m128_d4096") == 69006848.0
    _write_profile(tmp_path, "decode_m128_d4096", "0" * 16, 69006848)     # taken on another kernel
    assert bench.recorded_traffic("decode_m128_d4096") is None
    _write_profile(tmp_path, "decode_m128_d4096", bench.kernel_source_hash(), "n/a")
    assert bench.recorded_traffic("decode_m128_d4096") is None


def test_committed_summaries_parse():
    # each committed summary names its workload, its kernel source and a positive traffic figure
    d = bench.PROFILE_DIR
    names = [f for f in os.listdir(d) if f.startswith("chain_kernel_") and f.endswith(".md")]
    assert names
    for n in names:
        text = open(os.path.join(d, n)).read()
        assert "kernel_source_sha256: `" in text and "--clock-control none" in text
        line = next(l for l in text.splitlines() if l.startswith("- traffic_bytes_per_launch:"))
        assert float(line.split(":", 1)[1]) > 0


def test_peaks_from_the_measured_file_else_fallback(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    fb = bench.load_peaks()
    assert fb["source"] == "fallback" and fb["hbm_gbs"] == 6800.0 and fb["bf16_tflops"] == 1900.0
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 6698.5, "bf16_tflops": 1927.1,
                                                              "bf16_tflops_sustained": 1727.7}))
    p = bench.load_peaks()
    assert p["source"] == "measured" and p["hbm_gbs"] == 6698.5 and p["bf16_tflops_sustained"] == 1727.7


def test_phase_breakdown_from_a_hand_made_event_log():
    """Two producers feeding two consumers (every consumer needs both): the phases come out as
    the differences of the stamps, the hand-off from the later producer's release."""
    import numpy as np
    import bench
    from mlp_latency_gb300.chain import EVENT_DTYPE
    ev = np.zeros(4, dtype=EVENT_DTYPE)
    #            stage tile  t_start t_acc  t_end
    rows = [(0, 0, 1000, 5000, 6000), (0, 1, 1000, 6000, 8000),
            (1, 0, 9000, 12000, 13000), (1, 1, 10000, 12000, 14000)]
    for i, (s, t, a, b, c) in enumerate(rows):
        ev[i]["stage"], ev[i]["tile"], ev[i]["t_start"], ev[i]["t_acc"], ev[i]["t_end"] = s, t, a, b, c
    deps = [(np.array([0, 2, 4]), np.array([0, 1, 0, 1]))]
    ph = bench.phase_breakdown(ev, deps)
    assert ph["stage0"]["mainloop_us"] == 4.5 and ph["stage0"]["epilogue_T1_us"] == 1.5
    assert ph["stage1"]["handoff_T3_us"] == 1.5 and ph["stage1"]["handoff_T3_min_us"] == 1.0
    assert ph["stage1"]["first_start_us"] == 8.0 and ph["stage1"]["span_us"] == 5.0
    ctas = np.zeros(2, dtype=EVENT_DTYPE)
    ctas["stage"] = -1
    ctas["t_start"], ctas["t_acc"], ctas["t_end"] = [200, 400], [700, 1000], [14500, 15000]
    k = bench.phase_breakdown(ev, deps, ctas)["kernel"]
    assert k["span_us"] == 14.8 and k["entry_spread_us"] == 0.2 and k["setup_us"] == 0.55
    assert k["first_tile_after_entry_us"] == 0.8 and k["teardown_us"] == 1.0
