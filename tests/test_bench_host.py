"""Host logic of bench.py (no GPU): the recorded DRAM traffic is used only for the sources it was
taken on, and the clock record names this GPU's median SM clock and every throttle reason seen."""
import json
import os
import shutil

import bench


def _tree(tmp_path):
    root = tmp_path / "repo"
    shutil.copytree(os.path.join(bench.ROOT, "prefix_shared_kv_ra_gb300", "csrc"),
                    root / "prefix_shared_kv_ra_gb300" / "csrc")
    (root / "include").mkdir(parents=True)
    shutil.copy(os.path.join(bench.ROOT, "include", "ra.h"), root / "include" / "ra.h")
    (root / "profiles").mkdir()
    return root


def _record(root, digest, launches):
    (root / "profiles" / "traffic.json").write_text(json.dumps(
        {"source_digest": digest, "command": "ncu ...", "launches": launches}))


def test_recorded_traffic_follows_the_source_digest(tmp_path, monkeypatch):
    root = _tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(root))
    digest = bench.source_digest()
    assert digest != "" and len(digest) == 16
    _record(root, digest, [{"kernel": "attn_tc_kernel<extend>", "workload": "multiturn_mix", "dram_bytes": 123456},
                           {"kernel": "decode_kernel", "workload": "decode_8b", "dram_bytes": 999}])
    assert bench.recorded_traffic("attn_tc_kernel<extend>", "multiturn_mix") == 123456.0
    assert bench.recorded_traffic("attn_tc_kernel<extend>", "decode_8b") is None      # other workload
    assert bench.recorded_traffic("decode_kernel", "multiturn_mix") is None           # not recorded
    # a record of other sources is not used
    _record(root, "0000000000000000", [{"kernel": "decode_kernel", "workload": "multiturn_mix", "dram_bytes": 5}])
    assert bench.recorded_traffic("decode_kernel", "multiturn_mix") is None
    _record(root, digest, [{"kernel": "attn_tc_kernel<extend>", "workload": "multiturn_mix", "dram_bytes": 123456}])
    # any change to a kernel source (a comment included) retires the figure
    src = root / "prefix_shared_kv_ra_gb300" / "csrc" / "attn_tc.cuh"
    src.write_text(src.read_text() + "\n// edited\n")
    assert bench.source_digest() != digest
    assert bench.recorded_traffic("attn_tc_kernel<extend>", "multiturn_mix") is None
    # no record at all
    (root / "profiles" / "traffic.json").unlink()
    assert bench.recorded_traffic("attn_tc_kernel<extend>", "multiturn_mix") is None


def test_committed_traffic_record_is_complete():
    """The committed record names its command, a 16-digit source digest and integer bytes per launch."""
    with open(os.path.join(bench.ROOT, "profiles", "traffic.json")) as f:
        rec = json.load(f)
    assert "ncu" in rec["command"] and "--clock-control none" in rec["command"]
    assert len(rec["source_digest"]) == 16
    assert rec["launches"]
    for e in rec["launches"]:
        assert {"kernel", "workload", "dram_bytes"} <= set(e) and int(e["dram_bytes"]) > 0


def test_both_arms_print_the_same_config():
    """The GPU line and the oracle (reference) line describe the workload with one dict."""
    class B:
        total_q_extend, n_decode, meta = 9195, 224, {"construction_hit_ratio": 0.70091}
    assert bench.bench_config(B(), 1) == bench.bench_config(B(), 1)
    c = bench.bench_config(B(), 1)
    assert c["parallelism"] == "single GPU" and c["global_batch"] == 256 and "l2" in c


def test_clock_summary_picks_this_gpu_and_flags_reasons(tmp_path):
    s = bench.ClockSampler("GPU-b")
    s.out = str(tmp_path / "clocks.csv")
    s.proc = object()   # as if nvidia-smi had been started
    rows = [
        # uuid, sm, max sm, power, active mask, hw_slowdown, hw_thermal, sw_thermal, sw_power_cap
        "GPU-a, 900, 2070, 300.0, 0x1, Not Active, Not Active, Active, Not Active",
        "GPU-b, 2070, 2070, 900.5, 0x0, Not Active, Not Active, Not Active, Not Active",
        "GPU-b, 2040, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active",
        "GPU-b, 1995, 2070, 1400.0, 0x4, Not Active, Not Active, Not Active, Active",
        "garbage line",
        "GPU-b, [N/A], 2070, 0, 0x0, Not Active, Not Active, Not Active, Not Active",
    ]
    (tmp_path / "clocks.csv").write_text("\n".join(rows) + "\n")
    got = s.summary()
    assert got == {"sm_mhz": 2040.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}
    # another GPU's thermal slowdown is not this run's
    assert "sw_thermal_slowdown" not in got["reasons"]
    # nvidia-smi missing: no record rather than a made-up one
    s.proc = None
    assert s.summary() is None
