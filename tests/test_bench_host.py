"""Host-side logic of bench.py on CPU: the clock samples kept for the timed region and
the throttle reasons read from them, the source-hash gate on the committed DRAM-traffic
figure, and the workload description of the JSON line."""

import datetime
import dataclasses
import hashlib
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from sparse_top_routing_router_b300 import configs as K  # noqa: E402


class _FakeSmi:
    def __init__(self, text):
        self.text = text

    def terminate(self):
        pass

    def communicate(self, timeout=None):
        return self.text, ""


def _row(ts, sm, mx, power, reasons=("Not Active",) * 4):
    stamp = datetime.datetime.fromtimestamp(ts).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    return ", ".join([stamp, "0", str(sm), str(mx), str(power), "0x0", *reasons])


def test_clock_samples_inside_the_timed_window_only(monkeypatch):
    t0 = 1_800_000_000.0
    rows = [
        _row(t0 - 1.0, 2032, 2032, 200.0),                       # idle, before the region
        _row(t0 + 0.1, 1200, 2032, 1090.0,
             ("Not Active", "Not Active", "Not Active", "Active")),
        _row(t0 + 0.3, 1250, 2032, 1095.0),
        _row(t0 + 0.5, 1300, 2032, 1099.0),
        _row(t0 + 2.0, 2032, 2032, 210.0,
             ("Active", "Not Active", "Not Active", "Not Active")),   # after the region
        "garbage line",
    ]
    s = bench.ClockSampler(0)
    s.proc = _FakeSmi("\n".join(rows) + "\n")
    s.t0, s.t1 = t0, t0 + 0.6
    monkeypatch.setattr(bench.time, "sleep", lambda _: None)   # stop() waits for a last sample
    out = s.stop()
    assert out["samples"] == 3 and out["samples_total"] == 5
    assert out["sm_mhz"] == 1250 and out["sm_max_mhz"] == 2032
    # only reasons seen inside the window: the later hw_slowdown sample is not ours
    assert out["reasons"] == ["sw_power_cap"]
    assert abs(out["window_s"] - 0.6) < 1e-6


def test_clock_sampler_without_nvidia_smi():
    s = bench.ClockSampler(0)
    s.proc = None
    out = s.stop()
    assert out["sm_mhz"] is None and out["reasons"] == ["nvidia-smi unavailable"]


def test_traffic_figure_only_for_the_profiled_source(tmp_path, monkeypatch):
    src = tmp_path / "kernel.cu"
    src.write_bytes(b"// kernel source\n")
    sha = hashlib.sha256(src.read_bytes()).hexdigest()[:16]
    prof = tmp_path / "traffic.txt"
    prof.write_text(json.dumps([
        {"workload_name": "a", "kernel_sha": sha, "dram_bytes_per_launch": 123},
        {"workload_name": "b", "kernel_sha": "0" * 16, "dram_bytes_per_launch": 456}]))
    monkeypatch.setattr(bench, "KERNEL_SRC", str(src))
    monkeypatch.setattr(bench, "PROFILE_TRAFFIC", str(prof))
    assert bench.traffic_from_profile("a")["dram_bytes_per_launch"] == 123
    assert bench.traffic_from_profile("b") is None          # profiled on another source
    assert bench.traffic_from_profile("c") is None          # never profiled
    src.write_bytes(b"// kernel source, changed\n")
    assert bench.traffic_from_profile("a") is None
    monkeypatch.setattr(bench, "PROFILE_TRAFFIC", str(tmp_path / "missing.txt"))
    assert bench.traffic_from_profile("a") is None


def test_traffic_figure_only_for_the_profiled_routing(monkeypatch):
    monkeypatch.setattr(bench, "traffic_from_profile", lambda name: {"workload_name": name})
    dsv3, sw = K.DSV3_PREFILL, K.SWITCH
    assert bench.traffic_for_run(dsv3, None, None) == {"workload_name": dsv3.name}
    assert bench.traffic_for_run(sw, sw.capacity_factors[0], None) is not None
    # another capacity, a routing variant, FP8 weights, bias updates or other sizes: none
    assert bench.traffic_for_run(sw, 1.25, None) is None
    assert bench.traffic_for_run(dataclasses.replace(dsv3, n_groups=8, topk_groups=4),
                                 None, None) is None
    assert bench.traffic_for_run(dataclasses.replace(dsv3, expert_choice=True), None,
                                 None) is None
    assert bench.traffic_for_run(dataclasses.replace(dsv3, fp8_experts=True), None,
                                 None) is None
    assert bench.traffic_for_run(dsv3, None, 1e-3) is None
    assert bench.traffic_for_run(K.scaled(dsv3, name=dsv3.name + "@T=64", T=64), None,
                                 None) is None


def test_committed_traffic_profile_is_well_formed():
    with open(bench.PROFILE_TRAFFIC) as fh:
        entries = json.load(fh)
    assert isinstance(entries, list) and entries
    for j in entries:
        assert j["workload_name"] in K.BY_NAME
        assert j["dram_bytes_per_launch"] == j["dram_bytes_read"] + j["dram_bytes_write"]
        assert len(j["kernel_sha"]) == 16 and "--clock-control none" in j["command"]


def test_workload_config_names_the_workload():
    d = bench.workload_config(K.SWITCH, 1.25)
    assert d["workload"] == "switch_capacity_bf16" and d["capacity_factor"] == 1.25
    assert (d["T"], d["H"], d["E"], d["I"], d["k"]) == (16384, 4096, 64, 8192, 1)
    assert "model" not in d
    g = bench.workload_config(K.scaled(K.DSV3_PREFILL, n_groups=8, topk_groups=4), None)
    assert g["router_groups"] == {"n_groups": 8, "topk_groups": 4}


def test_peaks_are_read_from_the_measured_file():
    p = bench.peaks()
    if os.path.exists(os.path.join(ROOT, "MEASURED_PEAKS.json")):
        assert p["source"] == "measured" and p["hbm_gbs"] > 1000
    else:
        assert p == {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0,
                     "bf16_tflops_sustained": 1400.0, "source": "fallback"}


def test_cpu_baseline_sample_grows_to_the_batch(monkeypatch):
    from sparse_top_routing_router_b300.inputs import make_inputs
    cfg = K.TINY_F32                       # T=64, E=8, k=2
    d = make_inputs(cfg, device="cpu")
    sizes = []
    real = bench.oracle_sample

    def spy(cfg_, d_, cf_, n, seed):
        sizes.append(n)
        return real(cfg_, d_, cf_, n, seed)
    monkeypatch.setattr(bench, "oracle_sample", spy)
    # a time floor it never reaches: doubles from 5 up to the whole batch
    tr, tf, n, staging = bench.cpu_baseline_sample(cfg, d, None, 5, min_seconds=1e9)
    assert sizes == [5, 10, 20, 40, 64] and n == 64 and staging >= 0.0
    # a floor the first sample meets: one sample
    sizes.clear()
    bench.cpu_baseline_sample(cfg, d, None, 5, min_seconds=0.0)
    assert sizes == [5]


def test_oracle_sample_takes_weight_staging_off_the_clock(monkeypatch):
    from sparse_top_routing_router_b300.inputs import make_inputs
    cfg = K.TINY_F32
    d = make_inputs(cfg, device="cpu")
    bench._HOST_CACHE.clear()
    bench._HOST_CACHE_BYTES[0] = 0
    real = bench._host

    def slow(t):                           # staging that takes 20 ms per tensor
        bench.time.sleep(0.02)
        return real(t)
    monkeypatch.setattr(bench, "_host", slow)
    tr, tf, n, staging = bench.oracle_sample(cfg, d, None, 64, seed=1)
    # every touched expert's three matrices were staged inside combine_subset ...
    assert staging >= 0.02 * 3 * 2
    # ... and that time is not in the expert-stage figure
    assert tf < staging


def test_reference_sample_fits_the_step_budget():
    from sparse_top_routing_router_b300.inputs import make_inputs
    cfg = K.TINY_F32                       # T=64
    d = make_inputs(cfg, device="cpu")
    assert bench.reference_sample_tokens(cfg, d, None, step_budget_s=1e9) == 64
    assert bench.reference_sample_tokens(cfg, d, None, step_budget_s=0.0) == 2


def test_step_quantiles():
    q = bench.step_quantiles([5.0, 1.0, 3.0, 2.0, 4.0])
    assert q["median"] == 3.0 and q["mean"] == 3.0
    assert abs(q["p10"] - 1.4) < 1e-12 and abs(q["p90"] - 4.6) < 1e-12
    assert bench.step_quantiles([7.0]) == {"median": 7.0, "p10": 7.0, "p90": 7.0, "mean": 7.0}


def test_both_arms_describe_the_same_config():
    c = bench.run_config(K.DSV3_PREFILL, None, 1)
    assert c["workload"] == "dsv3_prefill_bf16" and c["parallelism"] == "replicas x1"
    assert "larger than L2" in c["l2"]
    assert "smaller" not in bench.run_config(K.TINY_F32, None, 1)["l2"]
    assert "fit in L2" in bench.run_config(K.TINY_F32, None, 1)["l2"]


def test_default_workload_is_the_largest_single_gpu_config():
    assert bench.DEFAULT_CONFIG == K.DSV3_PREFILL.name
