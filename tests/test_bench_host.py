"""Host-side logic of bench.py (no GPU): the multi-GPU refusal, the clock
summary of a window, and the DRAM traffic record keyed to the kernel sources."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(args, env_extra=None):
    env = dict(os.environ)
    env.update(env_extra or {})
    # a multi-GPU request must be answered without importing torch at all
    code = ("import runpy, sys; sys.argv = ['bench.py'] + %r; "
            "runpy.run_path('bench.py', run_name='__main__'); "
            "assert 'torch' not in sys.modules, 'torch imported'" % (args,))
    return subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True,
                          text=True, timeout=120)


def test_more_than_one_gpu_prints_one_unavailable_line_and_launches_nothing():
    r = _run(["--gpus", "2"])
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["value"] is None and d["n_gpus"] == 2
    assert "single-GPU" in d["unavailable"] and "multicast" in d["unavailable"]


def test_torchrun_ranks_other_than_zero_print_nothing():
    r0 = _run([], {"WORLD_SIZE": "4", "RANK": "0", "LOCAL_RANK": "0"})
    r1 = _run([], {"WORLD_SIZE": "4", "RANK": "1", "LOCAL_RANK": "1"})
    assert r0.returncode == 0 and r1.returncode == 0, (r0.stderr, r1.stderr)
    assert json.loads(r0.stdout.strip())["n_gpus"] == 4
    assert r1.stdout.strip() == ""


def test_clock_summary_keeps_only_the_window(tmp_path):
    sys.path.insert(0, ROOT)
    import bench
    cs = bench.ClockSampler(0, str(tmp_path))
    rows = [
        ("2026/01/01 00:00:00.000", 1900, "Not Active"),
        ("2026/01/01 00:00:01.000", 1500, "Active"),
        ("2026/01/01 00:00:01.500", 1600, "Active"),
        ("2026/01/01 00:00:02.000", 1700, "Not Active"),
        ("2026/01/01 00:00:05.000", 2000, "Not Active"),
    ]
    with open(cs.path, "w") as f:
        for ts, mhz, cap in rows:
            f.write(f"{ts}, 0, {mhz}, 2070, 1200.5, 0x4, Not Active, Not Active, Not Active, {cap}\n")
        f.write("2026/01/01 00:00:02.1, 0, 17")  # a line cut off mid-write is skipped
    cs.done = True
    import datetime
    t = lambda s: datetime.datetime.strptime(s, "%Y/%m/%d %H:%M:%S.%f").timestamp()  # noqa: E731
    s = cs.summary(t("2026/01/01 00:00:00.900"), t("2026/01/01 00:00:02.050"))
    assert s["samples"] == 3
    assert s["sm_mhz"] == 1600
    assert s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["sw_power_cap"]


def test_traffic_is_reported_only_for_the_sources_it_was_captured_on(tmp_path, monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    (tmp_path / "profiles").mkdir()
    with open(tmp_path / "profiles" / "ncu_traffic.json", "w") as f:
        json.dump({"gemm_rs": {"kernel_hash": "aaaa", "dram_bytes_per_launch": 123},
                   "ag_gemm": {"kernel_hash": "bbbb", "dram_bytes_per_launch": 456}}, f)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_hash", lambda op="gemm_rs": "aaaa")
    assert bench.load_traffic("gemm_rs") == 123
    assert bench.load_traffic("ag_gemm") is None  # captured on other sources
    assert bench.load_traffic("moe_layer0") is None  # never captured
    monkeypatch.setattr(bench, "ROOT", str(tmp_path / "missing"))
    assert bench.load_traffic("gemm_rs") is None


def test_committed_traffic_record_names_every_fused_op():
    with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
        d = json.load(f)
    for op in ("ag_gemm", "gemm_rs", "moe_layer0", "moe_layer1"):
        e = d[op]
        assert e["dram_bytes_per_launch"] == e["dram_bytes_read"] + e["dram_bytes_write"]
        assert len(e["kernel_hash"]) == 16 and e["duration_us"] > 0
