"""bench.py's reference arm (the CPU oracle) runs without a GPU: check its
JSON line carries the contract's keys."""
import json
import os
import subprocess
import sys

from conftest import ROOT


def test_reference_arm_prints_one_contract_line():
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "2", "--warmup", "3"], capture_output=True, text=True,
                         timeout=600, cwd=ROOT)
    assert res.returncode == 0, res.stderr
    lines = [l for l in res.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["steps"] == 2
    assert d["cpu_baseline"]["kind"] == "oracle"
    assert d["cpu_baseline"]["cores"] == len(os.sched_getaffinity(0))   # every host core
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def test_warmup_below_three_is_refused():
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "2"], capture_output=True, text=True,
                         timeout=300, cwd=ROOT)
    assert res.returncode != 0


def test_every_mode_has_its_function():
    import bench
    for name in ("bench_gpu", "bench_e2e", "bench_only", "bench_configs", "bench_sweep",
                 "bench_reference", "cpu_baseline", "aggregate_gbs"):
        assert callable(getattr(bench, name, None)), name


def test_link_bound_closed_forms():
    """The e2e step's link bound: with no device-to-host bytes it is the
    host-to-device time alone; with a link whose directions do not slow each
    other it is the longer direction's time; with equal bytes both ways it is
    the time of both at their shared rates."""
    import bench

    free = {"h2d_gbs": 200.0, "d2h_gbs": 100.0, "both": {"h2d_gbs": 200.0, "d2h_gbs": 100.0}}
    assert abs(bench.link_bound_gbs(10**9, 0, 10**9, free) - 200.0) < 1e-9
    assert abs(bench.link_bound_gbs(10**9, 10**9, 2 * 10**9, free) - 200.0) < 1e-9   # 10 ms
    shared = {"h2d_gbs": 210.0, "d2h_gbs": 190.0, "both": {"h2d_gbs": 170.0, "d2h_gbs": 170.0}}
    assert abs(bench.link_bound_gbs(17 * 10**8, 17 * 10**8, 34 * 10**8, shared) - 340.0) < 1e-6
    # 1.7 GB in, 0.85 GB out: 5 ms both ways, then 0.85 GB in alone at 210 GB/s
    t = 0.005 + 0.85e9 / 210e9
    assert abs(bench.link_bound_gbs(17 * 10**8, 85 * 10**7, 10**9, shared) - 1.0 / t) < 1e-6
