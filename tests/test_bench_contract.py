"""The benchmark's reference arm (the CPU oracle, timed on the host cores)
keeps the one-line JSON contract, and its launch rules hold, on the CPU."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench(*args, env=None, timeout=600):
    e = dict(os.environ)
    e.update(env or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, env=e,
                          capture_output=True, text=True, timeout=timeout)


def test_reference_arm_prints_one_json_line():
    r = _bench("--impl", "reference", "--steps", "2", "--warmup", "3", "--batch", "1")
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["unit"] == "queries/s" and d["value"] > 0
    assert d["steps"] == 2 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["higher_is_better"] is True and d["scaling"] == "weak" and d["vs_baseline"] is None
    assert d["config"]["workload"] == "long_262144"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert abs(d["ms_per_step"] * d["value"] / 1e3 - 1.0) < 1e-6  # one query per step at batch 1


def test_algorithmic_bytes_closed_forms():
    """The roofline's numerators for the benchmark workload, from the closed
    forms: per query 67,108,864 B of raw keys + 4,194,304 of selected K/V
    (2,048 rows x 2 heads x 128 x 4 B x 2) + 8,192 of slot entries + 2,048
    of indexer query + 16,384 of query and output; the scorer reads the keys
    and the indexer query (the scores it writes are an intermediate); the
    fused gather + attention reads the selected K/V rows and their slot
    entries and the query, and writes the output."""
    import types
    sys.path.insert(0, ROOT)
    import bench
    w = types.SimpleNamespace(batch=8, visible=np.full(8, 262144, np.int32), budget=512, idx_heads=8,
                              idx_dim=64, q_heads=16, kv_heads=2, head_dim=128)
    path, scorer = bench.algorithmic_bytes(w)
    assert path == 8 * (67108864 + 4194304 + 8192 + 2048 + 16384) == 570638336
    assert scorer == 8 * (67108864 + 2048) == 536887296
    assert bench.attend_bytes(w) == 8 * (4194304 + 8192 + 16384) == 33751040
    assert bench.attend_fma(w) == 8 * 2048 * 16 * 128 * 2
    # the batched workload: 65,537 tokens (16,384 groups and one tail token)
    w3 = types.SimpleNamespace(batch=32, visible=np.full(32, 65537, np.int32), budget=512, idx_heads=8,
                               idx_dim=64, q_heads=16, kv_heads=2, head_dim=128)
    path3, scorer3 = bench.algorithmic_bytes(w3)
    assert path3 == 32 * 21000452 == 672014464
    assert scorer3 == 32 * (16777472 + 2048)
    # a ragged query: 3 tail tokens join the row, and the scores count complete groups only
    w.batch, w.visible = 1, np.array([4 * 1000 + 3], np.int32)
    path, scorer = bench.algorithmic_bytes(w)
    W = 4 * 512 + 3
    assert path == 4003 * 64 * 4 + W * 2 * 128 * 4 * 2 + W * 4 + 8 * 64 * 4 + 2 * 16 * 128 * 4
    assert scorer == 4003 * 64 * 4 + 8 * 64 * 4


def test_reference_arm_other_ranks_exit_without_work():
    r = _bench("--impl", "reference", "--steps", "2", "--warmup", "3",
               env={"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"}, timeout=120)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""


@pytest.mark.parametrize("impl", ["reference", "gb300"])
def test_fewer_than_three_warmup_steps_are_refused(impl):
    r = _bench("--impl", impl, "--steps", "2", "--warmup", "2", timeout=120)
    assert r.returncode != 0 and "warmup" in (r.stderr + r.stdout)


@pytest.mark.gpu
def test_gpu_arm_prints_the_full_json_line():
    """One short run of the benchmark's own arm: every key of the line, the
    roofline of the scorer, the host-buffer end-to-end figure, the clock
    record, the launch count (3 per step) and the parity sample."""
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    r = _bench("--steps", "5", "--warmup", "3", "--e2e-steps", "3", "--no-chunked", timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    d = json.loads([ln for ln in r.stdout.splitlines() if ln.strip()][-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "clocks", "e2e", "gpu_launches",
                "roofline", "cpu_baseline"):
        assert key in d, key
    assert d["unit"] == "queries/s" and d["value"] > 0 and d["n_gpus"] == 1 and d["steps"] == 5
    assert d["config"]["workload"] == "long_262144" and "l2" in d["config"]
    assert d["gpu_launches"] == 3 * 5
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    rf = d["roofline"]
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s" and rf["peak"] > 0
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-9 and 0 < rf["frac"] < 1.5
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(d["clocks"])
    assert d["parity_sample"]["ids_bit_exact"] is True
    ra = d["roofline_attend"]
    assert ra["bound"] == "hbm" and ra["bytes_per_launch"] == 33751040
    assert abs(ra["frac"] - ra["achieved"] / ra["peak"]) < 1e-9 and 0 < ra["frac"] < 1.5
    b3 = d["batched_65537"]  # the 32 x 65,537 workload: its own sub-line
    assert b3["value"] > 0 and b3["ms_per_step"] > 0 and b3["queries_per_step"] == 32
    assert b3["path_hbm"]["algorithmic_bytes_per_step"] == 672014464
    for rf in (b3["roofline"], b3["roofline_attend"]):
        assert rf["bound"] == "hbm" and 0 < rf["frac"] < 1.5
    assert b3["cpu_baseline"]["cores"] >= 1 and b3["cpu_baseline_1thread"]["cores"] == 1
