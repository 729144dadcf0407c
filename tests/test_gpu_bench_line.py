"""bench.py's own arm on a small workload prints one JSON line with the keys
the benchmark contract asks for: the headline metric, the HBM roofline of the
dominant kernel, every logits path against its own byte count, the
end-to-end figure with the whole gradient coming back to the host, and the
clocks sampled during the timed region."""
import json
import os
import subprocess
import sys

import pytest

from vocab_wide_logprob_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_our_arm_line():
    w = wl.QWEN_G8
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--workload", w.name,
                        "--steps", "3", "--warmup", "3", "--e2e-steps", "2", "--per-config",
                        wl.TINY.name, "--no-cpu-baseline", "--no-copy-ceiling"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "roofline",
              "e2e", "gpu_launches", "clocks", "paths", "per_config", "useful_groups_per_s"):
        assert k in d, k
    assert d["steps"] == 3 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["config"]["workload"] == w.name and d["value"] > 0
    rf = d["roofline"]
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s" and rf["peak"] > 0
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-9
    # the whole gradient, logp, w and the loss come back every end-to-end step
    e = d["e2e"]
    grad_bytes = w.N * w.T * w.V * w.elem_bytes
    assert e["d2h_bytes_per_step"] >= grad_bytes + 2 * 4 * w.N * w.C + 4
    assert e["h2d_bytes_per_step"] >= d["workload_stats"]["valid_tokens_per_rank"] * w.V * 2
    assert e["results_match"] is True and e["value"] > 0
    for path in ("two_pass", "skip_zero_weight", "fused"):
        pr = d["paths"][path]
        assert pr["ms_per_step"] > 0 and pr["logits_bytes_per_step"] > 0
    assert wl.TINY.name in d["per_config"]
    assert d["gpu_launches"] == 6 * d["steps"]


@pytest.mark.parametrize("rows_per_pass,passes", [(-1, 2), (2048, 1)])
def test_lmhead_line_counts_every_pass(rows_per_pass, passes):
    """The LM-head loss line: a tensor-core roofline, and a launch count with
    the backward's four kernels once per pass (passes of the scored rows
    present leave an empty second pass over the 2,048 possible rows; passes
    of 2,048 rows one pass)."""
    w = wl.QWEN_G8
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--path",
                        "lmhead_fwd_bwd", "--workload", w.name, "--steps", "3", "--warmup", "3",
                        "--lmhead-rows-per-pass", str(rows_per_pass), "--no-cpu-baseline",
                        "--no-clocks"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["roofline"]["bound"] == "tensor" and d["roofline"]["frac"] > 0
    assert d["bwd_passes"] == passes
    assert d["gpu_launches"] == (9 + 4 * passes) * d["steps"]
