#!/usr/bin/env python
"""Benchmark of the Dr. GRPO loss hot path (forward + backward) on GB300.

One step = grpo_mask -> grpo_advantage -> grpo_loss_fwd -> grpo_loss_bwd on
one stream, over one batch of synthetic inputs already resident in HBM.  The
default workload is the largest one that fits one GPU: the long-completion
batch (B=4 prompts x G=8, P=512, C=3584, V=151936, bf16 logits ~N(0, 3^2),
k3 KL with beta=0.04): 39.8 GB of logits and a separate 39.8 GB dlogits
buffer, far larger than L2, so no flush is needed between steps.

Prints ONE JSON line (rank 0):
  value        completion tokens/s (valid tokens / device step time), all ranks
  roofline     the dominant kernel (dlogits_kernel, one launch per step):
               algorithmic bytes / its CUDA-event duration vs measured HBM peak
  paths        the same workload on each logits path (the two calls, the two
               calls skipping zero-weight rows, the single-pass call), each
               against its own byte count, with useful groups per second
  per_config   the same summary for the other Qwen2.5-shaped workloads
  e2e          the same metric through the public API with host buffers:
               the logits in pinned host memory (grpo_loss_fwd_bwd_host moves
               only the scored rows to the device and writes the whole dlogits
               into pinned host memory), host -> device copies of the other
               inputs and device -> host copies of logp, w and the loss, all
               inside the timed region
  cpu_baseline the float64 CPU oracle, timed on a bounded sample
``--impl reference`` times the oracle alone (host cores) as the reference arm.
"""
from __future__ import annotations

import argparse
import hashlib
import glob
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from vocab_wide_logprob_gb300 import workloads as wl  # noqa: E402

METRIC = "completion tokens/s and logits GB/s (% of HBM roofline), Dr.GRPO loss fwd+bwd"
UNIT = "completion tokens/s"
KERNELS_PER_STEP = 6  # mask, advantage, prep, lse_gather, surrogate, dlogits (fused: 5)
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0  # GB300's nominal HBM3e bandwidth, for context only


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=wl.LONG.name, choices=sorted(wl.BY_NAME))
    p.add_argument("--per-config", default="auto",
                   help="other workloads timed after the main one (comma-separated names); "
                        "auto: every Qwen2.5-shaped workload but the main one; none: skip")
    p.add_argument("--e2e-steps", type=int, default=20,
                   help="end-to-end steps per timed loop (fewer when a loop would pass 1.5 s)")
    p.add_argument("--no-e2e", action="store_true", help="skip the end-to-end leg")
    p.add_argument("--cpu-seconds", type=float, default=10.0)
    p.add_argument("--reference-seconds", type=float, default=90.0,
                   help="--impl reference: host seconds the whole run (warm-up + timed) aims at")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-clocks", action="store_true")
    p.add_argument("--no-copy-ceiling", action="store_true")
    p.add_argument("--skip-zero-weight", action="store_true",
                   help="backward skips reading rows whose gradient weight is exactly 0; "
                        "the skipped reads are left out of the byte count")
    p.add_argument("--path", choices=["two_pass", "fused", "lmhead_logprobs", "lmhead_fwd_bwd"],
                   default="two_pass",
                   help="two_pass: grpo_loss_fwd then grpo_loss_bwd; fused: grpo_loss_fwd_bwd; "
                        "lmhead_logprobs: log-probs from hidden states with the LM-head "
                        "projection on the tensor cores (the no-grad old/reference pass); "
                        "lmhead_fwd_bwd: the loss from hidden states and its gradients with "
                        "respect to the hidden states and the LM head, on the tensor cores")
    p.add_argument("--no-other-path", dest="also_other_path", action="store_false",
                   help="skip timing every logits path of the main workload for the record")
    p.add_argument("--hidden", type=int, default=896,
                   help="hidden size of the LM-head paths (Qwen2.5-0.5B: 896)")
    p.add_argument("--lmhead-rows-per-pass", type=int, default=-1,
                   help="LM-head backward: rows per pass of its workspace (-1: the scored "
                        "rows present, one pass over them; 0: every possible row)")
    return p.parse_args()


# --------------------------------------------------------------------------
# algorithmic byte counts: two reads of the scored rows + one write of
# dlogits (the method's count), and the fused path's one read + one write
# --------------------------------------------------------------------------

def algorithmic_bytes(w: wl.Workload, t_valid: int, t_read_bwd: int | None = None) -> dict:
    """Bytes each call must move.  t_read_bwd: scored rows the backward reads
    (all of them, unless rows with zero gradient weight are skipped)."""
    e = w.elem_bytes
    N, T, C, V = w.N, w.T, w.C, w.V
    small = 4 * N * C * (3 + (w.old_sigma is not None) + (w.ref_sigma is not None))
    tr = t_valid if t_read_bwd is None else t_read_bwd
    return {
        # the scored rows read once + ids of scored tokens + logp/lse/w vectors
        "fwd": t_valid * V * e + 8 * t_valid + small,
        # the scored rows read again + every row of dlogits written once
        "bwd": tr * V * e + N * T * V * e + 16 * t_valid,
        "mask_adv": 8 * N * C + N * C + 8 * N,
        # the roofline count of the whole method: two reads + one write
        "step_logits": (t_valid + tr) * V * e + N * T * V * e,
        # the fused call: one read of the scored rows + one write of dlogits
        "fused": t_valid * V * e + N * T * V * e + 8 * t_valid + small,
        "step_logits_fused": t_valid * V * e + N * T * V * e,
    }


def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f)
    except OSError:
        return {}


# the source files that define each kernel (the capture's hash covers these)
KERNEL_SOURCES = {
    "dlogits_kernel": ("dlogits.cu", "common.cuh"),
    "lse_gather_kernel": ("lse_gather.cu", "common.cuh"),
    "grpo_loss_fwd_bwd": ("fused.cu", "dlogits.cu", "lse_gather.cu", "common.cuh"),
    "lmhead_lse_kernel": ("lmhead.cu", "lmhead.cuh", "pair_pipeline.cuh", "tc.cuh", "common.cuh"),
    "lmhead_fwd_bwd": ("lmhead.cu", "lmhead_bwd.cu", "lmhead.cuh", "pair_pipeline.cuh", "tc.cuh",
                       "common.cuh", "mask_advantage.cu", "lse_gather.cu", "surrogate.cu"),
}


def sources_sha(kernel: str) -> str:
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "vocab_wide_logprob_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def lmhead_bwd_passes(w, rows_per_pass: int) -> int:
    """Passes of the LM-head backward over a workspace sized for
    ``rows_per_pass`` rows, by the library's layout rule: every possible row
    (N*C rounded up to 256) in passes of rows_per_pass rounded up to 256 (0:
    one pass).  Passes past the scored rows find no row and return at once."""
    cap = -(-w.N * w.C // 256) * 256
    r = cap if rows_per_pass <= 0 else min(cap, -(-rows_per_pass // 256) * 256)
    return -(-cap // r)


def recorded_traffic(kernel: str, w: wl.Workload, hidden: int | None = None):
    """DRAM bytes (read + write) per launch of `kernel` on workload `w` from a
    committed ncu capture (profiles/traffic.json); None when there is none for
    this workload or when the kernel's sources changed since the capture."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            recs = json.load(f)
    except (OSError, ValueError):
        return None
    # a capture of this workload ("kernel@workload"), else the kernel's default one
    rec = recs.get(f"{kernel}@{w.name}") or recs.get(kernel)
    if (not rec or rec.get("sources_sha") != sources_sha(kernel) or rec.get("workload") != w.name
            or rec.get("hidden") != hidden):
        return None
    return rec["dram_bytes_per_launch"]


def cpu_model() -> str | None:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name"):
                return line.split(":", 1)[1].strip()
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return None


def run_env(dev) -> dict:
    """What produced the numbers: GPU, driver, toolkit, torch, and a hash of
    the library's sources (a copy of the tree may come without its git history)."""
    import torch
    env = {"gpu": torch.cuda.get_device_name(dev), "torch": torch.__version__,
           "cuda_runtime": torch.version.cuda, "driver": None, "nvcc": None}
    try:
        out = subprocess.run(["nvidia-smi", "--query-gpu=driver_version", "--format=csv,noheader",
                              "-i", str(dev.index or 0)], capture_output=True, text=True,
                             timeout=20).stdout.strip()
        env["driver"] = out.splitlines()[0] if out else None
    except (OSError, subprocess.SubprocessError, IndexError):
        pass
    try:
        out = subprocess.run(["nvcc", "--version"], capture_output=True, text=True,
                             timeout=20).stdout
        env["nvcc"] = next((l.split("release", 1)[1].strip() for l in out.splitlines()
                            if "release" in l), None)
    except (OSError, subprocess.SubprocessError):
        pass
    h = hashlib.sha256()
    for path in sorted(glob.glob(os.path.join(ROOT, "vocab_wide_logprob_gb300", "csrc", "*"))
                       + glob.glob(os.path.join(ROOT, "include", "*.h"))):
        with open(path, "rb") as f:
            h.update(os.path.basename(path).encode())
            h.update(f.read())
    env["sources_sha256"] = h.hexdigest()[:16]
    return env


def input_record(w: wl.Workload, ids_np, R_np, logits) -> dict:
    """Seed and fingerprints of the step's inputs, and the workload's
    statistics (truncated completions, groups with reward contrast)."""
    import torch
    bits = logits.view(torch.int16 if logits.element_size() == 2 else torch.int32)
    # order-sensitive device checksum of the logits: sum of value * (index mod a prime)
    chk = 0
    rows = bits.reshape(-1, bits.shape[-1])
    weights = (torch.arange(bits.shape[-1], device=bits.device, dtype=torch.int64) % 1000003) + 1
    for r0 in range(0, rows.shape[0], 1024):
        part = rows[r0:r0 + 1024].to(torch.int64)
        chk = (chk + int(((part * weights).sum(dim=1) % 2147483647
                          * ((torch.arange(r0, r0 + part.shape[0], device=bits.device) % 65521)
                             + 1)).sum().item())) % 2147483647
    comp = ids_np[:, w.P:]
    truncated = float(np.mean(~np.any(comp == w.eos_id, axis=1))) if w.C > 0 else 0.0
    Rg = R_np.reshape(w.B, w.G)
    return {"seed": w.seed, "ids_sha256": hashlib.sha256(ids_np.tobytes()).hexdigest()[:16],
            "rewards_sha256": hashlib.sha256(R_np.tobytes()).hexdigest()[:16],
            "logits_checksum": chk, "truncated_fraction": truncated,
            "groups_without_contrast": int(np.sum(Rg.max(axis=1) == Rg.min(axis=1)))}


def copy_ceiling(g, dev, nbytes: int = 4 << 30, reps: int = 10) -> float:
    """Device-to-device copy with the library's 16-byte vector copy kernel
    over two 4 GiB buffers: (read + write bytes) / best time, GB/s."""
    import torch
    src = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    dst = torch.empty_like(src)
    src.fill_(1)
    for _ in range(2):
        g.grpo_copy(dst, src)
    best = float("inf")
    for _ in range(reps):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        g.grpo_copy(dst, src)
        b.record()
        torch.cuda.synchronize()
        best = min(best, a.elapsed_time(b) / 1e3)
    del src, dst
    torch.cuda.empty_cache()
    return 2 * nbytes / best / 1e9


def config_record(w: wl.Workload, world: int) -> dict:
    """The workload's configuration, the same in both arms."""
    return {"workload": w.name, "B": w.B, "G": w.G, "P": w.P, "C": w.C, "V": w.V,
            "logits_dtype": w.dtype, "beta": w.beta, "eps": w.eps,
            "l2": f"inputs larger than L2 ({w.logits_bytes / 1e9:.2f} GB logits); no flush",
            "parallelism": f"dp{world} (independent groups)"}


# --------------------------------------------------------------------------
# clocks during the timed region
# --------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"grpo_bench_clocks_{os.getpid()}.csv")
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "100"]
        if gpu_id:
            cmd += ["-i", gpu_id]
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(cmd, stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    sm.append(float(parts[2]))
                    smax.append(float(parts[3]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[6:10]):
                    if v.lower() == "active":
                        reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# --------------------------------------------------------------------------
# oracle on a bounded sample (CPU baseline and the reference arm)
# --------------------------------------------------------------------------

class OracleSample:
    """The float64 oracle's whole pipeline over rows of the workload: mask and
    advantages of the batch, then for a run of rows of the [N, P+C] row space
    (in order, cycling): log-probs, per-token loss terms and dlogits of the
    scored rows, zeros for the rest.  Logits rows come from a seeded CPU pool
    with the workload's distribution."""

    def __init__(self, w: wl.Workload, pool_rows: int = 64):
        import torch
        import oracle
        self.o = oracle.default()
        self.w = w
        self.ids = wl.make_ids(w)
        self.R = wl.make_rewards(w)
        _, self.lens = self.o.mask(self.ids, w.P, w.C, w.eos_id)
        gen = torch.Generator().manual_seed(w.seed + 17)
        x = torch.randn((pool_rows, w.V), generator=gen) * w.logit_std
        x = x.to(torch.bfloat16 if w.dtype == "bf16" else torch.float32)
        self.pool, self.dt = wl.logits_as_numpy(x)
        self.noise_old, self.noise_ref = wl.make_noise(w)
        self.cursor = 0
        self.out = np.zeros(w.V)

    def step(self, nrows: int) -> int:
        """Processes the next nrows rows; returns the valid tokens among them."""
        o, w = self.o, self.w
        _, lens = o.mask(self.ids, w.P, w.C, w.eos_id)
        A = o.advantage(self.R, w.G)
        total = w.N * w.T
        rows = [(self.cursor + k) % total for k in range(nrows)]
        self.cursor = (self.cursor + nrows) % total
        scored = []
        for r in rows:
            i, pos = divmod(r, w.T)
            t = pos - (w.P - 1)
            if 0 <= t < lens[i]:
                scored.append((i, t, r))
            else:
                self.out[:] = 0.0
        if not scored:
            return 0
        z = self.pool[[r % len(self.pool) for _, _, r in scored]]
        y = np.array([self.ids[i, w.P + t] for i, t, _ in scored])
        lp, lse = o.logp_rows(z, self.dt, y)
        n = len(scored)
        old = None if self.noise_old is None else (
            lp + np.array([self.noise_old[i, t] for i, t, _ in scored]))[:, None]
        ref = None if self.noise_ref is None else (
            lp + np.array([self.noise_ref[i, t] for i, t, _ in scored]))[:, None]
        Ai = np.array([A[i] for i, _, _ in scored])
        _, wt, _ = o.loss(lp[:, None], old, ref, Ai, np.ones(n, np.int32), w.eps, w.beta,
                          float(w.N * w.C))
        for k in range(n):
            self.out = o.dlogits_row(z[k], self.dt, int(y[k]), float(lse[k]), float(wt[k, 0]))
        return n


def time_oracle(w: wl.Workload, seconds: float, rows_per_call: int = 32):
    """Runs the oracle on successive row runs until `seconds` have passed."""
    s = OracleSample(w)
    s.step(4)  # load and warm the library
    tokens, rows, t0 = 0, 0, time.perf_counter()
    while True:
        tokens += s.step(rows_per_call)
        rows += rows_per_call
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    import oracle
    return {"value": tokens / el, "unit": UNIT, "cores": oracle.threads(), "kind": "oracle",
            "sample": f"{rows} rows of the [N, P+C] row space of {w.name} in order "
                      f"({tokens} scored tokens, {el:.1f} s): mask, advantage, log-probs, "
                      "loss terms and dlogits in float64"}


def time_oracle_lmhead(w: wl.Workload, d: int, seconds: float, train: bool, rows_per_call: int = 16):
    """The float64 oracle of the LM-head paths on runs of one completion's
    scored rows until `seconds` have passed: log-probs from hidden states (the
    float64 projection, then the row log-softmax), with `train` also the loss
    terms and both gradients.  The head [V, d] is widened to float64 once,
    outside the timed region."""
    import torch
    import oracle
    o = oracle.default()
    hidden = wl.make_hidden(w, d, "cpu")
    weight = wl.make_lm_head(w, d, "cpu")
    Hn = hidden.view(torch.int16).numpy().view(np.uint16)
    W = (weight.view(torch.int16).numpy().view(np.uint16).astype(np.uint32) << 16).view(
        np.float32).astype(np.float64)
    ids = wl.make_ids(w)
    _, lens = o.mask(ids, w.P, w.C, w.eos_id)
    i0 = int(np.argmax(lens))
    k = min(rows_per_call, int(lens[i0]))
    rng = np.random.default_rng(0)
    tokens, calls, t0 = 0, 0, None
    while True:
        t = int(rng.integers(0, int(lens[i0]) - k + 1))
        hs = Hn[i0:i0 + 1, w.P - 1 + t:w.P + t + k]   # rows scoring tokens t .. t+k-1, plus one
        ids_s = ids[i0:i0 + 1, w.P - 1 + t:w.P + t + k]
        ln = np.array([k], np.int32)
        lp, lse = o.lmhead_logp(hs, W, 1, k, ids_s, ln)
        if train:
            _, wt, _ = o.loss(lp, lp - 0.01, None, np.array([0.5]), ln, w.eps, 0.0, float(w.N * w.C))
            o.lmhead_grads(hs, W, 1, k, ids_s, ln, lse, wt)
        if t0 is None:  # the first call warms the libraries
            t0 = time.perf_counter()
            continue
        tokens += k
        calls += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    what = ("log-probs, loss terms, dhidden and dweight" if train else "log-probs")
    return {"value": tokens / el, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{calls} runs of {k} scored rows of {w.name} with hidden size {d} "
                      f"({tokens} tokens, {el:.1f} s): {what} in float64 (numpy matmuls on "
                      f"all cores)"}


# --------------------------------------------------------------------------
# the reference arm: the oracle alone
# --------------------------------------------------------------------------

def run_reference(args, w: wl.Workload):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    s = OracleSample(w)
    # calibrate rows per step so the whole run takes about --reference-seconds
    # (90 s by default): one whole sequence (its prompt rows and its scored
    # rows) gives the mean row cost
    t0 = time.perf_counter()
    s.step(w.T)
    per_row = (time.perf_counter() - t0) / w.T
    total_steps = args.steps + args.warmup
    rows = max(1, int(args.reference_seconds / max(total_steps, 1) / max(per_row, 1e-6)))
    for _ in range(args.warmup):
        s.step(rows)
    tokens = 0
    t0 = time.perf_counter()
    for _ in range(args.steps):
        tokens += s.step(rows)
    el = time.perf_counter() - t0
    value = tokens / el
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * el / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_record(w, args.gpus),
        "workload_stats": {"rows_per_step": rows},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.threads(),
                         "kind": "oracle",
                         "sample": f"{rows} rows of the [N, P+C] row space per step, cycling"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------
# our arm
# --------------------------------------------------------------------------

class Batch:
    """One workload's inputs on the device and the buffers of its step."""

    def __init__(self, g, w: wl.Workload, dev):
        import torch
        self.w = w
        self.ids_np = wl.make_ids(w)
        self.R_np = wl.make_rewards(w)
        tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
        self.logits = torch.empty((w.N, w.T, w.V), dtype=tdt, device=dev)
        wl.fill_logits_cuda(w, self.logits)
        self.ids = torch.from_numpy(self.ids_np).to(dev)
        self.R = torch.from_numpy(self.R_np).to(dev)
        # old/ref log-probs: the current ones (computed by the library) + noise
        self.mask, self.lens = g.grpo_mask(self.ids, w.P, w.C, w.eos_id)
        self.adv = g.grpo_advantage(self.R, w.G)
        cur = g.grpo_loss_fwd(self.logits, w.P, self.ids, self.lens, self.adv)
        n_old, n_ref = wl.make_noise(w)
        self.old = None if n_old is None else (
            cur["logp"] + torch.from_numpy(n_old).float().to(dev)).contiguous()
        self.ref = None if n_ref is None else (
            cur["logp"] + torch.from_numpy(n_ref).float().to(dev)).contiguous()
        self.t_valid = int(self.lens.sum().item())
        _, n_contrast = g.grpo_advantage_ex(self.R, w.G, count_contrast=True)
        self.contrast_groups = int(n_contrast.item())
        # scored rows with a nonzero gradient weight (the only ones a backward
        # that skips zero-weight rows reads)
        wfull = g.grpo_loss_fwd(self.logits, w.P, self.ids, self.lens, self.adv, self.old,
                                self.ref, w.eps, w.beta)["w"]
        self.t_nonzero = int((wfull != 0).sum().item())
        self.dlogits = torch.empty_like(self.logits)
        self.ws = cur["workspace"]
        self.out = None
        self.fout = None

    def step(self, g, path="two_pass", flags=None, record=None, stream=None):
        """One step: grpo_mask -> grpo_advantage -> grpo_loss_fwd ->
        grpo_loss_bwd (path "two_pass"), or the forward and backward in one
        call (path "fused").  record: 4 events around the calls."""
        w = self.w
        if record is not None:
            record[0].record(stream)
        _, ln = g.grpo_mask(self.ids, w.P, w.C, w.eos_id, self.mask, self.lens)
        a = g.grpo_advantage(self.R, w.G, self.adv)
        if record is not None:
            record[1].record(stream)
        if path == "fused":
            self.fout = g.grpo_loss_fwd_bwd(self.logits, w.P, self.ids, ln, a, self.old, self.ref,
                                            w.eps, w.beta, 0.0, None, self.fout, self.ws,
                                            self.dlogits)
            if record is not None:
                record[2].record(stream)
                record[3].record(stream)
            return
        self.out = g.grpo_loss_fwd(self.logits, w.P, self.ids, ln, a, self.old, self.ref, w.eps,
                                   w.beta, 0.0, self.out, self.ws)
        if record is not None:
            record[2].record(stream)
        g.grpo_loss_bwd(self.logits, w.P, self.ids, ln, self.out["lse"], self.out["w"], None,
                        self.dlogits, flags=flags)
        if record is not None:
            record[3].record(stream)

    def free(self):
        import torch
        for k in ("logits", "dlogits", "ids", "R", "mask", "lens", "adv", "old", "ref", "ws",
                  "out", "fout"):
            setattr(self, k, None)
        torch.cuda.empty_cache()


def time_loop(fn, steps: int, stream) -> float:
    """Seconds per call of fn over `steps` back-to-back calls, CUDA events at
    the two ends only (an event between two launches would keep the second
    from starting early)."""
    import torch
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record(stream)
    for _ in range(steps):
        fn()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / 1e3 / steps


def steps_for(ms_estimate: float, steps: int, seconds: float = 1.0) -> int:
    """Timed steps for a secondary measurement: `steps`, fewer when they would
    take longer than `seconds`, at least 5."""
    return max(5, min(steps, int(seconds * 1e3 / max(ms_estimate, 1e-3))))


def path_summary(g, b: Batch, peak: float, steps: int, warmup: int, stream) -> dict:
    """Step time, throughput and roofline fraction of one workload on every
    logits path: the two calls (the method's 2 reads + 1 write), the two calls
    with the zero-weight skip (the skipped reads left out of the byte count),
    and the single-pass call (1 read + 1 write)."""
    w = b.w
    out = {"workload": w.name, "valid_tokens": b.t_valid,
           "nonzero_weight_tokens": b.t_nonzero,
           "groups_with_reward_contrast": b.contrast_groups, "groups": w.B}
    for name, path, flags, t_read in (("two_pass", "two_pass", None, None),
                                      ("skip_zero_weight", "two_pass", 1, b.t_nonzero),
                                      ("fused", "fused", None, None)):
        fn = lambda: b.step(g, path, flags)  # noqa: E731
        for _ in range(max(warmup, 3)):
            fn()
        est = time_loop(fn, 1, stream) * 1e3
        n = steps_for(est, steps)
        t = time_loop(fn, n, stream)
        bb = algorithmic_bytes(w, b.t_valid, t_read)
        nbytes = bb["step_logits_fused"] if path == "fused" else bb["step_logits"]
        out[name] = {"ms_per_step": t * 1e3, "steps": n,
                     "completion_tokens_per_s": b.t_valid / t,
                     "useful_groups_per_s": b.contrast_groups / t,
                     "logits_bytes_per_step": nbytes, "logits_gbs": nbytes / t / 1e9,
                     "logits_roofline_frac": nbytes / t / 1e9 / peak}
    return out


def rank_aggregate(dist, dev, elapsed: float, t_valid: int, contrast: int):
    """Whole-job figures of a weak-scaling run: the slowest rank's time and the
    scored tokens and contrasted groups of all ranks."""
    import torch
    t = torch.tensor([elapsed], device=dev, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    n = torch.tensor([t_valid, contrast], device=dev, dtype=torch.int64)
    dist.all_reduce(n)
    return float(t[0]), int(n[0].item()), int(n[1].item())


def host_mem_available() -> int | None:
    """MemAvailable of the host, in bytes (None where /proc/meminfo is not
    readable)."""
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except (OSError, ValueError, IndexError):
        pass
    return None


def e2e_fits(b: "Batch", world: int, dist) -> tuple[bool, str]:
    """Whether every rank on this host can pin its end-to-end buffers (a host
    copy of the logits and one of the gradient per rank) within 60% of the
    host's available memory; all ranks take the same decision, since the leg
    has collectives inside."""
    import torch
    need = 2 * b.logits.numel() * b.logits.element_size()
    local = int(os.environ.get("LOCAL_WORLD_SIZE", "1"))
    unknown = 1 << 62
    avail = host_mem_available()
    avail = unknown if avail is None else avail
    if world > 1:  # the smallest over the ranks: every rank decides alike
        t = torch.tensor([avail], device=b.logits.device, dtype=torch.int64)
        dist.all_reduce(t, op=dist.ReduceOp.MIN)
        avail = int(t.item())
    ok = avail == unknown or need * local <= 0.6 * avail
    why = ("" if ok else f"{local} rank(s) on a host would pin {need * local / 1e9:.3g} GB of "
           f"host memory, more than 60% of the {avail / 1e9:.3g} GB available there")
    return ok, why


def run_e2e(args, g, b: Batch, stream, world: int, dist) -> dict:
    """The headline metric end to end through the public API, with the
    step's inputs and results in pinned host memory: every step copies the
    ids, rewards and old/reference log-probs in, runs grpo_mask,
    grpo_advantage and grpo_loss_fwd_bwd_host (the single-pass call for
    logits in host memory: only the scored rows cross the host link, into
    the device logits buffer, which serves as its staging buffer, and the
    kernels write the whole dlogits straight into pinned host memory, so the
    gradient crosses the link the other way while the rows arrive), then
    copies logp, w and the loss back."""
    import torch
    w = b.w

    def pinned_like(t):
        h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
        h.copy_(t)
        return h

    h_logits = pinned_like(b.logits)
    h_ids = pinned_like(b.ids)
    h_R = pinned_like(b.R)
    h_old = None if b.old is None else pinned_like(b.old)
    h_ref = None if b.ref is None else pinned_like(b.ref)
    h_dlogits = torch.empty(b.logits.shape, dtype=b.logits.dtype, pin_memory=True)
    h_logp = torch.empty((w.N, w.C), dtype=torch.float32, pin_memory=True)
    h_w = torch.empty((w.N, w.C), dtype=torch.float32, pin_memory=True)
    h_loss = torch.empty((1,), dtype=torch.float32, pin_memory=True)
    e = b.logits.element_size()
    h2d = b.t_valid * w.V * e + sum(t.numel() * t.element_size()
                                    for t in (h_ids, h_R, h_old, h_ref) if t is not None)
    d2h = sum(t.numel() * t.element_size() for t in (h_dlogits, h_logp, h_w, h_loss))
    state = {}

    def enqueue():
        b.ids.copy_(h_ids, non_blocking=True)
        b.R.copy_(h_R, non_blocking=True)
        if h_old is not None:
            b.old.copy_(h_old, non_blocking=True)
        if h_ref is not None:
            b.ref.copy_(h_ref, non_blocking=True)
        _, ln = g.grpo_mask(b.ids, w.P, w.C, w.eos_id, b.mask, b.lens)
        a = g.grpo_advantage(b.R, w.G, b.adv)
        o = g.grpo_loss_fwd_bwd_host(h_logits, w.P, b.ids, ln, a, b.old, b.ref, w.eps, w.beta,
                                     0.0, None, state.get("o"), b.ws, h_dlogits,
                                     staging=b.logits)
        state["o"] = o
        h_logp.copy_(o["logp"], non_blocking=True)
        h_w.copy_(o["w"], non_blocking=True)
        h_loss.copy_(o["loss"], non_blocking=True)

    def eager_step():
        enqueue()
        stream.synchronize()

    for _ in range(2):
        eager_step()
    n = steps_for(time_loop(eager_step, 1, stream) * 1e3, args.e2e_steps, 1.5)

    def timed(step_fn):
        # three timed loops of n steps; the median loop (one host stall would
        # otherwise move a short loop noticeably)
        for _ in range(2):
            step_fn()
        loops = []
        for _ in range(3):
            if world > 1:
                dist.barrier()
            loops.append(time_loop(step_fn, n, stream))
        return sorted(loops)[1]

    eager = timed(eager_step)
    # The same calls captured once into a CUDA graph and replayed each step
    # (one launch instead of the copies and kernels one by one; the host
    # still waits for the results every step).
    graph = None
    try:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            enqueue()
    except Exception as ex:  # capture refused: keep the eager number
        print(f"e2e graph capture failed: {ex!r}", file=sys.stderr)
        graph = None
        torch.cuda.synchronize()

    def graph_step():
        graph.replay()
        stream.synchronize()

    # every rank times a second pass (eager again where capture failed), so
    # all ranks meet the same barriers
    second = timed(graph_step if graph is not None else eager_step)
    graph_used = graph is not None and second <= eager
    best = second if graph_used else eager
    if world > 1:
        t = torch.tensor([best, eager], device=b.logits.device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        best, eager = float(t[0]), float(t[1])
    # the results that came back are the device path's: the loss, and the
    # gradient rows around each completion's first scored row (its last
    # prompt row is zero, the next two score tokens) have the bits of the
    # last device-memory step's dlogits
    ok = bool(torch.equal(h_loss, state["o"]["loss"].cpu()))
    for i in range(w.N):
        rows = slice(max(w.P - 2, 0), w.P + 1)
        ok = ok and bool(torch.equal(h_dlogits[i, rows].to(b.dlogits.device), b.dlogits[i, rows]))
    del graph
    return {"s_per_step": best, "eager_s_per_step": eager, "steps": n,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "cuda_graph": graph_used, "results_match": ok}


def run_ours(args, w0: wl.Workload):
    import torch
    import torch.distributed as dist
    from vocab_wide_logprob_gb300 import build as libbuild
    libbuild.build()
    from vocab_wide_logprob_gb300 import _native as g

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    # weak scaling: each rank holds its own prompt groups (different seeds)
    w = wl.variant(w0, seed=w0.seed + 1000 * rank)
    peaks = measured_peaks()
    peak = peaks.get("hbm_gbs")
    peak_src = "measured" if peak else "fallback"
    peak = peak or FALLBACK_HBM_GBS

    b = Batch(g, w, dev)
    stream = torch.cuda.current_stream()
    fused = args.path == "fused"
    flags = 1 if args.skip_zero_weight else None

    def step(record=None):
        b.step(g, args.path, flags, record, stream)

    gpu_id = None
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        gpu_id = None
    sampler = None if args.no_clocks else ClockSampler(gpu_id)
    if sampler is not None:
        time.sleep(1.0)  # nvidia-smi needs a moment before its first sample
    for _ in range(max(args.warmup, 3)):
        step()
    assert g.grpo_check_error(b.ws) == 0
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    start.record(stream)
    for k in range(args.steps):
        step()
    end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = sampler.stop() if sampler is not None else None
    elapsed = start.elapsed_time(end) / 1e3

    # Per-call times, from a separate run with an event between the calls
    # (outside the timed region: an event between two launches keeps the
    # second from starting early, so these calls run one after the other).
    n_inst = max(3, min(args.steps, 50))
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n_inst)]
    for k in range(n_inst):
        step(events[k])
    torch.cuda.synchronize()
    t_mask = statistics.mean(e[0].elapsed_time(e[1]) for e in events) / 1e3
    t_fwd = statistics.mean(e[1].elapsed_time(e[2]) for e in events) / 1e3
    t_bwd = statistics.mean(e[2].elapsed_time(e[3]) for e in events) / 1e3
    res = b.fout if fused else b.out
    loss_val = float(res["loss"].item())
    t_valid, t_nonzero, contrast = b.t_valid, b.t_nonzero, b.contrast_groups

    # every logits path on the same inputs, for the record (each against its
    # own byte count)
    paths = None
    if args.also_other_path and world == 1:
        paths = path_summary(g, b, peak, args.steps, args.warmup, stream)

    e2e, e2e_skipped = None, None
    if not args.no_e2e:
        fits, why = e2e_fits(b, world, dist)
        if fits:
            e2e = run_e2e(args, g, b, stream, world, dist)
        else:
            e2e_skipped = why
    inputs = input_record(w, b.ids_np, b.R_np, b.logits)

    # the other workloads of the benchmark plan, one at a time, after this
    # workload's buffers are released
    per_config = None
    if world == 1 and args.per_config != "none":
        names = ([c.name for c in wl.CONFIGS[1:] if c.name != w0.name]
                 if args.per_config == "auto" else args.per_config.split(","))
        b.free()
        per_config = {}
        for name in names:
            bc = Batch(g, wl.BY_NAME[name], dev)
            per_config[name] = path_summary(g, bc, peak, args.steps, args.warmup, stream)
            per_config[name]["inputs"] = input_record(bc.w, bc.ids_np, bc.R_np, bc.logits)
            bc.free()
    b = None

    # aggregate over ranks: units of all ranks / max time
    if world > 1:
        elapsed, t_valid_all, contrast_all = rank_aggregate(dist, dev, elapsed, t_valid, contrast)
    else:
        t_valid_all, contrast_all = t_valid, contrast

    copy_gbs = None if args.no_copy_ceiling else copy_ceiling(g, dev)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = time_oracle(w, args.cpu_seconds)
        # the same oracle on one core, for the record (a shorter sample)
        import oracle
        n_threads = oracle.threads()
        oracle.set_threads(1)
        try:
            one = time_oracle(w, max(1.0, args.cpu_seconds / 4), rows_per_call=8)
        finally:
            oracle.set_threads(n_threads)
        cpu["single_core"] = {"value": one["value"], "cores": 1, "sample": one["sample"]}
        cpu["cpu_model"] = cpu_model()

    if rank == 0:
        bb = algorithmic_bytes(w, t_valid, t_nonzero if args.skip_zero_weight else None)
        ms = elapsed / args.steps
        if fused:
            # the fused call: prep + zero-row writer + lse_grad_kernel, timed together
            step_bytes = bb["step_logits_fused"]
            kernel, kbytes, kt = "grpo_loss_fwd_bwd", bb["fused"], t_fwd
        else:
            step_bytes = bb["step_logits"]
            kernel, kbytes, kt = "dlogits_kernel", bb["bwd"], t_bwd
        achieved = kbytes / kt / 1e9
        traffic = recorded_traffic(kernel, w)
        line = {
            "metric": METRIC, "value": t_valid_all / ms, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16"
            if w.dtype == "bf16" else "f32", "data": "synthetic",
            "config": config_record(w0, world),
            "path": args.path,
            "workload_stats": {"valid_tokens_per_rank": t_valid,
                               "nonzero_weight_tokens_per_rank": t_nonzero,
                               "groups_with_reward_contrast_per_rank": contrast,
                               "groups_per_rank": w.B,
                               "skip_zero_weight": bool(args.skip_zero_weight)},
            "useful_groups_per_s": contrast_all / ms,
            "logits_gbs": step_bytes / ms / 1e9,
            "logits_roofline_frac": step_bytes / ms / 1e9 / peak,
            "logits_bytes_per_step": step_bytes,
            "kernel_ms": {"mask+advantage": t_mask * 1e3, "fwd": t_fwd * 1e3,
                          "bwd": t_bwd * 1e3},
            "kernel_timing": f"CUDA events between the calls over {n_inst} further steps on the "
                             "launching stream (the headline loop has events only at its ends)",
            "fwd_gbs": (bb["fused"] if fused else bb["fwd"]) / t_fwd / 1e9,
            "roofline": {"kernel": kernel, "bound": "hbm", "achieved": achieved,
                         "peak": peak, "peak_source": peak_src, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic,
                         "algorithmic_bytes": kbytes},
            "e2e": ({"value": None, "unit": UNIT, "skipped": e2e_skipped}
                    if e2e_skipped is not None else None) if e2e is None else {
                "value": t_valid_all / e2e["s_per_step"], "unit": UNIT,
                "h2d_bytes_per_step": e2e["h2d_bytes_per_step"],
                "d2h_bytes_per_step": e2e["d2h_bytes_per_step"],
                "path": "the single-pass call for host buffers: grpo_mask + grpo_advantage + "
                        "grpo_loss_fwd_bwd_host (logits in pinned host memory, only the scored "
                        "rows cross the host link; the kernels write the whole dlogits into "
                        "pinned host memory across the link), then logp, w and the loss copied "
                        "back",
                "cuda_graph": e2e["cuda_graph"], "steps": e2e["steps"],
                "eager_value": t_valid_all / e2e["eager_s_per_step"],
                "results_match": e2e["results_match"]},
            "copy_ceiling_gbs": copy_gbs,
            "paths": paths,
            "per_config": per_config,
            "gpu_launches": (KERNELS_PER_STEP - 1 if fused else KERNELS_PER_STEP) * args.steps,
            "cpu_baseline": cpu,
            "clocks": clocks,
            "loss": loss_val,
            "logits_nominal_frac": step_bytes / ms / 1e9 / NOMINAL_HBM_GBS,
            "inputs": inputs,
            "env": run_env(dev),
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def run_lmhead(args, w: wl.Workload):
    """--path lmhead_logprobs: grpo_mask + grpo_lmhead_logprobs (log-probs of
    the sampled tokens from hidden states [N, P+C, d] and a [V, d] LM head,
    logits never materialised; 2 * T_valid * V * d FLOPs per step).
    --path lmhead_fwd_bwd: grpo_mask + grpo_advantage + grpo_lmhead_loss_fwd +
    grpo_lmhead_loss_bwd (the projection in the forward, its recomputation in
    the backward, and the two gradient contractions: 4 * 2 * T_valid * V * d
    FLOPs per step).  Roofline: tensor."""
    import torch
    from vocab_wide_logprob_gb300 import build as libbuild
    libbuild.build()
    from vocab_wide_logprob_gb300 import _native as g
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    train = args.path == "lmhead_fwd_bwd"
    d = args.hidden
    hidden = wl.make_hidden(w, d, "cuda")
    weight = wl.make_lm_head(w, d, "cuda")
    ids = torch.from_numpy(wl.make_ids(w)).to(dev)
    R = torch.from_numpy(wl.make_rewards(w)).to(dev)
    mask, lens = g.grpo_mask(ids, w.P, w.C, w.eos_id)
    t_valid = int(lens.sum().item())
    lp, lse, ws = g.grpo_lmhead_logprobs(hidden, weight, w.P, ids, lens)
    stream = torch.cuda.current_stream()
    old = ref = None
    if train:
        # old / reference log-probs: this policy's log-probs plus the workload's noise
        n_old, n_ref = wl.make_noise(w)
        if n_old is not None:
            old = (lp + torch.from_numpy(n_old).float().to(dev)).contiguous()
        if n_ref is not None:
            ref = (lp + torch.from_numpy(n_ref).float().to(dev)).contiguous()
        adv = g.grpo_advantage(R, w.G)
        fwd = g.grpo_lmhead_loss_fwd(hidden, weight, w.P, ids, lens, adv, old, ref, w.eps, w.beta)
        bflags = 1 if args.skip_zero_weight else None
        # the backward's workspace sized by the scored rows actually present
        # (one pass over them), not by every possible row
        dh, dw, bws = g.grpo_lmhead_loss_bwd(hidden, weight, w.P, ids, lens, fwd["lse"], fwd["w"],
                                             flags=bflags,
                                             rows_per_pass=(t_valid if args.lmhead_rows_per_pass < 0
                                                            else args.lmhead_rows_per_pass))
        bwd_ws_bytes = bws.numel()
        bwd_passes = lmhead_bwd_passes(w, t_valid if args.lmhead_rows_per_pass < 0
                                       else args.lmhead_rows_per_pass)
        bwd_ws_full = g.grpo_lmhead_bwd_workspace_size(w.N, w.C, w.V, d)
        t_nonzero = int((fwd["w"] != 0).sum().item())

    def step_fwd():
        g.grpo_mask(ids, w.P, w.C, w.eos_id, mask, lens)
        if train:
            g.grpo_advantage(R, w.G, adv)
            g.grpo_lmhead_loss_fwd(hidden, weight, w.P, ids, lens, adv, old, ref, w.eps, w.beta,
                                   out=fwd, workspace=ws)
        else:
            g.grpo_lmhead_logprobs(hidden, weight, w.P, ids, lens, (lp, lse), ws)

    def step_bwd():
        if train:
            g.grpo_lmhead_loss_bwd(hidden, weight, w.P, ids, lens, fwd["lse"], fwd["w"],
                                   out=(dh, dw), workspace=bws, flags=bflags)

    def step():
        step_fwd()
        step_bwd()

    sampler = None if args.no_clocks else ClockSampler(None)
    if sampler is not None:
        time.sleep(1.0)
    for _ in range(max(args.warmup, 3)):
        step()
    assert g.grpo_check_error(fwd["workspace"] if train else ws) == 0
    if train:
        assert g.grpo_check_error(bws) == 0
    torch.cuda.synchronize()

    def timed(fn):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record(stream)
        for _ in range(args.steps):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / args.steps

    ms = timed(step)
    clocks = sampler.stop() if sampler is not None else None
    ms_fwd = timed(step_fwd) if train else ms
    ms_bwd = timed(step_bwd) if train else 0.0
    unit_flops = 2.0 * t_valid * w.V * d
    # the backward recomputes the projection and runs both contractions over its rows:
    # every scored row, or with --skip-zero-weight those whose gradient weight is not 0
    bwd_rows = (t_nonzero if args.skip_zero_weight else t_valid) if train else 0
    flops = unit_flops + 3 * 2.0 * bwd_rows * w.V * d
    peaks = measured_peaks()
    burst = peaks.get("bf16_tflops") or 1900.0
    # the burst peak for a short timed loop, the sustained one (a seconds-long
    # GEMM loop under the power cap) when the loop is as long or the clocks
    # sampled during it show the power cap
    sustained_run = (args.steps * ms >= 1000.0 or
                     (clocks is not None and "sw_power_cap" in (clocks.get("reasons") or [])))
    peak_kind = "sustained" if sustained_run and peaks.get("bf16_tflops_sustained") else "burst"
    peak = peaks["bf16_tflops_sustained"] if peak_kind == "sustained" else burst
    tflops = flops / (ms * 1e-3) / 1e12
    line = {
        "metric": ("completion tokens/s, Dr. GRPO loss fwd+bwd from hidden states (LM head "
                   "fused: logits never materialised)") if train else
                  "completion tokens/s, log-probs from hidden states (LM head fused, no grad)",
        "value": t_valid / (ms * 1e-3), "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "path": args.path,
        "config": {"workload": w.name, "B": w.B, "G": w.G, "P": w.P, "C": w.C, "V": w.V,
                   "hidden": d, "valid_tokens": t_valid,
                   "l2": "weights larger than L2 (%.2f GB); no flush" % (w.V * d * 2 / 1e9)},
        "roofline": {"kernel": ("lmhead fwd + bwd (projection, recomputed projection, "
                                "dhidden and dweight contractions)") if train else
                               "lmhead_lse_kernel (+ gather)",
                     "bound": "tensor", "achieved": tflops, "peak": peak,
                     "peak_source": "measured" if peaks.get("bf16_tflops") else "fallback",
                     "peak_kind": peak_kind, "frac_of_burst_peak": tflops / burst,
                     "unit": "TFLOP/s", "frac": tflops / peak, "flops_per_step": flops,
                     "traffic": recorded_traffic("lmhead_fwd_bwd" if train else
                                                 "lmhead_lse_kernel", w, d)},
        # per step: mask, prep, gather, log-sum-exp (+ advantage, surrogate, and
        # the backward's prep, row scan and gather, then per pass its
        # logits-gradient, dhidden, dweight and reduce kernels)
        "gpu_launches": ((9 + 4 * bwd_passes) if train else 4) * args.steps, "clocks": clocks,
        "cpu_baseline": None if args.no_cpu_baseline else
        time_oracle_lmhead(w, d, args.cpu_seconds, train),
    }
    line["env"] = run_env(torch.device("cuda", 0))
    if train:
        line["kernel_ms"] = {"fwd": ms_fwd, "bwd": ms_bwd}
        line["fwd_tflops"] = unit_flops / (ms_fwd * 1e-3) / 1e12
        line["bwd_tflops"] = 3 * 2.0 * bwd_rows * w.V * d / (ms_bwd * 1e-3) / 1e12
        line["config"]["nonzero_weight_tokens"] = t_nonzero
        line["config"]["skip_zero_weight"] = bool(args.skip_zero_weight)
        line["bwd_workspace_bytes"] = bwd_ws_bytes
        line["bwd_workspace_bytes_every_possible_row"] = bwd_ws_full
        line["bwd_passes"] = bwd_passes
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    w = wl.BY_NAME[args.workload]
    if args.impl == "reference":
        run_reference(args, w)
    elif args.path in ("lmhead_logprobs", "lmhead_fwd_bwd"):
        run_lmhead(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
