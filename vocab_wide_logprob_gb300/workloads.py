"""Seeded synthetic inputs for the Dr. GRPO loss path.

This module only draws random inputs; it holds none of the method's
arithmetic (no mask, no advantage, no log-softmax, no loss).  Both the CUDA
path's tests/benchmark and the CPU oracle consume what it produces.

The shapes follow the setup of "Making Dr GRPO go brrr" (salahadawi.com):
Qwen2.5-0.5B-Instruct (vocabulary V = 151936), B prompts each sampled G times
("Sample G completions for the same prompt"; prompts repeated with
``repeat_interleave`` so completions b*G .. b*G+G-1 share prompt b), a prompt
of P tokens followed by a completion of C tokens, full-sequence logits
[B*G, P+C, V].  ``generate`` pads with EOS after a completion finishes, so
every position after the first EOS holds EOS; a truncated completion holds no
EOS at all.  Rewards are binary verifier outcomes (page 1, "The sparse-reward
bottleneck": reward 1 with probability p, else 0).

Recipe (stated once here, used everywhere):
  * prompt ids: uniform in [0, V) (EOS allowed: the mask reads completion
    columns only);
  * completion: a truncated draw comes first (Bernoulli(trunc)); a truncated
    completion holds C ids uniform in [0, V) minus {EOS}; otherwise a length L
    is drawn, ids 0..L-2 uniform in [0, V) minus {EOS}, EOS at L-1 and at every
    later position;
  * length draws: "uniform" L ~ U{1..C}; "geometric" L ~ Geometric(1/mean) on
    {1, 2, ...} and L > C means truncated (no separate truncation draw);
  * rewards: Bernoulli(p) per completion, p fixed or p ~ U(lo, hi) per prompt;
  * logits: N(0, std^2) float32 from torch's seeded generator, then rounded
    to the logits dtype;
  * old / reference log-prob noise: N(0, sigma^2) float64 per token; the
    caller adds it to the current log-probs.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace

import numpy as np

QWEN25_VOCAB = 151936
# <|im_end|>, the end-of-turn token Qwen2.5-Instruct stops generation with
QWEN25_EOS = 151645


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    G: int
    P: int
    C: int
    V: int
    dtype: str              # "f32" or "bf16"
    logit_std: float
    eos_id: int
    reward_p: float = 0.05  # Bernoulli success probability (fixed)
    reward_p_range: tuple | None = None  # per-prompt p ~ U(lo, hi) instead
    length: str = "uniform"  # "uniform" or "geometric"
    trunc: float = 0.0      # probability a completion is truncated (uniform)
    geo_mean: float = 300.0
    old_sigma: float | None = None  # None: old log-probs equal current ones
    ref_sigma: float | None = None  # None: no reference log-probs
    beta: float = 0.0
    eps: float = 0.2
    seed: int = 1000
    special: str = ""       # "tiny": plant the edge cases of the tiny case
    forced: dict = field(default_factory=dict)

    @property
    def N(self) -> int:
        return self.B * self.G

    @property
    def T(self) -> int:
        return self.P + self.C

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    @property
    def logits_bytes(self) -> int:
        return self.N * self.T * self.V * self.elem_bytes


# The five workloads of the benchmark plan, in order.
TINY = Workload("tiny_N8_P16_C32_V1024_f32", B=2, G=4, P=16, C=32, V=1024, dtype="f32",
                logit_std=2.0, eos_id=2, reward_p=0.3, length="uniform", old_sigma=None,
                beta=0.0, eps=0.2, seed=1001, special="tiny")
QWEN_G8 = Workload("qwen05b_N8_P128_C256_bf16", B=1, G=8, P=128, C=256, V=QWEN25_VOCAB,
                   dtype="bf16", logit_std=3.0, eos_id=QWEN25_EOS, reward_p=0.05,
                   length="uniform", trunc=0.20, old_sigma=0.05, beta=0.0, eps=0.2, seed=1002)
QWEN_G16_KL = Workload("qwen05b_N16_P256_C512_bf16_kl", B=1, G=16, P=256, C=512,
                       V=QWEN25_VOCAB, dtype="bf16", logit_std=3.0, eos_id=QWEN25_EOS,
                       reward_p=0.05, length="uniform", trunc=0.25, old_sigma=0.1,
                       ref_sigma=0.1, beta=0.04, eps=0.2, seed=1003)
BATCHED = Workload("batched_N64_P256_C1024_bf16", B=8, G=8, P=256, C=1024, V=QWEN25_VOCAB,
                   dtype="bf16", logit_std=3.0, eos_id=QWEN25_EOS, reward_p_range=(0.0, 0.5),
                   length="geometric", geo_mean=300.0, old_sigma=0.05, beta=0.0, eps=0.2,
                   seed=1004)
LONG = Workload("long_N32_P512_C3584_bf16_kl", B=4, G=8, P=512, C=3584, V=QWEN25_VOCAB,
                dtype="bf16", logit_std=3.0, eos_id=QWEN25_EOS, reward_p=0.05,
                length="uniform", trunc=0.30, old_sigma=0.1, ref_sigma=0.1, beta=0.04,
                eps=0.2, seed=1005)

CONFIGS = [TINY, QWEN_G8, QWEN_G16_KL, BATCHED, LONG]
BY_NAME = {w.name: w for w in CONFIGS}


def variant(w: Workload, **kw) -> Workload:
    """A copy of ``w`` with some fields changed (edge-case shapes in tests)."""
    return replace(w, **kw)


def _rng(w: Workload, stream: int) -> np.random.Generator:
    return np.random.default_rng([w.seed, stream])


def _non_eos(rng, n, V, eos):
    """n ids uniform in [0, V) minus {eos} (V >= 2)."""
    x = rng.integers(0, V - 1, size=n, dtype=np.int64)
    return x + (x >= eos)


def completion_lengths(w: Workload) -> np.ndarray:
    """Per completion: the index of its first EOS plus one, or 0 when the
    completion is truncated (no EOS).  This is the generator's own plan; the
    tests never use it as an expected value."""
    rng = _rng(w, 1)
    N, C = w.N, w.C
    L = np.zeros(N, np.int64)
    for i in range(N):
        if w.length == "geometric":
            li = int(rng.geometric(1.0 / w.geo_mean))
            L[i] = li if li <= C else 0
        else:
            truncated = rng.random() < w.trunc
            li = int(rng.integers(1, C + 1))
            L[i] = 0 if truncated else li
    if w.special == "tiny" and N >= 3 and C >= 2:
        L[0] = 0   # no EOS at all: the argmax-returns-0 trap
        L[1] = 2   # a one-token answer: one content token, then EOS
        L[2] = 1   # EOS as the very first token
    for i, li in w.forced.get("lengths", {}).items():
        L[i] = li
    return L


def make_ids(w: Workload) -> np.ndarray:
    """input_ids [N, P+C] int64: prompt b (uniform ids) repeated for its G
    completions, then each completion per the recipe."""
    rng = _rng(w, 2)
    N, P, C, V, eos = w.N, w.P, w.C, w.V, w.eos_id
    ids = np.empty((N, P + C), np.int64)
    prompts = rng.integers(0, V, size=(w.B, P), dtype=np.int64)
    ids[:, :P] = np.repeat(prompts, w.G, axis=0)
    L = completion_lengths(w)
    for i in range(N):
        if L[i] == 0:
            ids[i, P:] = _non_eos(rng, C, V, eos)
        else:
            li = int(L[i])
            ids[i, P:P + li - 1] = _non_eos(rng, li - 1, V, eos)
            ids[i, P + li - 1:] = eos
    return ids


def make_rewards(w: Workload) -> np.ndarray:
    """Binary rewards [N] float32, Bernoulli per completion.  The tiny case
    forces group 1 to all ones (a uniform group, no contrast) and redraws
    group 0 until it has contrast."""
    rng = _rng(w, 3)
    N, G = w.N, w.G
    if w.reward_p_range is not None:
        lo, hi = w.reward_p_range
        p = np.repeat(rng.uniform(lo, hi, size=w.B), G)
    else:
        p = np.full(N, w.reward_p)
    R = (rng.random(N) < p).astype(np.float32)
    if w.special == "tiny" and w.B >= 2 and G >= 2:
        R[G:2 * G] = 1.0
        while R[:G].min() == R[:G].max():
            R[:G] = (rng.random(G) < p[:G]).astype(np.float32)
    if "rewards" in w.forced:
        R[:] = np.asarray(w.forced["rewards"], np.float32)
    return R


def make_noise(w: Workload):
    """(old_noise, ref_noise): float64 [N, C] N(0, sigma^2) arrays, or None
    when the workload has no such input.  Old log-probs are current + noise;
    reference log-probs are current + noise."""
    rng = _rng(w, 4)
    old = None if w.old_sigma is None else rng.normal(0.0, w.old_sigma, size=(w.N, w.C))
    ref = None if w.ref_sigma is None else rng.normal(0.0, w.ref_sigma, size=(w.N, w.C))
    return old, ref


def _torch_dtype(w: Workload):
    import torch
    return torch.float32 if w.dtype == "f32" else torch.bfloat16


def make_logits_cpu(w: Workload):
    """Logits [N, P+C, V] as a CPU torch tensor (small workloads)."""
    import torch
    g = torch.Generator().manual_seed(w.seed)
    x = torch.randn((w.N, w.T, w.V), generator=g, dtype=torch.float32) * w.logit_std
    return x.to(_torch_dtype(w))


def fill_logits_cuda(w: Workload, out) -> None:
    """Fills the device tensor ``out`` [N, P+C, V] one sequence at a time from
    torch's seeded CUDA generator (keeps the float32 temporary small)."""
    import torch
    g = torch.Generator(device=out.device).manual_seed(w.seed)
    for i in range(w.N):
        x = torch.randn((w.T, w.V), generator=g, device=out.device, dtype=torch.float32)
        out[i].copy_(x.mul_(w.logit_std))
        del x


def make_hidden(w: Workload, d: int, device="cpu"):
    """Last hidden states [N, P+C, d] bfloat16 ~ N(0, 1) (seeded), for the
    LM-head path."""
    import torch
    g = torch.Generator(device=device).manual_seed(w.seed + 7)
    x = torch.randn((w.N, w.T, d), generator=g, device=device, dtype=torch.float32)
    return x.to(torch.bfloat16)


def make_lm_head(w: Workload, d: int, device="cpu"):
    """LM-head weight [V, d] bfloat16 ~ N(0, (std / sqrt(d))^2), so that the
    logits hidden x W^T have the workload's logit standard deviation."""
    import torch
    g = torch.Generator(device=device).manual_seed(w.seed + 9)
    x = torch.randn((w.V, d), generator=g, device=device, dtype=torch.float32)
    return x.mul_(w.logit_std / d ** 0.5).to(torch.bfloat16)


def logits_as_numpy(t):
    """(numpy array, dtype tag) of a CPU tensor: float32 as is, bfloat16 as its
    uint16 bit patterns."""
    import torch
    t = t.contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16), "bf16"
    if t.dtype == torch.float32:
        return t.numpy(), "f32"
    raise TypeError(f"unsupported logits dtype {t.dtype}")
