"""Seeded synthetic inputs for the optimizer-step workloads.

This module only draws inputs (tensor sizes, parameters, gradients, initial
states); it holds none of the optimizer's arithmetic.  Both the CUDA library
(through tests and bench.py) and the CPU oracle (through tests) are fed from
here, so the two always see the same bytes.  torch's seeded generators are
used on either device; a given (seed, device) always yields the same inputs.

Workloads (sizes and distributions follow the configurations that stand in
for the pages' measurements):

* ``adamw_1m``      one fp32 tensor of 1,048,576, fp32 grads N(0,1) fresh each
                    step, lr = wd = 0.1, 10 steps, no clipping.
* ``clip_740``      740 tensors with sizes log-uniform in [1, 4M]; BF16 grads
                    N(0,1) * per-tensor scale log-uniform in [1e-4, 10];
                    clip max_norm 1.0; lr 1e-3, wd 0.01; 20 steps.
* ``ademamix_gpt2`` GPT-2-small list (148 tensors, 124,439,808 params), fp32
                    grads N(0, 1e-2^2), three fp32 states, alpha 5, b3 0.9999,
                    lr 1e-3, wd 0.1; 50 steps.
* ``lowp_gpt2``     same list, BF16 grads N(0, s_t^2) with s_t falling 10x
                    linearly over 1,000 steps; BF16 m; v BF16 / E4M3 / E2M2.
* ``llama3_8b``     Llama-3-8B list (291 tensors, 8,030,261,248 params), BF16
                    grads N(0, 1e-3^2), fp32 m/v, lr 3e-4, wd 0.1, clip 1.0;
                    5 steps.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch


# ---------------------------------------------------------------- tensor lists
def gpt2_small_sizes() -> list[int]:
    d, v, ctx, layers = 768, 50257, 1024, 12
    sizes = [v * d, ctx * d]
    for _ in range(layers):
        sizes += [d, d,                       # ln_1 weight, bias
                  d * 3 * d, 3 * d,           # attn c_attn weight, bias
                  d * d, d,                   # attn c_proj weight, bias
                  d, d,                       # ln_2 weight, bias
                  d * 4 * d, 4 * d,           # mlp c_fc weight, bias
                  4 * d * d, d]               # mlp c_proj weight, bias
    sizes += [d, d]                           # ln_f weight, bias
    return sizes


def llama3_8b_sizes() -> list[int]:
    h, kv, ff, vocab, layers = 4096, 1024, 14336, 128256, 32
    sizes = [vocab * h]
    for _ in range(layers):
        sizes += [h * h, kv * h, kv * h, h * h,    # q, k, v, o
                  ff * h, ff * h, h * ff,          # gate, up, down
                  h, h]                            # two RMSNorm weights
    sizes += [h, vocab * h]                        # final norm, untied head
    return sizes


def loguniform_sizes(n: int = 740, max_numel: int = 1 << 22, seed: int = 740) -> list[int]:
    rng = np.random.default_rng(seed)
    raw = np.exp(rng.uniform(0.0, math.log(max_numel), n))
    return [max(1, int(round(x))) for x in raw]


# The size sweep of "Investigate SM103 bias-correction broadcast in 32-bit
# optimizers" ('Correctness oracle'): tile edges and ragged tails.
SWEEP_SIZES = [1, 2, 3, 7, 8, 9, 255, 256, 257, 4095, 4096, 4097, 8191, 8192, 8193,
               32767, 32768, 32769, 65536, 65539, 100003]


@dataclass
class Workload:
    name: str
    sizes: list[int]
    grad_dtype: str                 # "bf16" or "f32"
    m_dtype: str = "f32"
    v_dtype: str = "f32"
    algo: str = "adamw"             # or "ademamix"
    steps: int = 1
    max_norm: float = 0.0           # <= 0: no clipping
    p_std: float = 0.02
    grad_std: float = 1.0
    grad_scales: list[float] | None = None   # per-tensor multipliers
    hp: dict = field(default_factory=dict)
    sigma_decay_steps: int = 0      # >0: grad std falls 10x linearly over this many steps

    @property
    def numel(self) -> int:
        return sum(self.sizes)

    def grad_std_at(self, step: int) -> float:
        if self.sigma_decay_steps <= 0:
            return self.grad_std
        t = min(step, self.sigma_decay_steps)
        return self.grad_std * (1.0 - 0.9 * (t - 1) / (self.sigma_decay_steps - 1))


def workload(name: str, **over) -> Workload:
    if name == "adamw_1m":
        w = Workload(name, [1 << 20], "f32", steps=10, p_std=0.02, grad_std=1.0,
                     hp=dict(lr=0.1, weight_decay=0.1, beta1=0.9, beta2=0.999, eps=1e-8))
    elif name == "clip_740":
        sizes = loguniform_sizes()
        rng = np.random.default_rng(741)
        scales = list(np.exp(rng.uniform(math.log(1e-4), math.log(10.0), len(sizes))))
        w = Workload(name, sizes, "bf16", steps=20, max_norm=1.0, p_std=0.02, grad_std=1.0,
                     grad_scales=scales, hp=dict(lr=1e-3, weight_decay=0.01))
    elif name == "ademamix_gpt2":
        w = Workload(name, gpt2_small_sizes(), "f32", algo="ademamix", steps=50, p_std=0.02,
                     grad_std=1e-2, hp=dict(lr=1e-3, weight_decay=0.1, beta1=0.9, beta2=0.999,
                                            beta3=0.9999, alpha=5.0))
    elif name == "lowp_gpt2":
        w = Workload(name, gpt2_small_sizes(), "bf16", m_dtype="bf16", v_dtype="bf16", steps=1000,
                     p_std=0.02, grad_std=1.0, sigma_decay_steps=1000,
                     hp=dict(lr=1e-3, weight_decay=0.1, beta1=0.9, beta2=0.999))
    elif name == "llama3_8b":
        w = Workload(name, llama3_8b_sizes(), "bf16", steps=5, max_norm=1.0, p_std=0.02,
                     grad_std=1e-3, hp=dict(lr=3e-4, weight_decay=0.1, beta1=0.9, beta2=0.999))
    elif name == "sweep":
        w = Workload(name, list(SWEEP_SIZES), "bf16", steps=3, max_norm=1.0, p_std=0.02,
                     grad_std=1.0, hp=dict(lr=1e-2, weight_decay=0.1))
    else:
        raise KeyError(name)
    for k, v in over.items():
        setattr(w, k, v)
    return w


# ------------------------------------------------------------------- tensors
_TORCH = {"f32": torch.float32, "bf16": torch.bfloat16}


def state_storage(dtype: str, n: int, device) -> torch.Tensor:
    """Zero-initialised storage for n elements of a state dtype (raw codes for
    the low-precision formats; zero is the code of 0.0 in all of them)."""
    if dtype == "f32":
        return torch.zeros(n, dtype=torch.float32, device=device)
    if dtype == "bf16":
        return torch.zeros(n, dtype=torch.int16, device=device)
    if dtype == "e4m3":
        return torch.zeros(n, dtype=torch.uint8, device=device)
    if dtype == "e2m2":
        return torch.zeros((n + 1) // 2, dtype=torch.uint8, device=device)
    raise KeyError(dtype)


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) & 0x7FFFFFFFFFFFFFFF)
    return g


def make_params(w: Workload, device, seed: int = 0, indices=None) -> list[torch.Tensor]:
    idx = range(len(w.sizes)) if indices is None else indices
    out = []
    for i in idx:
        g = _gen(device, seed * 1_000_003 + i)
        out.append(torch.empty(w.sizes[i], dtype=torch.float32, device=device).normal_(0.0, w.p_std, generator=g))
    return out


def fill_grads(w: Workload, grads, step: int, seed: int = 0, indices=None) -> None:
    """Overwrite gradient tensors (list aligned with `indices`) with the
    gradients of `step` (1-based); fresh draws every step."""
    idx = range(len(w.sizes)) if indices is None else indices
    std = w.grad_std_at(step)
    for t, i in zip(grads, idx):
        g = _gen(t.device, (seed + 7919) * 1_000_003 + step * 65_537 + i)
        s = std * (w.grad_scales[i] if w.grad_scales is not None else 1.0)
        if t.dtype == torch.bfloat16:
            # draw in fp32, round once to BF16 (nearest-even)
            tmp = torch.empty(t.numel(), dtype=torch.float32, device=t.device).normal_(0.0, s, generator=g)
            t.copy_(tmp)
        else:
            t.normal_(0.0, s, generator=g)


def make_grads(w: Workload, device, step: int = 1, seed: int = 0, indices=None) -> list[torch.Tensor]:
    idx = range(len(w.sizes)) if indices is None else list(indices)
    grads = [torch.empty(w.sizes[i], dtype=_TORCH[w.grad_dtype], device=device) for i in idx]
    fill_grads(w, grads, step, seed, idx)
    return grads


def inject_nonfinite(grads, seed: int = 13, frac: float = 0.01, kinds=("nan", "+inf", "-inf")):
    """Put NaN / +Inf / -Inf at three seeded positions in 1% of the tensors
    (at least one).  Returns the indices of the tensors touched."""
    rng = np.random.default_rng(seed)
    k = max(1, int(round(frac * len(grads))))
    chosen = sorted(rng.choice(len(grads), size=k, replace=False).tolist())
    vals = {"nan": float("nan"), "+inf": float("inf"), "-inf": float("-inf")}
    for i in chosen:
        t = grads[i]
        for j, kind in enumerate(kinds):
            pos = int(rng.integers(0, t.numel()))
            t.view(-1)[pos] = vals[kind]
    return chosen


def to_numpy_codes(t: torch.Tensor) -> np.ndarray:
    """Host numpy view for the oracle: float32 stays float32, BF16 / int16
    storage becomes uint16 codes, uint8 stays uint8."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    if t.dtype == torch.int16:
        return t.numpy().view(np.uint16).copy()
    return t.numpy().copy()
