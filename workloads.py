"""Seeded synthetic inputs for the MoE layer forward.

This module only draws numbers. It holds none of the layer's arithmetic:
no routing, no softmax, no capacity rule, no GEMM. Both the CPU oracle
(through the tests) and the CUDA library (through the tests, ``bench.py``
and ``smoke()``) receive the very same tensors from here.

Workloads
---------
The five named workloads are the layer shapes this library is measured and
checked on. The large-expert one is the worked example of the MoE
communication-bottleneck page, section 2.2 (H=4096, expert width 14336,
8 experts, top-2, sequence 4096 x micro-batch 8). The others stress skew
(a Zipf-like logit bias, section 3.1 of the same page: a few experts take
most tokens, capacity forces drops), many small segments (64 experts, top-6)
and many experts with a random bias that leaves about a third of them idle.

Distributions (read "N(0, s2)" as variance s2):
  tokens x ~ N(0, 1); gate ~ N(0, 1/H); W1 ~ N(0, 1/H); W2 ~ N(0, 1/h);
  imbalanced bias b_e = 2 ln(1/(e+1)); many-expert bias ~ N(0, 1.5).
Every draw is fp32 ``torch.randn`` from one ``torch.Generator`` seeded with
``seed``, scaled by the standard deviation and rounded to bf16 (RNE), in
the fixed order x, gate, bias, W1, W2. Large tensors are drawn in fixed
chunks (x by 16384-row blocks, W1/W2 one expert at a time) so host memory
stays bounded; the chunking is part of the recipe.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import Optional

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    T: int            # tokens
    H: int            # hidden size
    E: int            # experts
    k: int            # top_k
    h: int            # expert FFN width
    cf: float         # capacity factor
    bias: str = "none"   # "none" | "zipf" | "normal1.5"
    note: str = field(default="", compare=False)

    def describe(self) -> dict:
        return {"workload": self.name, "T": self.T, "H": self.H, "E": self.E,
                "top_k": self.k, "h": self.h, "capacity_factor": self.cf,
                "gate_bias": self.bias}


WORKLOADS = {
    "tiny": Workload("tiny", 512, 256, 8, 2, 512, 1.25,
                     note="tiny layer, all of it fits in L2"),
    "imbalanced": Workload("imbalanced", 4096, 1024, 16, 2, 2816, 1.0, "zipf",
                           note="Zipf-like logit bias, capacity forces drops"),
    "large_expert": Workload("large_expert", 32768, 4096, 8, 2, 14336, 1.25,
                             note="seq 4096 x micro-batch 8, the worked example"),
    "fine_grained": Workload("fine_grained", 16384, 2048, 64, 6, 1408, 1.25,
                             note="many small ragged expert segments"),
    "many_expert": Workload("many_expert", 131072, 4096, 128, 2, 2048, 1.1,
                            "normal1.5",
                            note="random bias idles about 30% of the experts"),
}
# A small case of the large-expert layer's expert FFN for profiler captures:
# the same K, N and tile shapes (H=4096, h=14336), two experts of 4096 rows,
# weights (235 MB each) still larger than L2, under 1 GB on the device.
PROFILE_WORKLOADS = {
    "ffn_profile": Workload("ffn_profile", 4096, 4096, 2, 2, 14336, 1.25,
                            note="profiler capture case of the large-expert FFN"),
    # the large-expert router and dispatch (T=32768, H=4096, E=8, k=2) with a
    # 64-wide FFN: about 1.5 GB on the device
    "route_profile": Workload("route_profile", 32768, 4096, 8, 2, 64, 1.25,
                              note="profiler capture case of the large-expert router"),
}
# Positional aliases, in the order the workloads are usually listed.
WORKLOAD_ORDER = ["tiny", "imbalanced", "large_expert", "fine_grained", "many_expert"]


def get(name_or_index) -> Workload:
    if isinstance(name_or_index, int):
        return WORKLOADS[WORKLOAD_ORDER[name_or_index - 1]]
    if name_or_index in PROFILE_WORKLOADS:
        return PROFILE_WORKLOADS[name_or_index]
    return WORKLOADS[name_or_index]


def custom(T, H, E, k, h, cf, bias="none", name="custom") -> Workload:
    return Workload(name, T, H, E, k, h, cf, bias)


_X_CHUNK_ROWS = 16384


def _randn_bf16(gen: torch.Generator, shape, std: float) -> torch.Tensor:
    return (torch.randn(shape, generator=gen, dtype=torch.float32) * std).to(torch.bfloat16)


def _draw_rows(gen, rows, cols, std):
    out = torch.empty((rows, cols), dtype=torch.bfloat16)
    for r0 in range(0, rows, _X_CHUNK_ROWS):
        r1 = min(rows, r0 + _X_CHUNK_ROWS)
        out[r0:r1] = _randn_bf16(gen, (r1 - r0, cols), std)
    return out


def _draw_experts(gen, E, rows, cols, std):
    out = torch.empty((E, rows, cols), dtype=torch.bfloat16)
    for e in range(E):
        out[e] = _randn_bf16(gen, (rows, cols), std)
    return out


def bias_vector(w: Workload, gen: Optional[torch.Generator] = None) -> Optional[torch.Tensor]:
    if w.bias == "none":
        return None
    if w.bias == "zipf":
        e = torch.arange(w.E, dtype=torch.float64)
        return (2.0 * torch.log(1.0 / (e + 1.0))).to(torch.float32)
    if w.bias == "normal1.5":
        assert gen is not None
        return torch.randn((w.E,), generator=gen, dtype=torch.float32) * math.sqrt(1.5)
    raise ValueError(w.bias)


def make_inputs(w: Workload, seed: int = 0, with_weights: bool = True) -> dict:
    """All layer inputs as CPU tensors: x [T,H] bf16, gate [H,E] bf16,
    bias [E] fp32 or None, W1 [E,H,h] bf16, W2 [E,h,H] bf16."""
    gen = torch.Generator().manual_seed(seed)
    x = _draw_rows(gen, w.T, w.H, 1.0)
    gate = _randn_bf16(gen, (w.H, w.E), 1.0 / math.sqrt(w.H))
    bias = bias_vector(w, gen)
    out = {"x": x, "gate": gate, "bias": bias}
    if with_weights:
        out["W1"] = _draw_experts(gen, w.E, w.H, w.h, 1.0 / math.sqrt(w.H))
        out["W2"] = _draw_experts(gen, w.E, w.h, w.H, 1.0 / math.sqrt(w.h))
    return out


def make_inputs_on_device(w: Workload, device, seed: int = 0) -> dict:
    """The same distributions as ``make_inputs`` (and the same bias rule),
    drawn by a seeded generator on ``device``: a different but equally
    seeded stream of numbers, for timing runs of the larger workloads where
    drawing gigabytes of weights on the host would take half a minute. The
    parity tests use ``make_inputs``."""
    gen = torch.Generator(device=device).manual_seed(seed)

    def draw(shape, std):
        return (torch.randn(shape, generator=gen, dtype=torch.float32, device=device) * std
                ).to(torch.bfloat16)

    x = draw((w.T, w.H), 1.0)
    gate = draw((w.H, w.E), 1.0 / math.sqrt(w.H))
    if w.bias == "normal1.5":
        bias = torch.randn((w.E,), generator=gen, dtype=torch.float32, device=device) * \
            math.sqrt(1.5)
    else:
        b = bias_vector(w)
        bias = None if b is None else b.to(device)
    W1 = torch.empty((w.E, w.H, w.h), dtype=torch.bfloat16, device=device)
    W2 = torch.empty((w.E, w.h, w.H), dtype=torch.bfloat16, device=device)
    for e in range(w.E):
        W1[e] = draw((w.H, w.h), 1.0 / math.sqrt(w.H))
        W2[e] = draw((w.h, w.H), 1.0 / math.sqrt(w.h))
    return {"x": x, "gate": gate, "bias": bias, "W1": W1, "W2": W2}


def make_logits(T: int, E: int, seed: int = 0, bias: Optional[torch.Tensor] = None,
                quantum: float = 0.0) -> torch.Tensor:
    """Synthetic fp32 router logits [T,E] ~ N(0,1) (+ bias), for the
    routing-only entry point. With ``quantum`` > 0 every logit is rounded to
    a multiple of it, which plants exact ties for the tie-break checks."""
    gen = torch.Generator().manual_seed(seed)
    lg = torch.randn((T, E), generator=gen, dtype=torch.float32)
    if bias is not None:
        lg = lg + bias.to(torch.float32)[None, :]
    if quantum > 0:
        lg = torch.round(lg / quantum) * quantum
    return lg.contiguous()


def make_topk_idx(T: int, E: int, k: int, seed: int = 0, skew: float = 0.0) -> torch.Tensor:
    """Synthetic routing decisions [T,k] int32: k distinct experts per token,
    drawn without replacement with probability proportional to exp(-skew*e)."""
    gen = torch.Generator().manual_seed(seed)
    probs = torch.exp(-skew * torch.arange(E, dtype=torch.float64))
    probs = (probs / probs.sum()).expand(T, E)
    return torch.multinomial(probs, k, replacement=False, generator=gen).to(torch.int32).contiguous()


def make_weights(T: int, k: int, seed: int = 0) -> torch.Tensor:
    """Synthetic positive routing weights [T,k] fp32 that sum to 1 per token."""
    gen = torch.Generator().manual_seed(seed)
    w = torch.rand((T, k), generator=gen, dtype=torch.float64) + 0.05
    return (w / w.sum(dim=1, keepdim=True)).to(torch.float32).contiguous()


def sample_rows(T: int, n: int, seed: int = 1) -> torch.Tensor:
    """A sorted, seeded subset of token indices (for outputs checked one by one)."""
    gen = torch.Generator().manual_seed(seed)
    n = min(n, T)
    return torch.sort(torch.randperm(T, generator=gen)[:n]).values
