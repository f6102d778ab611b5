"""The seeded input recipe, checked on the CPU: the named workloads carry the
shapes they are described with, the draws follow the stated distributions,
the draws are reproducible, and the skewed workloads have the structure
they stand in for (a few experts taking most tokens with capacity forcing
drops; a random bias leaving about a third of the experts idle)."""
import math

import numpy as np
import pytest
import torch

import workloads as W
from oracle import moe_oracle as O
from tests._helpers import np64


def test_named_shapes():
    got = {n: (w.T, w.H, w.E, w.k, w.h, w.cf, w.bias) for n, w in W.WORKLOADS.items()}
    assert got == {
        "tiny": (512, 256, 8, 2, 512, 1.25, "none"),
        "imbalanced": (4096, 1024, 16, 2, 2816, 1.0, "zipf"),
        "large_expert": (32768, 4096, 8, 2, 14336, 1.25, "none"),
        "fine_grained": (16384, 2048, 64, 6, 1408, 1.25, "none"),
        "many_expert": (131072, 4096, 128, 2, 2048, 1.1, "normal1.5"),
    }
    # the worked example of the MoE comm bottleneck page, section 2.2:
    # sequence 4096 x micro-batch 8 tokens, hidden 4096, expert width 14336
    w = W.get("large_expert")
    assert w.T == 4096 * 8 and (w.H, w.h, w.E, w.k) == (4096, 14336, 8, 2)
    assert [W.get(i).name for i in range(1, 6)] == W.WORKLOAD_ORDER


def test_draws_follow_the_stated_distributions():
    w = W.get("tiny")
    inp = W.make_inputs(w, seed=0)
    assert inp["x"].shape == (w.T, w.H) and inp["x"].dtype == torch.bfloat16
    assert inp["gate"].shape == (w.H, w.E)
    assert inp["W1"].shape == (w.E, w.H, w.h) and inp["W2"].shape == (w.E, w.h, w.H)
    assert inp["bias"] is None
    for name, std, tol in [("x", 1.0, 0.01), ("gate", 1 / math.sqrt(w.H), 0.05),
                           ("W1", 1 / math.sqrt(w.H), 0.01), ("W2", 1 / math.sqrt(w.h), 0.01)]:
        t = inp[name].double()
        assert abs(t.mean().item()) < 4 * std / math.sqrt(t.numel()), name
        assert abs(t.std().item() / std - 1) < tol, name


def test_draws_are_reproducible_and_seeded():
    w = W.get("tiny")
    a, b, c = W.make_inputs(w, seed=3), W.make_inputs(w, seed=3), W.make_inputs(w, seed=4)
    for key in ("x", "gate", "W1", "W2"):
        assert torch.equal(a[key], b[key]), key
        assert not torch.equal(a[key], c[key]), key
    # weights are drawn after x and the gate: leaving them out changes neither
    d = W.make_inputs(w, seed=3, with_weights=False)
    assert torch.equal(d["x"], a["x"]) and torch.equal(d["gate"], a["gate"])


def test_zipf_bias_and_drops_of_the_imbalanced_layer():
    w = W.get("imbalanced")
    b = W.bias_vector(w).double().numpy()
    assert b[0] == 0.0
    assert np.allclose(b, 2.0 * np.log(1.0 / (np.arange(w.E) + 1.0)), atol=1e-6)
    assert (np.diff(b) < 0).all()
    inp = W.make_inputs(w, seed=0, with_weights=False)
    logits = O.router_logits(np64(inp["x"]), np64(inp["gate"]), inp["bias"].numpy())
    r = O.route_from_logits(logits, w.k)
    d = O.dispatch_plan(r.idx, w.E, O.capacity(w.T, w.E, w.k, w.cf))
    routed = np.bincount(r.idx.ravel(), minlength=w.E)
    # a few experts take most of the traffic and capacity drops most of it
    assert routed[:4].sum() > 0.5 * w.T * w.k
    dropped = 1.0 - d.N / (w.T * w.k)
    assert 0.6 < dropped < 0.8


@pytest.mark.parametrize("seed", [5])
def test_many_expert_bias_idles_about_a_third_of_the_experts(seed):
    w = W.get("many_expert")
    inp = W.make_inputs(w, seed=0, with_weights=False)   # the bias is drawn after x and gate
    b = inp["bias"]
    assert b.shape == (w.E,) and b.dtype == torch.float32
    assert 0.8 < b.std().item() / math.sqrt(1.5) < 1.2
    # logits of std 1 (x ~ N(0,1), gate ~ N(0,1/H)) plus this bias, top-2
    gen = torch.Generator().manual_seed(seed)
    lg = torch.randn((w.T, w.E), generator=gen) + b[None, :]
    idx = torch.topk(lg, w.k, dim=1).indices
    cnt = torch.bincount(idx.flatten(), minlength=w.E).double()
    idle = (cnt < 0.01 * cnt.mean()).double().mean().item()
    assert 0.2 < idle < 0.45
    C = O.capacity(w.T, w.E, w.k, w.cf)
    dropped = 1.0 - torch.clamp(cnt, max=C).sum().item() / (w.T * w.k)
    assert 0.55 < dropped < 0.75


def test_synthetic_routing_helpers():
    idx = W.make_topk_idx(1000, 12, 3, seed=1, skew=0.5)
    assert idx.dtype == torch.int32 and idx.shape == (1000, 3)
    assert all(len(set(row)) == 3 for row in idx.tolist())
    assert int(idx.min()) >= 0 and int(idx.max()) < 12
    wt = W.make_weights(1000, 3, seed=1)
    assert (wt > 0).all() and torch.allclose(wt.double().sum(1), torch.ones(1000, dtype=torch.float64),
                                             atol=1e-6)
    rows = W.sample_rows(32768, 1024)
    assert rows.numel() == 1024 and (rows[1:] > rows[:-1]).all()
    assert int(rows[0]) >= 0 and int(rows[-1]) < 32768
    lg = W.make_logits(64, 8, seed=2, quantum=0.5)
    assert torch.equal(lg, torch.round(lg / 0.5) * 0.5)
