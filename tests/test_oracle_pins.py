"""Pins of the CPU oracle to facts that do not come from the oracle itself:
closed forms, brute force on tiny inputs, library routines on special cases
and the numbers the pages print. CPU only."""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(1234)


# ------------------------------------------------------------------ bf16 ---

def test_bf16_round_matches_torch_on_fp32_values():
    # On values that are exact in fp32, torch's fp32 -> bf16 conversion is a
    # single RNE rounding: the oracle must agree bit for bit.
    with np.errstate(over="ignore"):   # the few that overflow are dropped below
        vals = np.concatenate([
            rng.standard_normal(20000).astype(np.float32),
            (rng.standard_normal(2000) * 1e-39).astype(np.float32),   # subnormals
            (rng.standard_normal(2000) * 3e38).astype(np.float32),    # near overflow
            np.array([0.0, -0.0, 1.0, -1.0, 65504.0, 3.3895314e38, 1e-45], np.float32),
        ])
    # halfway points between neighbouring bf16 values, both parities
    base = (rng.integers(0, 0x7F00, 3000).astype(np.uint32) << 16)
    halfway = (base | 0x8000).view(np.float32)
    vals = np.concatenate([vals, halfway, -halfway])
    vals = vals[np.isfinite(vals)]
    ours = O.f64_to_bf16_bits(vals.astype(np.float64))
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_bf16_round_is_single_rounding_from_double():
    one = 1.0
    cases = {
        one + 2.0 ** -8: 1.0,                        # tie -> even (1.0)
        one + 3 * 2.0 ** -8: one + 2.0 ** -6,        # tie -> even (upper)
        one + 2.0 ** -8 + 2.0 ** -40: one + 2.0 ** -7,  # above the tie: up
        -(one + 2.0 ** -8 + 2.0 ** -40): -(one + 2.0 ** -7),
        2.0 ** 128: math.inf,
        (2 - 2.0 ** -8) * 2.0 ** 127: math.inf,      # rounds up past the max
        (2 - 2.0 ** -7) * 2.0 ** 127: (2 - 2.0 ** -7) * 2.0 ** 127,  # bf16 max
        2.0 ** -133: 2.0 ** -133,                   # smallest subnormal
        2.0 ** -134: 0.0,                           # tie -> even (zero)
        1.5 * 2.0 ** -134: 2.0 ** -133,
    }
    for v, want in cases.items():
        got = O.bf16_round(np.array([v]))[0]
        assert got == want, (v, got, want)


def test_bf16_bits_roundtrip():
    bits = np.arange(0, 0x10000, dtype=np.uint32).astype(np.uint16)
    vals = O.bf16_bits_to_f64(bits)
    fin = np.isfinite(vals)
    back = O.f64_to_bf16_bits(vals[fin])
    # -0.0 and 0.0 keep their sign; every finite pattern maps to itself
    assert np.array_equal(back, bits[fin])


# ---------------------------------------------------------------- router ---

def test_router_logits_match_library_matmul():
    x = O.bf16_round(rng.standard_normal((37, 64)))
    g = O.bf16_round(rng.standard_normal((64, 5)) / 8)
    b = rng.standard_normal(5).astype(np.float32)
    ref = torch.matmul(torch.from_numpy(x), torch.from_numpy(g)).to(torch.float32) + torch.from_numpy(b)
    assert np.array_equal(O.router_logits(x, g, b), ref.numpy())


def _topk_brute(row, k):
    # the k-subset whose keys (logit, -index), sorted descending, form the
    # lexicographically largest tuple; then its members in that order
    E = len(row)
    key = lambda e: (float(row[e]), -e)
    best = None
    for S in itertools.combinations(range(E), k):
        ks = sorted((key(e) for e in S), reverse=True)
        if best is None or ks > best[0]:
            best = (ks, S)
    return [-kk[1] for kk in best[0]]


@pytest.mark.parametrize("kind", ["normal", "binary", "few_levels"])
def test_topk_brute_force(kind):
    for trial in range(40):
        T = int(rng.integers(1, 65))
        E = int(rng.integers(1, 9))
        k = int(rng.integers(1, min(E, 3) + 1))
        if kind == "normal":
            lg = rng.standard_normal((T, E)).astype(np.float32)
        elif kind == "binary":
            lg = rng.integers(0, 2, (T, E)).astype(np.float32)
        else:
            lg = (rng.integers(-2, 3, (T, E)) * 0.5).astype(np.float32)
        idx = O.topk(lg, k)
        for t in range(T):
            assert list(idx[t]) == _topk_brute(lg[t], k)


def test_topk_equal_logits_lowest_indices_first():
    lg = np.zeros((3, 7), np.float32)
    assert (O.topk(lg, 4) == np.arange(4)).all()


def test_softmax_closed_forms():
    E = 6
    p = O.softmax(np.zeros((2, E), np.float32))
    assert np.allclose(p, 1.0 / E, rtol=0, atol=1e-15)
    L = 2.5
    lg = np.zeros((1, E), np.float32)
    lg[0, 3] = L
    p = O.softmax(lg)
    assert math.isclose(p[0, 3], math.exp(L) / (math.exp(L) + E - 1), rel_tol=1e-14)
    for k in (1, 2, 4):
        r = O.route_from_logits(lg, k)
        assert r.idx[0, 0] == 3
        assert math.isclose(r.w[0, 0], math.exp(L) / (math.exp(L) + k - 1), rel_tol=1e-14)


def test_renormalised_weights():
    lg = rng.standard_normal((50, 9)).astype(np.float32)
    for k in range(1, 10):
        r = O.route_from_logits(lg, k)
        assert np.allclose(r.w.sum(axis=1), 1.0, rtol=0, atol=1e-14)
        assert (np.diff(r.w, axis=1) <= 0).all()          # sorted like the logits
        if k == 1:
            assert (r.w == 1.0).all()
        if k == 9:
            assert np.allclose(np.take_along_axis(r.p, r.idx.astype(np.int64), 1), r.w, atol=1e-15)


def test_gumbel_noise_closed_forms():
    # g(u) = -log(-log(u)) up to the 1e-9 guards: g = 0 at u = 1/e, and g is
    # increasing; its mean over uniforms is the Euler-Mascheroni constant
    assert abs(O.gumbel_noise(np.array([math.exp(-1.0) - 1e-9]))[0]) < 1e-8
    u = np.sort(rng.random(1000))
    assert (np.diff(O.gumbel_noise(u)) >= 0).all()
    big = rng.random(2_000_000)
    assert abs(O.gumbel_noise(big).mean() - 0.5772156649) < 0.005


def test_gumbel_router_reduces_to_plain_router_without_noise():
    lg = rng.standard_normal((200, 9)).astype(np.float32)
    u = np.full(lg.shape, math.exp(-1.0) - 1e-9)         # g = 0
    for k in (1, 3):
        g = O.route_gumbel(lg, u, 1.0, k)
        r = O.route_from_logits(lg, k)
        assert np.array_equal(g.idx, r.idx)
        assert np.allclose(g.w, r.w, atol=1e-12)
        assert np.allclose(g.p, r.p, atol=1e-12)


def test_gumbel_router_temperature():
    lg = rng.standard_normal((300, 7)).astype(np.float32)
    u = rng.random(lg.shape)
    base = O.route_gumbel(lg, u, 1.0, 3)
    for tau in (0.25, 4.0):
        r = O.route_gumbel(lg, u, tau, 3)
        assert np.array_equal(r.idx, base.idx)          # order is unchanged by tau > 0
        z = (lg.astype(np.float64) + O.gumbel_noise(u)) / tau
        assert np.allclose(np.log(r.p[:, 0] / r.p[:, 1]), z[:, 0] - z[:, 1], atol=1e-9)
    # a high temperature flattens p towards uniform
    assert np.abs(O.route_gumbel(lg, u, 1e6, 3).p - 1 / 7).max() < 1e-5


def test_gumbel_max_selects_with_softmax_probabilities():
    # the Gumbel-max trick: argmax(logits + g) is a sample from softmax(logits)
    lg = np.array([[1.5, 0.0, -0.7, 0.3]], np.float32)
    n = 200_000
    u = rng.random((n, 4))
    r = O.route_gumbel(np.repeat(lg, n, axis=0), u, 1.0, 1)
    freq = np.bincount(r.idx[:, 0], minlength=4) / n
    p = O.softmax(lg)[0]
    assert np.abs(freq - p).max() < 4 * np.sqrt(p * (1 - p) / n).max()


def test_nonfinite_logits_rejected():
    lg = np.zeros((2, 4), np.float32)
    lg[1, 2] = np.nan
    with pytest.raises(ValueError):
        O.softmax(lg)


# ------------------------------------------------------------------- aux ---

@pytest.mark.parametrize("T,E,k", [(16, 4, 1), (30, 8, 2), (64, 64, 6), (5, 3, 3)])
def test_aux_is_one_for_uniform_logits(T, E, k):
    lg = np.zeros((T, E), np.float32)
    r = O.route_from_logits(lg, k)
    st = O.load_balance_stats(r.idx, r.p, E)
    # every token picks experts 0..k-1: f_e = 1/k there, P_e = 1/E
    assert np.allclose(st.f[:k], 1.0 / k) and (st.f[k:] == 0).all()
    assert math.isclose(st.aux, 1.0, rel_tol=1e-13)


def test_aux_is_one_when_either_distribution_is_uniform():
    E, k = 8, 2
    # balanced assignments (uniform f) with arbitrary router probabilities
    idx = np.array([[e, (e + 1) % E] for e in range(E)] * 5, np.int32)
    p = rng.dirichlet(np.ones(E), size=idx.shape[0])
    st = O.load_balance_stats(idx, p, E)
    assert np.allclose(st.f, 1.0 / E)
    assert math.isclose(st.aux, 1.0, rel_tol=1e-13)
    # skewed assignments with uniform probabilities
    idx2 = np.array([[0, 1]] * 30 + [[2, 5]] * 3, np.int32)
    st2 = O.load_balance_stats(idx2, np.full((33, E), 1.0 / E), E)
    assert math.isclose(st2.aux, 1.0, rel_tol=1e-13)
    assert math.isclose(st2.f.sum(), 1.0, rel_tol=1e-15)


def test_aux_above_one_when_mass_and_traffic_coincide():
    # all tokens send both slots to experts 0,1 and put most probability
    # there: aux = E * (1/2 * P0 + 1/2 * P1) with P0 = P1 = 0.45
    E = 10
    idx = np.tile(np.array([[0, 1]], np.int32), (20, 1))
    p = np.full((20, E), 0.1 / 8)
    p[:, 0] = p[:, 1] = 0.45
    st = O.load_balance_stats(idx, p, E)
    assert math.isclose(st.aux, E * 0.45, rel_tol=1e-13)


# ------------------------------------------------------ capacity / drop ----

def test_capacity_of_named_workloads():
    # hand evaluation of max(1, ceil(cf*T*k/E)):
    #   1.25*1024/8 = 160, 1.0*8192/16 = 512, 1.25*65536/8 = 10240,
    #   1.25*98304/64 = 1920, 1.1*262144/128 = 2252.8 -> 2253 (floor: 2252)
    assert O.capacity(512, 8, 2, 1.25) == 160
    assert O.capacity(4096, 16, 2, 1.0) == 512
    assert O.capacity(32768, 8, 2, 1.25) == 10240
    assert O.capacity(16384, 64, 6, 1.25) == 1920
    assert O.capacity(131072, 128, 2, 1.1) == 2253
    assert O.capacity(1, 256, 1, 0.01) == 1
    assert O.capacity(0, 4, 2, 1.0) == 1


def _dispatch_brute(idx, E, C):
    T, k = idx.shape
    seen = [0] * E
    pos = np.zeros((T, k), np.int64)
    for t in range(T):
        for j in range(k):
            e = int(idx[t, j])
            pos[t, j] = seen[e]
            seen[e] += 1
    kept = pos < C
    kept_counts = np.array([min(s, C) for s in seen])
    off = [0]
    for e in range(E):
        off.append(off[-1] + int(kept_counts[e]))
    dest = np.full((T, k), -1, np.int64)
    for t in range(T):
        for j in range(k):
            if kept[t, j]:
                dest[t, j] = off[int(idx[t, j])] + pos[t, j]
    return pos, kept_counts, np.array(off), dest


def _random_idx(T, E, k, skew=0.0):
    pr = np.exp(-skew * np.arange(E))
    pr /= pr.sum()
    return np.stack([rng.choice(E, size=k, replace=False, p=pr) for _ in range(T)]).astype(np.int32)


@pytest.mark.parametrize("T,E,k,cf,skew", [
    (1, 1, 1, 1.0, 0), (7, 3, 2, 0.5, 0), (64, 8, 2, 1.25, 0.0), (64, 8, 2, 0.6, 0.7),
    (200, 16, 3, 1.0, 0.3), (50, 5, 5, 1.0, 0), (300, 12, 4, 0.2, 0.1)])
def test_dispatch_matches_sequential_simulation(T, E, k, cf, skew):
    idx = _random_idx(T, E, k, skew)
    C = O.capacity(T, E, k, cf)
    d = O.dispatch_plan(idx, E, C)
    pos, kc, off, dest = _dispatch_brute(idx, E, C)
    assert np.array_equal(d.pos, pos)
    assert np.array_equal(d.kept_counts, kc)
    assert np.array_equal(d.offsets, off)
    assert np.array_equal(d.dest_row, dest)
    # counts: sum routed = T*k, sum kept = T*k - drops
    routed = np.bincount(idx.reshape(-1), minlength=E)
    assert routed.sum() == T * k
    drops = int((d.dest_row < 0).sum())
    assert d.kept_counts.sum() == T * k - drops == d.N
    # bijection onto [0, N), inverse map, (expert, token) order of rows
    rows = d.dest_row[d.dest_row >= 0]
    assert np.array_equal(np.sort(rows), np.arange(d.N))
    tt, jj = np.nonzero(d.dest_row >= 0)
    assert np.array_equal(d.src_token[d.dest_row[tt, jj]], tt)
    ek = np.array([(int(idx[t, j]), int(t)) for t, j in zip(tt, jj)])
    by_row = ek[np.argsort(d.dest_row[tt, jj])]
    assert all(tuple(by_row[i]) < tuple(by_row[i + 1]) for i in range(len(by_row) - 1))


@pytest.mark.parametrize("world,T,E,k,cf,skew", [
    (2, 97, 12, 3, 0.9, 0.2), (3, 64, 6, 2, 0.5, 0.0), (4, 200, 16, 2, 1.0, 0.4),
    (2, 33, 8, 8, 0.3, 0.0), (8, 57, 8, 1, 2.0, 1.0)])
def test_ep_dispatch_in_global_order_is_the_unsharded_dispatch(world, T, E, k, cf, skew):
    """Experts spread over `world` ranks, tokens split into contiguous shards:
    with each expert serving the group's tokens in global order, every
    rank's kept decisions and expert-major rows, regrouped on the rank that
    holds the expert, must be exactly the single-device dispatch (sequential
    per-expert counters over all tokens, the same simulation that pins
    dispatch_plan)."""
    idx = _random_idx(T, E, k, skew)
    C = O.capacity(T, E, k, cf)
    pos, kc, off, dest = _dispatch_brute(idx, E, C)
    shards = np.array_split(np.arange(T), world)
    E_loc = E // world
    before = np.zeros(E, np.int64)
    sent = []   # per source rank: its expert-major kept (token, expert) rows
    for r, sh in enumerate(shards):
        d = O.ep_dispatch_plan(idx[sh], E, C, before)
        # kept decisions equal the unsharded ones
        assert np.array_equal(d.dest_row >= 0, dest[sh] >= 0), r
        assert np.array_equal(O.ep_send_counts(d.kept_counts, world),
                              d.kept_counts.reshape(world, E_loc).sum(1))
        # the rank's expert-major buffer as (expert, global token) per row
        expert_of_row = np.repeat(np.arange(E), d.kept_counts)
        sent.append([(int(e), int(sh[t])) for e, t in zip(expert_of_row, d.src_token)])
        before += np.bincount(idx[sh].reshape(-1), minlength=E)
    # rank g receives, from each source in rank order, that source's rows of
    # its experts; regrouped expert-major (sources ascending inside an expert)
    # they are the unsharded buffer's segments of those experts
    unsharded = sorted((int(idx[t, j]), t) for t, j in zip(*np.nonzero(dest >= 0)))
    for g in range(world):
        mine = set(range(g * E_loc, (g + 1) * E_loc))
        got = [et for src in sent for et in src if et[0] in mine]
        regrouped = [et for e in sorted(mine) for et in got if et[0] == e]
        assert regrouped == [et for et in unsharded if et[0] in mine], g


def test_ep_dispatch_per_rank_capacity_is_the_local_dispatch():
    """Without the other ranks' counts a rank applies its own batch's
    capacity to its own tokens (the module notes' listing): the sequential
    simulation on the shard alone."""
    idx = _random_idx(80, 8, 2, 0.5)
    sh = np.arange(40, 80)
    C = O.capacity(len(sh), 8, 2, 1.0)
    d = O.ep_dispatch_plan(idx[sh], 8, C)
    pos, kc, off, dest = _dispatch_brute(idx[sh], 8, C)
    assert np.array_equal(d.dest_row, dest) and np.array_equal(d.kept_counts, kc)


def test_dispatch_hand_example():
    # 6 tokens, 4 experts, top-2, cf = 0.75 -> C = ceil(0.75*12/4) = 3
    idx = np.array([[0, 1], [1, 0], [2, 0], [0, 3], [1, 2], [3, 1]], np.int32)
    C = O.capacity(6, 4, 2, 0.75)
    assert C == 3
    d = O.dispatch_plan(idx, 4, C)
    # expert 0 is chosen by tokens 0,1,2,3 -> token 3 dropped; expert 1 by
    # 0,1,4,5 -> token 5 dropped; expert 2 by 2,4; expert 3 by 3,5
    assert list(d.kept_counts) == [3, 3, 2, 2]
    assert list(d.offsets) == [0, 3, 6, 8, 10]
    assert d.dest_row.tolist() == [[0, 3], [4, 1], [6, 2], [-1, 8], [5, 7], [9, -1]]
    assert d.src_token.tolist() == [0, 1, 2, 0, 1, 4, 2, 4, 3, 5]


def test_uniform_logits_drop_every_late_token():
    T, E, k, H = 40, 4, 2, 8
    cf = 0.5                                    # C = ceil(0.5*80/4) = 10
    x = O.bf16_round(rng.standard_normal((T, H)))
    gate = np.zeros((H, E))
    W1 = O.bf16_round(rng.standard_normal((E, H, 16)) * 0.3)
    W2 = O.bf16_round(rng.standard_normal((E, 16, H)) * 0.3)
    out = O.layer_forward(x, gate, None, W1, W2, k, cf)
    C = out.dispatch.C
    assert C == 10
    assert (out.routing.idx == np.arange(k)).all()
    assert (out.dispatch.dest_row[:C] >= 0).all()
    assert (out.dispatch.dest_row[C:] == -1).all()
    assert (out.y[C:] == 0).all()
    assert list(out.dispatch.kept_counts) == [C, C, 0, 0]


# ------------------------------------------------------------------- FFN ---

def test_gelu_tanh_matches_library():
    u = np.concatenate([rng.standard_normal(5000) * 4, [0.0, -30.0, 30.0]])
    ref = torch.nn.functional.gelu(torch.from_numpy(u), approximate="tanh").numpy()
    assert np.allclose(O.gelu_tanh(u), ref, rtol=1e-15, atol=1e-15)
    v = rng.standard_normal(100)
    assert np.allclose(O.gelu_tanh(v) - O.gelu_tanh(-v), v, atol=1e-14)


def _torch_bf16(t64):
    return t64.to(torch.float32).to(torch.bfloat16).to(torch.float64)


def test_single_expert_layer_is_a_dense_ffn():
    # E = 1, k = 1, cf >= 1: nothing is dropped, every weight is 1, and the
    # layer is the dense FFN x -> gelu(x W1) W2 with the same rounding points.
    T, H, h = 33, 64, 96
    x = O.bf16_round(rng.standard_normal((T, H)))
    gate = O.bf16_round(rng.standard_normal((H, 1)))
    W1 = O.bf16_round(rng.standard_normal((1, H, h)) / 8)
    W2 = O.bf16_round(rng.standard_normal((1, h, H)) / 10)
    out = O.layer_forward(x, gate, None, W1, W2, 1, 1.0)
    xt, w1, w2 = (torch.from_numpy(a) for a in (x, W1[0], W2[0]))
    act = _torch_bf16(torch.nn.functional.gelu(xt @ w1, approximate="tanh"))
    ref = _torch_bf16(act @ w2).numpy()
    # both sides round act and y to bf16; a matmul summed in another order
    # can flip an act rounding, which moves y by a few bf16 ulps at most
    assert np.allclose(out.y, ref, rtol=2.0 ** -5, atol=1e-3 * np.abs(ref).max())
    assert np.mean(out.y == ref) > 0.95
    assert (out.routing.w == 1).all() and (out.dispatch.dest_row >= 0).all()


def test_all_experts_layer_is_a_soft_mixture():
    # k = E and cf >= 1: every token visits every expert, so
    # y = sum_e p_e FFN_e(x) with p the full softmax.
    T, H, E, h = 20, 64, 3, 64
    x = O.bf16_round(rng.standard_normal((T, H)))
    gate = O.bf16_round(rng.standard_normal((H, E)) / 8)
    W1 = O.bf16_round(rng.standard_normal((E, H, h)) / 8)
    W2 = O.bf16_round(rng.standard_normal((E, h, H)) / 8)
    out = O.layer_forward(x, gate, None, W1, W2, E, 1.0)
    xt = torch.from_numpy(x)
    lg = (xt @ torch.from_numpy(gate)).to(torch.float32).to(torch.float64)
    p = torch.softmax(lg, dim=1)
    acc = torch.zeros((T, H), dtype=torch.float64)
    for e in range(E):
        act = _torch_bf16(torch.nn.functional.gelu(xt @ torch.from_numpy(W1[e]), approximate="tanh"))
        acc += p[:, e:e + 1] * _torch_bf16(act @ torch.from_numpy(W2[e]))
    ref = _torch_bf16(acc).numpy()
    assert np.allclose(out.y, ref, rtol=2.0 ** -5, atol=1e-3 * np.abs(ref).max())
    assert np.mean(out.y == ref) > 0.9


def _partial_drop_case():
    """40 tokens, 3 experts, top-2, cf = 1 (C = ceil(80/3) = 27). The gate and
    bias give logits (1.0, 0.5, 0.5 + x[t,0]/8), so every token takes expert
    0 first and expert 1 or 2 (by the sign of x[t,0]) second: expert 0 is
    asked by all 40 tokens and serves tokens 0..26 only, experts 1 and 2 are
    asked by about 20 each and serve them all. Tokens 27..39 therefore keep
    their second slot and lose their first."""
    g = np.random.default_rng(77)
    T, H, E, k, h, cf = 40, 64, 3, 2, 64, 1.0
    x = O.bf16_round(g.standard_normal((T, H)))
    gate = np.zeros((H, E))
    gate[0, 2] = 0.125
    bias = np.array([1.0, 0.5, 0.5], np.float32)
    W1 = O.bf16_round(g.standard_normal((E, H, h)) / 8)
    W2 = O.bf16_round(g.standard_normal((E, h, H)) / 8)
    return x, gate, bias, W1, W2, k, cf


def test_partial_drop_keeps_the_surviving_weight_unrenormalised():
    # The pages drop assignments past capacity (comm bottleneck 3.1) into a
    # combine buffer that starts at zero (module notes 4.2, _scatter_back);
    # nothing rescales the survivors, so a token that keeps one slot of two
    # outputs w_kept * FFN_e(x) with w_kept < 1.
    x, gate, bias, W1, W2, k, cf = _partial_drop_case()
    T, E = x.shape[0], gate.shape[1]
    C = 27
    out = O.layer_forward(x, gate, bias, W1, W2, k, cf)
    # routing and drops from the closed-form structure of the case
    second = np.where(x[:, 0] > 0, 2, 1)
    assert (np.sort(out.routing.idx, axis=1) == np.stack([np.zeros(T, int), second], 1)).all()
    assert max((second == 1).sum(), (second == 2).sum()) <= C
    kept = np.ones((T, k), bool)
    slot0 = np.argmax(out.routing.idx == 0, axis=1)          # the slot naming expert 0
    kept[np.arange(T)[C:], slot0[C:]] = False
    assert np.array_equal(out.dispatch.dest_row >= 0, kept)
    assert (kept.sum(1) == 1).sum() == T - C
    # expected outputs by torch ops in float64: weights from the softmax of
    # the logits renormalised over the chosen two, one expert FFN per slot,
    # only the kept slots summed, in slot order
    lg = torch.from_numpy(out.logits.astype(np.float64))
    p = torch.softmax(lg, dim=1)
    idx = torch.from_numpy(out.routing.idx.astype(np.int64))
    pk = torch.gather(p, 1, idx)
    w = pk / pk.sum(1, keepdim=True)
    xt = torch.from_numpy(x)
    ffn = []
    for e in range(E):
        act = _torch_bf16(torch.nn.functional.gelu(xt @ torch.from_numpy(W1[e]), approximate="tanh"))
        ffn.append(_torch_bf16(act @ torch.from_numpy(W2[e])))
    acc = torch.zeros_like(xt)
    renorm = torch.zeros_like(xt)
    for t in range(T):
        wk = [float(w[t, j]) for j in range(k) if kept[t, j]]
        for j in range(k):
            if kept[t, j]:
                acc[t] += w[t, j] * ffn[int(idx[t, j])][t]
                renorm[t] += w[t, j] / sum(wk) * ffn[int(idx[t, j])][t]
    ref = _torch_bf16(acc).numpy()
    assert np.allclose(out.y, ref, rtol=2.0 ** -5, atol=1e-3 * np.abs(ref).max())
    assert np.mean(out.y == ref) > 0.9
    # the rescaled alternative differs by the factor 1/w_kept on those tokens
    alt = _torch_bf16(renorm).numpy()
    part = np.arange(C, T)
    assert not np.allclose(out.y[part], alt[part], rtol=0.05, atol=1e-3 * np.abs(alt).max())
    assert (w.numpy()[part][~kept[part]] > 0.1).all()


def test_token_outputs_equal_layer_rows():
    T, H, E, k, h = 60, 64, 6, 2, 64
    x = O.bf16_round(rng.standard_normal((T, H)))
    gate = O.bf16_round(rng.standard_normal((H, E)) / 8)
    W1 = O.bf16_round(rng.standard_normal((E, H, h)) / 8)
    W2 = O.bf16_round(rng.standard_normal((E, h, H)) / 8)
    out = O.layer_forward(x, gate, None, W1, W2, k, 0.8)
    rows = np.array([0, 5, 17, 44, 59])
    kept = out.dispatch.dest_row[rows] >= 0
    y = O.token_outputs(x[rows], out.routing.idx[rows], out.routing.w[rows], kept, W1, W2)
    assert np.array_equal(y, out.y[rows])


# ------------------------------------------------------------ accounting ---

def test_worked_example_accounting():
    with open(os.path.join(GOLDEN, "worked_example_comm_bottleneck_2_2.json")) as f:
        g = json.load(f)
    i, n = g["inputs"], g["as_numbers"]
    B = i["seq_len"] * i["micro_batch"]
    assert B == n["tokens_B"]
    assert O.dispatch_bytes(B, i["top_k"], i["H"], i["dtype_bytes"]) == n["dispatch_bytes_per_layer"]
    fte = O.ffn_flops_per_token_expert(i["H"], i["h_exp"])
    assert abs(fte - n["flop_per_token_expert_approx"]) / fte < 0.01
    assert abs(2 * fte - n["flop_per_token_top2_approx"]) / fte < 0.02
    layer = B * i["top_k"] * fte
    assert abs(layer - n["flop_per_layer_approx"]) / layer < 0.03
    a2a = 2 * O.dispatch_bytes(B, i["top_k"], i["H"], i["dtype_bytes"]) * i["moe_layers"]
    assert abs(a2a - n["a2a_bytes_32_layers_approx"]) / a2a < 0.08
    assert abs(O.comm_compute_ratio(14336, 2) - n["comm_compute_ratio_h14336_approx"]) < 0.05e-5
    assert abs(O.comm_compute_ratio(2048, 2) - n["comm_compute_ratio_h2048_approx"]) < 0.05e-4


# ------------------------------------- planted mistakes must trip a pin ----

def test_planted_mistakes_are_caught(monkeypatch):
    """Each plausible slip in the oracle makes at least one pin fail."""
    # floor instead of ceil in the capacity
    monkeypatch.setattr(O, "capacity", lambda T, E, k, cf: max(1, int(cf * T * k / E)))
    with pytest.raises(AssertionError):
        test_capacity_of_named_workloads()
    monkeypatch.undo()
    # f normalised by T instead of T*k
    real = O.load_balance_stats

    def by_T(idx, p, E):
        s = real(idx, p, E)
        s.aux *= idx.shape[1]
        return s
    monkeypatch.setattr(O, "load_balance_stats", by_T)
    with pytest.raises(AssertionError):
        test_aux_is_one_for_uniform_logits(30, 8, 2)
    monkeypatch.undo()
    # ties broken toward the higher index
    monkeypatch.setattr(O, "topk", lambda lg, k: (lg.shape[1] - 1 - np.argsort(
        -np.asarray(lg)[:, ::-1], axis=1, kind="stable")[:, :k]).astype(np.int32))
    with pytest.raises(AssertionError):
        test_topk_brute_force("binary")
    monkeypatch.undo()
    # slot-major ("all first choices first") drop priority
    def slot_major(idx, E, C):
        T, k = idx.shape
        d = real_plan(idx.T.copy(), E, C)
        d.dest_row = d.dest_row.T.copy()
        d.pos = d.pos.T.copy()
        return d
    real_plan = O.dispatch_plan
    monkeypatch.setattr(O, "dispatch_plan", slot_major)
    with pytest.raises(AssertionError):
        test_dispatch_hand_example()
    monkeypatch.undo()
    # surviving weights rescaled to sum to 1 after a drop
    real_combine = O.combine

    def renormalising(y_perm, d, w, H):
        kw = np.where(d.dest_row >= 0, w, 0.0)
        s = kw.sum(axis=1, keepdims=True)
        return real_combine(y_perm, d, np.where(s > 0, kw / np.where(s > 0, s, 1.0), 0.0), H)
    monkeypatch.setattr(O, "combine", renormalising)
    with pytest.raises(AssertionError):
        test_partial_drop_keeps_the_surviving_weight_unrenormalised()
    monkeypatch.undo()
    # expert-parallel ranks that ignore the earlier ranks' claims on capacity
    real_ep = O.ep_dispatch_plan
    monkeypatch.setattr(O, "ep_dispatch_plan", lambda idx, E, C, before=None: real_ep(idx, E, C))
    with pytest.raises(AssertionError):
        test_ep_dispatch_in_global_order_is_the_unsharded_dispatch(2, 97, 12, 3, 0.9, 0.2)
    monkeypatch.undo()


# ------------------------------------------------------------------ FP8 ----

def test_e4m3_round_matches_torch():
    vals = np.concatenate([rng.standard_normal(20000) * 30, rng.standard_normal(2000) * 1e-2,
                           [0.0, 448.0, -448.0, 2.0 ** -9, 2.0 ** -6, 1.0, 1.0625, 1.1875, 240.0,
                            2.0 ** -10, 3 * 2.0 ** -11]]).astype(np.float32)
    vals = vals[np.abs(vals) <= 448]
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(O.e4m3_round(vals.astype(np.float64)), ref)


def test_e4m3_round_hand_cases():
    cases = {1.0 + 2 ** -4: 1.0, 1.0 + 3 * 2 ** -4: 1.25, 1.0 + 2 ** -4 + 2 ** -20: 1.125,
             2.0 ** -10: 0.0, 3 * 2.0 ** -11: 2.0 ** -9, 460.0: 448.0, 1e6: 448.0, -1e6: -448.0}
    for v, want in cases.items():
        assert O.e4m3_round(np.array([v]))[0] == want, (v, want)


def test_row_quantisation_bounds():
    a = (rng.standard_normal((64, 300)) * np.exp(rng.standard_normal((64, 1)) * 3)).astype(np.float32)
    a[5] = 0.0
    q, s = O.quantize_rows_fp8(a)
    deq = q * s[:, None]
    # the row maximum lands on +-448 and every element within half a step
    nz = np.abs(a).max(axis=1) > 0
    assert np.allclose(np.abs(q[nz]).max(axis=1), 448.0)
    tiny = np.abs(a) * (448.0 / np.maximum(np.abs(a).max(axis=1, keepdims=True), 1e-30)) < 2 ** -6
    rel = np.abs(deq - a) / np.maximum(np.abs(a), 1e-30)
    assert (rel[~tiny & nz[:, None] & (a != 0)] <= 2.0 ** -4 * 1.0001).all()
    assert (q[5] == 0).all() and s[5] == 0


def test_fp8_ffn_is_exact_on_representable_inputs():
    # inputs already on the e4m3 grid with amax 448 per row/column: scale 1,
    # so the FP8 FFN's GEMM1 equals the float64 GEMM exactly
    H, h, n = 64, 96, 20
    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 448.0])
    x = rng.choice(grid, size=(n, H)) * rng.choice([-1, 1], size=(n, H))
    x[:, 0] = 448.0
    W1 = rng.choice(grid, size=(H, h)) * rng.choice([-1, 1], size=(H, h))
    W1[0, :] = 448.0
    xq, xs = O.quantize_rows_fp8(x)
    w1q, w1s = O.quantize_weights_fp8(W1)
    assert np.array_equal(xq, x) and (xs == 1.0).all()
    assert np.array_equal(w1q, W1.T) and (w1s == 1.0).all()
    u = (xq @ w1q.T) * xs[:, None] * w1s[None, :]
    assert np.array_equal(u, x @ W1)


def test_fp8_ffn_close_to_bf16_ffn():
    H, h, n = 256, 384, 200
    x = O.bf16_round(rng.standard_normal((n, H)))
    W1 = O.bf16_round(rng.standard_normal((H, h)) / 16)
    W2 = O.bf16_round(rng.standard_normal((h, H)) / 20)
    y16 = O.expert_mlp(x, W1, W2)
    xq, xs = O.quantize_rows_fp8(x)
    y8 = O.expert_mlp_fp8(xq, xs, *O.quantize_weights_fp8(W1), *O.quantize_weights_fp8(W2))
    # e4m3 keeps 4 significant bits: a few percent, well away from bf16 error
    rel = np.abs(y8 - y16).sum() / np.abs(y16).sum()
    assert 0.005 < rel < 0.08


def test_block_quantisation_scales_each_block_alone():
    # blocks of 128 columns, the last one 64 wide; magnitudes differ by 1e6
    # between blocks, so one scale per row would crush the small blocks
    a = rng.standard_normal((6, 320)).astype(np.float32)
    a[:, :128] *= 1e-3
    a[:, 128:256] *= 1e3
    a[4, 256:] = 0.0
    q, s = O.quantize_blocks_fp8(a)
    assert q.shape == (6, 320) and s.shape == (6, 3)
    for b, (lo, hi) in enumerate([(0, 128), (128, 256), (256, 320)]):
        blk = a[:, lo:hi]
        amax = np.abs(blk).max(axis=1).astype(np.float32)
        nz = amax > 0
        assert np.array_equal(s[nz, b], (amax[nz] / np.float32(448)).astype(np.float64))
        inv = (np.float32(448) / amax[nz]).astype(np.float32)
        ref = torch.from_numpy((blk[nz] * inv[:, None]).astype(np.float32)).to(
            torch.float8_e4m3fn).to(torch.float64).numpy()
        assert np.array_equal(q[nz, lo:hi], ref)
        assert np.allclose(np.abs(q[nz, lo:hi]).max(axis=1), 448.0)
    assert s[4, 2] == 0 and (q[4, 256:] == 0).all()
    deq = O.dequantize_blocks_fp8(q, s)
    rel = np.abs(deq - a) / np.maximum(np.abs(a), 1e-30)
    # normal-range values of every block keep 4 significant bits
    tiny = np.zeros_like(a, bool)
    for lo, hi in [(0, 128), (128, 256), (256, 320)]:
        m = np.abs(a[:, lo:hi]).max(axis=1, keepdims=True)
        tiny[:, lo:hi] = np.abs(a[:, lo:hi]) * 448.0 / np.maximum(m, 1e-30) < 2 ** -6
    assert (rel[~tiny & (a != 0)] <= 2.0 ** -4 * 1.0001).all()


def test_block_quantisation_of_a_narrow_row_is_row_quantisation():
    a = rng.standard_normal((5, 96))
    q1, s1 = O.quantize_blocks_fp8(a)
    q2, s2 = O.quantize_rows_fp8(a)
    assert np.array_equal(q1, q2) and np.array_equal(s1[:, 0], s2)


def test_fp8_combine_changes_outputs_by_at_most_an_e4m3_step():
    H, h, E, k, n = 256, 128, 4, 2, 40
    x = O.bf16_round(rng.standard_normal((n, H)))
    W1 = [O.bf16_round(rng.standard_normal((H, h)) / 16) for _ in range(E)]
    W2 = [O.bf16_round(rng.standard_normal((h, H)) / 11) for _ in range(E)]
    Q1 = [O.quantize_weights_fp8(w) for w in W1]
    Q2 = [O.quantize_weights_fp8(w) for w in W2]
    idx = np.stack([rng.permutation(E)[:k] for _ in range(n)])
    w = rng.uniform(0.1, 1.0, (n, k))
    kept = np.ones((n, k), bool)
    kept[3, 1] = False
    y = O.token_outputs_fp8(x, idx, w, kept, Q1, Q2)
    y8 = O.token_outputs_fp8(x, idx, w, kept, Q1, Q2, fp8_combine=True)
    assert not np.array_equal(y, y8)
    # bound: half an e4m3 step (2^-4 relative) of each summed term, plus the
    # final bf16 rounding of both results
    xq, xs = O.quantize_rows_fp8(x)
    bound = np.zeros((n, H))
    for t in range(n):
        for j in range(k):
            if kept[t, j]:
                e = idx[t, j]
                ye = O.expert_mlp_fp8(xq[t:t + 1], xs[t:t + 1], *Q1[e], *Q2[e])[0]
                bound[t] += w[t, j] * np.abs(ye)
    bound = 2.0 ** -4 * bound + 2.0 ** -7 * (np.abs(y) + np.abs(y8))
    assert (np.abs(y8 - y) <= bound + 1e-30).all()
