"""CUDA path vs the CPU oracle, element by element, through the C ABI.

Integer results (indices, counts, offsets, destinations, permuted rows) must
match bit for bit; floating-point results within the stated tolerances.
Sizes span several tiles and a ragged tail; edge cases cover empty and
single-token inputs, k = E, E = 1, heavy drops, ties, bad indices."""
import numpy as np
import pytest
import torch

import top_routing_expert_gb300 as moe
import workloads as W
from oracle import moe_oracle as O
from tests._helpers import (NEAR_TIE, STAT_REL, W_ABS, assert_dispatch_on_gpu_indices,
                            assert_ffn_close, fill_nan_bf16, gumbel_fp32_error, np64,
                            oracle_logits_chunked, routing_flips, topk_margins)

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    moe.build()
    moe.load_library()


def _shape(T, H, E, k, h, cf):
    return moe.MoeShape.make(T, H, E, k, h, cf)


def _zeros(shape, dtype):
    return torch.zeros(shape, dtype=dtype, device=DEV)


def _status():
    return torch.zeros(1, dtype=torch.int32, device=DEV)


# ============================================================ routing ====

def _route_logits_gpu(T, E, k, logits, ws_shape=None):
    s = _shape(T, 64, E, k, 64, 1.0)
    ws = moe.Workspace(s)
    idx = _zeros((T, k), torch.int32)
    w = _zeros((T, k), torch.float32)
    routed = _zeros(E, torch.int32)
    P = _zeros(E, torch.float32)
    aux = _zeros(1, torch.float32)
    st = _status()
    moe.moe_route_logits(s, logits.to(DEV), idx, w, routed, P, aux, st, ws)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), w.cpu().numpy(), routed.cpu().numpy(), P.cpu().numpy(), \
        float(aux.item()), int(st.item())


def _check_routing(logits_cpu, k, got):
    idx, w, routed, P, aux, st = got
    T, E = logits_cpu.shape
    lg = logits_cpu.numpy()
    r = O.route_from_logits(lg, k)
    stt = O.load_balance_stats(r.idx, r.p, E)
    assert st == 0
    assert np.array_equal(idx, r.idx)                      # bit-exact given equal logits
    assert np.abs(w - r.w).max() <= W_ABS
    assert np.abs(w.astype(np.float64).sum(1) - 1).max() <= W_ABS
    assert np.array_equal(routed, stt.routed)
    assert routed.sum() == T * k
    assert np.allclose(P, stt.P, rtol=STAT_REL, atol=1e-12)
    assert abs(aux - stt.aux) <= STAT_REL * abs(stt.aux)


@pytest.mark.parametrize("T,E,k,seed,quantum,bias", [
    (512, 8, 2, 0, 0.0, None),          # tiny workload shape
    (1000, 12, 3, 1, 0.0, None),        # ragged tail, E not a multiple of 8
    (777, 16, 4, 2, 0.25, None),        # many exact ties (quantised logits)
    (300, 256, 8, 3, 0.0, None),        # maximum E and k
    (129, 4, 4, 4, 0.0, None),          # k = E
    (64, 1, 1, 5, 0.0, None),           # one expert
    (1, 33, 5, 6, 0.0, None),           # one token
    (4096, 16, 2, 7, 0.0, "zipf"),      # skewed logits
    (2000, 64, 6, 8, 0.5, None),        # fine-grained, heavy ties
])
def test_route_logits_bit_exact(T, E, k, seed, quantum, bias):
    b = None
    if bias == "zipf":
        b = W.bias_vector(W.custom(T, 64, E, k, 64, 1.0, "zipf"))
    logits = W.make_logits(T, E, seed=seed, bias=b, quantum=quantum)
    _check_routing(logits, k, _route_logits_gpu(T, E, k, logits))


def test_route_logits_all_equal_pick_lowest_experts():
    T, E, k = 300, 10, 3
    logits = torch.zeros((T, E), dtype=torch.float32)
    idx, w, routed, P, aux, st = _route_logits_gpu(T, E, k, logits)
    assert (idx == np.arange(k)).all()
    assert np.allclose(w, 1.0 / k, atol=1e-7)
    assert list(routed) == [T] * k + [0] * (E - k)
    assert abs(aux - 1.0) < 1e-5


def test_route_logits_nonfinite_sets_status():
    T, E, k = 200, 8, 2
    logits = W.make_logits(T, E, seed=3)
    logits[17, 3] = float("nan")
    logits[150, 0] = float("inf")
    *_, st = _route_logits_gpu(T, E, k, logits)
    assert st & moe.DEV_NONFINITE


@pytest.mark.parametrize("name", ["many_expert", "fine_grained", "large_expert"])
def test_route_logits_full_size_workloads(name):
    w = W.get(name)
    logits = W.make_logits(w.T, w.E, seed=11, bias=W.bias_vector(w, torch.Generator().manual_seed(5)))
    _check_routing(logits, w.k, _route_logits_gpu(w.T, w.E, w.k, logits))


# ============================================================ router GEMM ==

@pytest.mark.parametrize("E,k", [(12, 3), (64, 6), (256, 8)])
def test_router_persistent_against_oracle(E, k):
    """More 128-token tiles than SMs (the persistent router: stage ring across
    tiles, two TMEM accumulators), including the largest E and k."""
    T, H = 160 * 128 + 77, 256
    gen = torch.Generator().manual_seed(E + k)
    x = torch.randn((T, H), generator=gen).to(torch.bfloat16)
    gate = (torch.randn((H, E), generator=gen) / H ** 0.5).to(torch.bfloat16)
    bias = torch.randn(E, generator=gen) * 0.5
    s = _shape(T, H, E, k, 64, 1.0)
    ws = moe.Workspace(s)
    idx = _zeros((T, k), torch.int32)
    wt = _zeros((T, k), torch.float32)
    routed = _zeros(E, torch.int32)
    P = _zeros(E, torch.float32)
    aux = _zeros(1, torch.float32)
    lg = _zeros((T, E), torch.float32)
    st = _status()
    moe.moe_route(s, x.to(DEV), gate.to(DEV), bias.to(DEV), idx, wt, routed, P, aux, lg, st, ws)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref_lg = O.router_logits(np64(x), np64(gate), bias.numpy())
    got_lg = lg.cpu().numpy().astype(np.float64)
    assert np.abs(got_lg - ref_lg).max() <= 1e-4 * (1 + np.abs(ref_lg).max())
    # routing against the oracle's own logits: differences only on near-ties
    r = O.route_from_logits(ref_lg.astype(np.float32), k)
    gidx = idx.cpu().numpy()
    mism = np.zeros(T, bool)
    mism[routing_flips(gidx, r.idx, topk_margins(ref_lg, k), f"persistent router E={E}")] = True
    # weights: fp32 logits within 1e-4 relative of float64 ones move w by
    # at most a few 1e-5
    assert np.abs(wt.cpu().numpy()[~mism] - r.w[~mism]).max() <= 1e-4
    # counts on the GPU's own indices, flips or not
    st_ref, _ = assert_dispatch_on_gpu_indices(gidx, r.p, E, 1, routed=routed.cpu().numpy(),
                                               aux=float(aux.item()), aux_rel=1e-3)
    assert np.allclose(P.cpu().numpy(), st_ref.P, rtol=1e-3, atol=1e-6)


def _route_gpu(s, x, gate, bias):
    T, E, k = s.T, s.E, s.top_k
    ws = moe.Workspace(s)
    idx = _zeros((T, k), torch.int32)
    w = _zeros((T, k), torch.float32)
    routed = _zeros(E, torch.int32)
    P = _zeros(E, torch.float32)
    aux = _zeros(1, torch.float32)
    lg = _zeros((T, E), torch.float32)
    st = _status()
    moe.moe_route(s, x.to(DEV), gate.to(DEV), None if bias is None else bias.to(DEV), idx, w,
                  routed, P, aux, lg, st, ws)
    torch.cuda.synchronize()
    return dict(idx=idx.cpu().numpy(), w=w.cpu().numpy(), routed=routed.cpu().numpy(),
                P=P.cpu().numpy(), aux=float(aux.item()), logits=lg.cpu().numpy(),
                status=int(st.item()))


@pytest.mark.parametrize("T,H,E,k,bias", [
    (512, 256, 8, 2, None),       # tiny workload
    (1000, 512, 12, 3, "normal"), # ragged tail, E = 12 padded to 16, bias
    (300, 64, 256, 8, None),      # one K block, maximum E
    (700, 1024, 64, 6, None),
    (130, 4096, 128, 2, "normal"),  # long K, many experts
    # stages hold 4, 2 or 1 k-blocks (the largest dividing H/64 that leaves
    # two stages): three single-k-block stages; two-k-block stages with the
    # gate read as given and its second 64-expert box mostly zero fill; and
    # the persistent kernel (more 128-token tiles than SMs) with two
    (1000, 192, 12, 3, None),
    (700, 384, 72, 4, "normal"),
    (20000, 384, 12, 2, None),
    # 256 experts (four 64-expert gate boxes per k-block): two k-blocks per
    # stage in the per-tile kernel; one in the persistent kernel, where the
    # top-8 epilogue scratch leaves room for no more
    (400, 512, 256, 8, None),
    (20000, 256, 256, 8, "normal"),
])
def test_router_gemm_against_oracle(T, H, E, k, bias):
    gen = torch.Generator().manual_seed(T + H + E)
    x = (torch.randn((T, H), generator=gen)).to(torch.bfloat16)
    gate = (torch.randn((H, E), generator=gen) / H ** 0.5).to(torch.bfloat16)
    b = None if bias is None else torch.randn(E, generator=gen) * 1.2
    g = _route_gpu(_shape(T, H, E, k, 64, 1.0), x, gate, b)
    assert g["status"] == 0
    ref_lg = oracle_logits_chunked(x, gate, b)
    tol = 1e-4 * (1 + np.abs(ref_lg).max())
    assert np.abs(g["logits"] - ref_lg).max() <= tol
    r = O.route_from_logits(ref_lg, k)
    # a routing difference is only acceptable on a near-tie (logged, not failed)
    mism = routing_flips(g["idx"], r.idx, topk_margins(ref_lg, k), f"router T={T} E={E}")
    ok = np.setdiff1d(np.arange(T), mism)
    assert np.abs(g["w"][ok] - r.w[ok]).max() <= 1e-5
    st, _ = assert_dispatch_on_gpu_indices(g["idx"], r.p, E, 1, routed=g["routed"],
                                           aux=g["aux"], aux_rel=1e-4)
    assert np.allclose(g["P"], st.P, rtol=1e-4, atol=1e-7)


# ============================================================ dispatch ====

def _permute_gpu(s, x, idx):
    T, H, E, k = s.T, s.H, s.E, s.top_k
    ws = moe.Workspace(s)
    kept = _zeros(E, torch.int32)
    off = _zeros(E + 1, torch.int32)
    dest = _zeros((T, k), torch.int32)
    src = torch.full((T * k,), -7, dtype=torch.int32, device=DEV)
    xp = _zeros((max(T * k, 1), H), torch.bfloat16)
    st = _status()
    moe.moe_permute(s, x.to(DEV), idx.to(DEV), kept, off, dest, src, xp, st, ws)
    torch.cuda.synchronize()
    return kept.cpu().numpy(), off.cpu().numpy(), dest.cpu().numpy(), src.cpu().numpy(), xp.cpu(), \
        int(st.item())


@pytest.mark.parametrize("T,H,E,k,cf,skew", [
    (512, 256, 8, 2, 1.25, 0.0),
    (1000, 192, 12, 3, 1.0, 0.4),      # ragged, drops
    (4096, 1024, 16, 2, 1.0, 0.9),     # heavy skew, most assignments dropped
    (300, 64, 256, 8, 1.0, 0.02),
    (129, 128, 4, 4, 2.0, 0.0),        # k = E, no drops
    (640, 64, 3, 1, 0.05, 0.0),        # C tiny
    (1, 64, 5, 2, 1.0, 0.0),           # one token
    (16384, 2048, 64, 6, 1.25, 0.05),  # fine-grained workload shape
    # the large-expert routing shape (C = 10240), skewed so that expert 0
    # overflows
    (32768, 4096, 8, 2, 1.25, 0.3),
    # the many-expert routing shape: C = ceil(1.1 * 262144 / 128) = 2253 (a
    # floor would give 2252); the row width does not enter any dispatch
    # decision, so H is kept at 1024 to bound host memory
    (131072, 1024, 128, 2, 1.1, 0.02),
])
def test_permute_bit_exact(T, H, E, k, cf, skew):
    idx = W.make_topk_idx(T, E, k, seed=T + E, skew=skew)
    x = W.make_inputs(W.custom(T, H, E, k, 64, cf), seed=3, with_weights=False)["x"]
    s = _shape(T, H, E, k, 64, cf)
    kept, off, dest, src, xp, st = _permute_gpu(s, x, idx)
    d = O.dispatch_plan(idx.numpy(), E, O.capacity(T, E, k, cf))
    if T * k >= 65536:
        assert d.N < T * k, "the large cases are meant to drop"
    if (T, E, k) == (131072, 128, 2):
        assert d.C == 2253 and d.kept_counts.max() == 2253
    assert st == 0
    assert np.array_equal(kept, d.kept_counts)
    assert np.array_equal(off, d.offsets)
    assert np.array_equal(dest, d.dest_row)
    assert np.array_equal(src[:d.N], d.src_token)
    xv = x.view(torch.int16)
    assert torch.equal(xp[:d.N].view(torch.int16), xv[torch.from_numpy(d.src_token).long()])


def test_permute_bad_and_repeated_indices_are_dropped():
    T, H, E, k, cf = 300, 64, 6, 3, 1.0
    idx = W.make_topk_idx(T, E, k, seed=9)
    idx[5, 1] = 17          # out of range
    idx[40, 0] = -1         # out of range
    idx[77, 2] = idx[77, 0]  # repeats slot 0
    x = W.make_inputs(W.custom(T, H, E, k, 64, cf), seed=4, with_weights=False)["x"]
    kept, off, dest, src, xp, st = _permute_gpu(_shape(T, H, E, k, 64, cf), x, idx)
    assert st & moe.DEV_BAD_INDEX and st & moe.DEV_DUP_INDEX
    # expected: the unusable slots go to an extra expert E that nobody reads
    clean = idx.numpy().copy()
    for t, j in [(5, 1), (40, 0), (77, 2)]:
        clean[t, j] = E
    d = O.dispatch_plan(clean, E + 1, O.capacity(T, E, k, cf))
    want = d.dest_row.copy()
    for t, j in [(5, 1), (40, 0), (77, 2)]:
        want[t, j] = -1
    assert np.array_equal(dest, want)
    assert np.array_equal(off, d.offsets[:E + 1])
    assert np.array_equal(kept, d.kept_counts[:E])


def test_permute_empty_input():
    s = _shape(0, 64, 4, 2, 64, 1.0)
    ws = moe.Workspace(s)
    kept = torch.full((4,), 9, dtype=torch.int32, device=DEV)
    off = torch.full((5,), 9, dtype=torch.int32, device=DEV)
    dummy_i = _zeros((1, 2), torch.int32)
    dummy_x = _zeros((1, 64), torch.bfloat16)
    moe.moe_permute(s, dummy_x, dummy_i, kept, off, dummy_i, None, dummy_x, None, ws)
    torch.cuda.synchronize()
    assert (kept.cpu() == 0).all() and (off.cpu() == 0).all()


# ============================================================ expert FFN ==

def _ffn_case(E, H, h, counts, seed=0):
    k = min(2, E)
    counts = np.asarray(counts)
    N = int(counts.sum())
    T = max((N + k - 1) // k, 1)
    gen = torch.Generator().manual_seed(seed)
    xp = torch.empty((T * k, H), dtype=torch.bfloat16)
    fill_nan_bf16(xp)                                  # rows past N must not matter
    xp[:N] = torch.randn((N, H), generator=gen).to(torch.bfloat16)
    W1 = (torch.randn((E, H, h), generator=gen) / H ** 0.5).to(torch.bfloat16)
    W2 = (torch.randn((E, h, H), generator=gen) / h ** 0.5).to(torch.bfloat16)
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    return T, N, xp, W1, W2, off


def _ffn_gpu(s, xp, off, W1, W2):
    A = s.T * s.top_k
    act = _zeros((A, s.h), torch.bfloat16)
    yp = _zeros((A, s.H), torch.bfloat16)
    st = _status()
    moe.moe_expert_ffn(s, xp.to(DEV), torch.from_numpy(off).to(DEV), W1.to(DEV), W2.to(DEV),
                       act, yp, st)
    torch.cuda.synchronize()
    return act.cpu(), yp.cpu(), int(st.item())


@pytest.mark.parametrize("E,H,h,counts", [
    (1, 128, 128, [300]),                         # dense, ragged M
    (5, 128, 192, [0, 1, 129, 300, 64]),          # empty / single-row segments, partial N tile
    (3, 512, 320, [256, 0, 383]),                 # two n-tiles, second partial
    (8, 256, 512, [160] * 8),                     # tiny workload, full capacity
    (16, 1024, 2816, [512, 512, 384, 300, 200, 150, 100, 90, 50, 30, 10, 5, 2, 1, 0, 0]),
    (64, 2048, 1408, list(np.random.default_rng(0).integers(0, 300, 64))),  # fine-grained shape
    # >= 4096 rows: the CTA-pair kernel, with empty, 1-row and odd-m-tile segments
    (6, 128, 192, [0, 1, 129, 4000, 257, 1]),
    (3, 256, 320, [2048, 0, 2176]),
    # 16 experts on the pair path, with odd m-tile counts whose last m-tile
    # is full, partial or one row
    (16, 256, 320, [0, 1, 127, 128, 129, 255, 256, 257, 383, 384, 385, 511, 512, 640, 700, 900]),
])
def test_expert_ffn_against_oracle(E, H, h, counts):
    T, N, xp, W1, W2, off = _ffn_case(E, H, h, counts, seed=E + H)
    s = _shape(T, H, E, min(2, E), h, 1.0)
    act, yp, st = _ffn_gpu(s, xp, off, W1, W2)
    assert st == 0
    x64 = np64(xp[:N])
    W1n, W2n = np64(W1), np64(W2)
    ref_act = np.zeros((N, h))
    ref_y = np.zeros((N, H))
    for e in range(E):
        a, b = int(off[e]), int(off[e + 1])
        if b > a:
            u = x64[a:b] @ W1n[e]
            ref_act[a:b] = O.bf16_round(O.gelu_tanh(u))
            ref_y[a:b] = O.bf16_round(ref_act[a:b] @ W2n[e])
    assert_ffn_close(np64(act[:N]), ref_act, "act")
    assert_ffn_close(np64(yp[:N]), ref_y, "y_perm")
    # the oracle's own chain (act recomputed in float64) agrees as well
    assert_ffn_close(np64(yp[:N]), O.expert_ffn(x64, off, W1n, W2n), "y_perm (oracle chain)")


@pytest.mark.parametrize("T,H,E,k,h,cf,skew", [
    (300, 128, 5, 2, 192, 1.0, 1.0),         # small: ragged segments, drops
    (1000, 256, 12, 3, 320, 0.8, 0.5),       # partial N tile, drops
    (4096, 512, 8, 2, 256, 1.25, 0.0),       # >= 4096 rows: same kernel as moe_expert_ffn
])
def test_expert_ffn_gathered_against_oracle(T, H, E, k, h, cf, skew):
    """GEMM1 reads x[src_token] by TMA row gathers: same results as the
    oracle FFN on the permuted rows, and (same kernel) the same bits as
    moe_expert_ffn on the permuted copy."""
    gen = torch.Generator().manual_seed(T + E)
    x = torch.randn((T, H), generator=gen).to(torch.bfloat16)
    W1 = (torch.randn((E, H, h), generator=gen) / H ** 0.5).to(torch.bfloat16)
    W2 = (torch.randn((E, h, H), generator=gen) / h ** 0.5).to(torch.bfloat16)
    idx = W.make_topk_idx(T, E, k, skew=skew, seed=T)
    d = O.dispatch_plan(idx.numpy(), E, O.capacity(T, E, k, cf))
    N, A = int(d.offsets[-1]), T * k
    src = torch.full((A,), 10 ** 8, dtype=torch.int32)   # rows past N: never read
    src[:N] = torch.from_numpy(d.src_token[:N].astype(np.int32))
    off = torch.from_numpy(d.offsets.astype(np.int32))
    s = _shape(T, H, E, k, h, cf)
    act = _zeros((A, h), torch.bfloat16)
    yp = _zeros((A, H), torch.bfloat16)
    st = _status()
    moe.moe_expert_ffn_gathered(s, x.to(DEV), src.to(DEV), off.to(DEV), W1.to(DEV), W2.to(DEV),
                                act, yp, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    xp64 = np64(x)[d.src_token[:N]]
    W1n, W2n = np64(W1), np64(W2)
    ref_act = np.zeros((N, h))
    for e in range(E):
        a, b = int(d.offsets[e]), int(d.offsets[e + 1])
        if b > a:
            ref_act[a:b] = O.bf16_round(O.gelu_tanh(xp64[a:b] @ W1n[e]))
    assert_ffn_close(np64(act[:N]), ref_act, "act (gathered)")
    assert_ffn_close(np64(yp[:N]), O.expert_ffn(xp64, d.offsets, W1n, W2n), "y_perm (gathered)")
    if A >= 4096:
        xp = torch.zeros((A, H), dtype=torch.bfloat16)
        xp[:N] = x[torch.from_numpy(d.src_token[:N].astype(np.int64))]
        act2, yp2, st2 = _ffn_gpu(s, xp, d.offsets.astype(np.int32), W1, W2)
        assert st2 == 0
        assert torch.equal(act2[:N], act[:N].cpu()) and torch.equal(yp2[:N], yp[:N].cpu())


def test_permute_indices_only():
    """moe_permute without x_perm writes the same permutation."""
    T, H, E, k = 1000, 64, 12, 3
    idx = W.make_topk_idx(T, E, k, skew=1.0, seed=2)
    x = torch.randn((T, H)).to(torch.bfloat16)
    s = _shape(T, H, E, k, 64, 0.9)
    ws = moe.Workspace(s)
    outs = []
    for with_rows in (True, False):
        off = _zeros(E + 1, torch.int32)
        dest = _zeros((T, k), torch.int32)
        src = _zeros(T * k, torch.int32)
        xp = _zeros((T * k, H), torch.bfloat16) if with_rows else None
        moe.moe_permute(s, x.to(DEV), idx.to(DEV), None, off, dest, src, xp, ws=ws)
        torch.cuda.synchronize()
        n = int(off[-1].item())
        outs.append((off.cpu(), dest.cpu(), src[:n].cpu()))
    for a, b in zip(*outs):
        assert torch.equal(a, b)


# ============================================================ combine ====

@pytest.mark.parametrize("T,H,k,drop", [(512, 256, 2, 0.0), (1000, 512, 3, 0.3), (77, 64, 8, 0.5),
                                        (32768, 4096, 2, 0.01)])
def test_combine_against_oracle(T, H, k, drop):
    gen = torch.Generator().manual_seed(T + k)
    N = T * k
    perm = torch.randperm(N, generator=gen).reshape(T, k).to(torch.int32)
    dropm = torch.rand((T, k), generator=gen) < drop
    dest = torch.where(dropm, torch.full_like(perm, -1), perm)
    w = W.make_weights(T, k, seed=T)
    yp = torch.randn((N, H), generator=gen).to(torch.bfloat16)
    y = _zeros((T, H), torch.bfloat16)
    moe.moe_combine(_shape(T, H, max(k, 1), k, 64, 1.0), yp.to(DEV), dest.to(DEV), w.to(DEV), y)
    torch.cuda.synchronize()
    d = O.Dispatch(C=0, pos=None, kept_counts=None, offsets=None, dest_row=dest.numpy(),
                   src_token=None, N=N)
    w64 = w.numpy().astype(np.float64)
    ref = O.combine(np64(yp), d, w64, H)
    got = np64(y.cpu())
    # fp32 accumulation vs float64: one bf16 step of the result plus the
    # fp32 rounding of the terms (which matters where terms cancel)
    mag = O.combine(np.abs(np64(yp)), d, np.abs(w64), H)
    assert (np.abs(got - ref) <= np.abs(ref) * 2.0 ** -7 + mag * 2.0 ** -20).all()
    assert np.mean(got == ref) > 0.98
    assert (got[(dest.numpy() < 0).all(axis=1)] == 0).all()


# ============================================================ whole layer ==

def _layer_gpu(w: W.Workload, inp, events=False):
    s = _shape(w.T, w.H, w.E, w.k, w.h, w.cf)
    ws = moe.Workspace(s)
    T, E, k = w.T, w.E, w.k
    out = dict(
        y=_zeros((max(T, 1), w.H), torch.bfloat16), aux=_zeros(1, torch.float32),
        topk_idx=_zeros((T, k), torch.int32), topk_w=_zeros((T, k), torch.float32),
        routed_counts=_zeros(E, torch.int32), P=_zeros(E, torch.float32),
        kept_counts=_zeros(E, torch.int32), offsets=_zeros(E + 1, torch.int32),
        dest_row=_zeros((T, k), torch.int32), dev_status=_status())
    bias = inp["bias"]
    moe.moe_layer_fwd(s, inp["x"].to(DEV), inp["gate"].to(DEV),
                      None if bias is None else bias.to(DEV), inp["W1"].to(DEV),
                      inp["W2"].to(DEV), ws=ws, **out)
    torch.cuda.synchronize()
    return {kk: v.cpu() for kk, v in out.items()}


def _check_layer(w: W.Workload, inp, g, sample=None):
    T, E, k = w.T, w.E, w.k
    assert int(g["dev_status"].item()) == 0
    lg = oracle_logits_chunked(inp["x"], inp["gate"], inp["bias"])
    r = O.route_from_logits(lg, k)
    C = O.capacity(T, E, k, w.cf)
    d = O.dispatch_plan(r.idx, E, C)
    gidx = g["topk_idx"].numpy()
    routing_flips(gidx, r.idx, topk_margins(lg, k), w.name)
    gdest = g["dest_row"].numpy()
    # counts, capacity drops and the permutation bit for bit against the
    # oracle's dispatch of the GPU's own indices (equal to its own routing
    # wherever no near-tie flipped)
    st, _ = assert_dispatch_on_gpu_indices(
        gidx, r.p, E, C, routed=g["routed_counts"].numpy(), kept=g["kept_counts"].numpy(),
        offsets=g["offsets"].numpy(), dest_row=gdest, aux=float(g["aux"].item()))
    assert np.allclose(g["P"].numpy(), st.P, rtol=1e-4, atol=1e-7)
    # y: tokens whose routing and kept mask agree with the oracle's
    rows = np.arange(T) if sample is None else np.asarray(sample)
    same = (gidx[rows] == r.idx[rows]).all(1) & ((gdest[rows] >= 0) == (d.dest_row[rows] >= 0)).all(1)
    assert same.mean() > 0.99
    rows = rows[same]
    kept = d.dest_row[rows] >= 0
    ref = O.token_outputs(np64(inp["x"][torch.from_numpy(rows)]), r.idx[rows], r.w[rows], kept,
                          _Lazy64(inp["W1"]), _Lazy64(inp["W2"]))
    assert_ffn_close(np64(g["y"][torch.from_numpy(rows)]), ref, f"{w.name} y")
    assert (np64(g["y"][torch.from_numpy(rows[~kept.any(1)])]) == 0).all()
    return r, d


class _Lazy64:
    """Per-expert float64 view of a bf16 [E, a, b] weight tensor."""

    def __init__(self, t):
        self.t = t

    def __getitem__(self, e):
        return np64(self.t[int(e)])


@pytest.mark.parametrize("name", ["tiny", "imbalanced"])
def test_layer_named_small_workloads(name):
    w = W.get(name)
    inp = W.make_inputs(w, seed=0)
    g = _layer_gpu(w, inp)
    _check_layer(w, inp, g)


@pytest.mark.parametrize("T,H,E,k,h,cf,bias", [
    (1000, 192, 12, 3, 320, 1.0, "zipf"),   # ragged everything, drops
    (1, 64, 4, 2, 64, 1.0, "none"),         # one token
    (200, 128, 1, 1, 128, 1.0, "none"),     # dense FFN
    (150, 64, 4, 4, 192, 1.0, "none"),      # k = E
    (600, 128, 8, 2, 64, 0.02, "zipf"),     # C = 3: almost everything dropped
])
def test_layer_edge_shapes(T, H, E, k, h, cf, bias):
    w = W.custom(T, H, E, k, h, cf, bias, name=f"edge{T}_{E}_{k}")
    inp = W.make_inputs(w, seed=T)
    g = _layer_gpu(w, inp)
    _check_layer(w, inp, g)


def test_layer_maximum_experts_and_k():
    """E = 256, k = 8 (the supported maximum) with 8192 assignments: the
    CTA-pair GEMM with the 6-stage ring (7 stages need E <= 234)."""
    w = W.custom(1024, 128, 256, 8, 128, 1.5, "normal1.5", name="maxE")
    inp = W.make_inputs(w, seed=7)
    g = _layer_gpu(w, inp)
    _check_layer(w, inp, g)


def test_layer_empty_batch():
    w = W.custom(0, 64, 4, 2, 64, 1.0)
    s = _shape(0, 64, 4, 2, 64, 1.0)
    ws = moe.Workspace(s)
    one = _zeros((1, 64), torch.bfloat16)
    off = torch.full((5,), 3, dtype=torch.int32, device=DEV)
    aux = torch.full((1,), 3.0, device=DEV)
    moe.moe_layer_fwd(s, one, _zeros((64, 4), torch.bfloat16), None,
                      _zeros((4, 64, 64), torch.bfloat16), _zeros((4, 64, 64), torch.bfloat16),
                      one, aux=aux, offsets=off, ws=ws)
    torch.cuda.synchronize()
    assert (off.cpu() == 0).all() and float(aux.item()) == 0.0
    del w


def test_binding_refuses_undersized_or_mistyped_buffers():
    """The C ABI takes bare pointers; the binding refuses a buffer smaller
    than the shape needs, or of the wrong dtype, before anything launches."""
    T, H, E, k, h = 64, 64, 4, 2, 64
    s = _shape(T, H, E, k, h, 1.0)
    ws = moe.Workspace(s)
    x = _zeros((T, H), torch.bfloat16)
    gate = _zeros((H, E), torch.bfloat16)
    W1 = _zeros((E, H, h), torch.bfloat16)
    W2 = _zeros((E, h, H), torch.bfloat16)
    y_short = torch.full((T * H - 1,), 7.0, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(ValueError, match="y holds"):
        moe.moe_layer_fwd(s, x, gate, None, W1, W2, y_short, ws=ws)
    with pytest.raises(ValueError, match="W2 holds"):
        moe.moe_layer_fwd(s, x, gate, None, W1, W2[:, :h - 1].contiguous(),
                          _zeros((T, H), torch.bfloat16), ws=ws)
    with pytest.raises(ValueError, match="must be torch.bfloat16"):
        moe.moe_layer_fwd(s, x.float(), gate, None, W1, W2, _zeros((T, H), torch.bfloat16),
                          ws=ws)
    with pytest.raises(ValueError, match="offsets holds"):
        moe.moe_layer_fwd(s, x, gate, None, W1, W2, _zeros((T, H), torch.bfloat16),
                          offsets=_zeros(E, torch.int32), ws=ws)
    torch.cuda.synchronize()
    assert (y_short.float().cpu() == 7.0).all()


def test_layer_is_deterministic_and_reuses_workspace():
    w = W.get("imbalanced")
    inp = W.make_inputs(w, seed=1)
    g1 = _layer_gpu(w, inp)
    g2 = _layer_gpu(w, inp)
    for key in g1:
        assert torch.equal(g1[key], g2[key]), key


def test_components_chain_equals_layer():
    """route -> permute -> expert_ffn -> combine through the separate entry
    points gives the layer's bits exactly."""
    w = W.custom(1000, 256, 12, 3, 320, 1.0, "zipf", name="chain")
    inp = W.make_inputs(w, seed=5)
    g = _layer_gpu(w, inp)
    s = _shape(w.T, w.H, w.E, w.k, w.h, w.cf)
    ws = moe.Workspace(s)
    T, E, k, A = w.T, w.E, w.k, w.T * w.k
    dv = {n: v.to(DEV) for n, v in inp.items() if v is not None}
    idx = _zeros((T, k), torch.int32)
    wt = _zeros((T, k), torch.float32)
    moe.moe_route(s, dv["x"], dv["gate"], dv["bias"], idx, wt, ws=ws)
    off = _zeros(E + 1, torch.int32)
    dest = _zeros((T, k), torch.int32)
    xp = _zeros((A, w.H), torch.bfloat16)
    moe.moe_permute(s, dv["x"], idx, None, off, dest, None, xp, ws=ws)
    act = _zeros((A, w.h), torch.bfloat16)
    yp = _zeros((A, w.H), torch.bfloat16)
    moe.moe_expert_ffn(s, xp, off, dv["W1"], dv["W2"], act, yp, ws=ws)
    y = _zeros((T, w.H), torch.bfloat16)
    moe.moe_combine(s, yp, dest, wt, y)
    torch.cuda.synchronize()
    assert torch.equal(idx.cpu(), g["topk_idx"])
    assert torch.equal(dest.cpu(), g["dest_row"])
    assert torch.equal(y.cpu(), g["y"])


@pytest.mark.parametrize("name", ["large_expert", "fine_grained", "many_expert"])
def test_layer_full_size_workloads_sampled(name):
    """Full-size workloads in the launch configuration the benchmark times:
    routing, counts and permutation in full, outputs on 1024 sampled tokens."""
    w = W.get(name)
    inp = W.make_inputs(w, seed=0)
    g = _layer_gpu(w, inp)
    _check_layer(w, inp, g, sample=W.sample_rows(w.T, 1024, seed=1).numpy())


def _check_y_same_indices(x, gate, bias, W1, W2, k, cf, gidx, y, what):
    """y of one micro-batch against the oracle: routing flips only on
    near-ties, then the oracle's outputs for the GPU's own indices (its
    weights renormalised from the oracle's probabilities, its capacity drops
    from the oracle's dispatch of those indices), every token."""
    E = gate.shape[1]
    T = x.shape[0]
    lg = oracle_logits_chunked(x, gate, bias)
    r = O.route_from_logits(lg, k)
    routing_flips(gidx, r.idx, topk_margins(lg, k), what)
    d = O.dispatch_plan(gidx, E, O.capacity(T, E, k, cf))
    wts = O.renormalise(r.p, gidx)
    ref = O.token_outputs(np64(x), gidx, wts, d.dest_row >= 0, _Lazy64(W1), _Lazy64(W2))
    assert_ffn_close(np64(y), ref, what)
    return d


def test_layer_host_pipeline_equals_device_layer():
    """moe_layer_fwd_host over three micro-batches (copies overlapped with
    the layer on three streams) gives each micro-batch's moe_layer_fwd
    output bit for bit, and each micro-batch's y matches the oracle."""
    w = W.custom(1000, 256, 12, 3, 320, 1.0, "zipf", name="pipe")
    shape = _shape(w.T, w.H, w.E, w.k, w.h, w.cf)
    base = W.make_inputs(w, seed=21)
    xs = [W.make_inputs(w, seed=s, with_weights=False)["x"] for s in (22, 23, 24)]
    dv = {n: base[n].to(DEV) for n in ("gate", "W1", "W2")}
    bias = base["bias"].to(DEV)
    pipe = moe.HostPipeline(shape)
    x_host = [x.pin_memory() for x in xs]
    y_host = [torch.empty((w.T, w.H), dtype=torch.bfloat16).pin_memory() for _ in xs]
    aux_host = torch.zeros(len(xs), dtype=torch.float32).pin_memory()
    status = _status()
    out_stream = pipe.run(x_host, y_host, dv["gate"], bias, dv["W1"], dv["W2"], aux_host, status)
    out_stream.synchronize()
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ws = moe.Workspace(shape)
    for i, x in enumerate(xs):
        y = _zeros((w.T, w.H), torch.bfloat16)
        aux = _zeros(1, torch.float32)
        idx = _zeros((w.T, w.k), torch.int32)
        moe.moe_layer_fwd(shape, x.to(DEV), dv["gate"], bias, dv["W1"], dv["W2"], y, aux=aux,
                          topk_idx=idx, ws=ws)
        torch.cuda.synchronize()
        assert torch.equal(y.cpu(), y_host[i]), i
        assert float(aux.item()) == float(aux_host[i])
        _check_y_same_indices(x, base["gate"], base["bias"], base["W1"], base["W2"], w.k, w.cf,
                              idx.cpu().numpy(), y_host[i], f"host pipeline micro-batch {i}")


@pytest.mark.parametrize("T,H,E,k,h,n_micro", [(1000, 256, 12, 3, 320, 3), (2048, 256, 8, 2, 384, 4)])
def test_layer_device_pipeline_equals_layer_and_oracle(T, H, E, k, h, n_micro):
    """moe_layer_fwd_pipelined (dispatch and expert streams, alternate
    workspaces): every micro-batch's y and aux are moe_layer_fwd's bits on
    its rows, and its y matches the oracle. The second case runs the CTA-pair
    GEMM (4096 rows per micro-batch)."""
    w = W.custom(T, H, E, k, h, 1.0, "zipf", name="devpipe")
    shape = _shape(T, H, E, k, h, 1.0)
    base = W.make_inputs(w, seed=61)
    xs = [W.make_inputs(w, seed=62 + i, with_weights=False)["x"] for i in range(n_micro)]
    dv = {n: base[n].to(DEV) for n in ("gate", "W1", "W2", "bias")}
    x_all = torch.cat(xs).to(DEV)
    y_all = torch.full((n_micro * T, H), 7.0, dtype=torch.bfloat16, device=DEV)
    aux_all = _zeros(n_micro, torch.float32)
    status = _status()
    pipe = moe.DevicePipeline(shape)
    pipe.run(n_micro, x_all, dv["gate"], dv["bias"], dv["W1"], dv["W2"], y_all, aux_all,
             status).synchronize()
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ws = moe.Workspace(shape)
    for i, x in enumerate(xs):
        y = _zeros((T, H), torch.bfloat16)
        aux = _zeros(1, torch.float32)
        idx = _zeros((T, k), torch.int32)
        moe.moe_layer_fwd(shape, x.to(DEV), dv["gate"], dv["bias"], dv["W1"], dv["W2"], y,
                          aux=aux, topk_idx=idx, ws=ws)
        torch.cuda.synchronize()
        assert torch.equal(y_all[i * T:(i + 1) * T].cpu(), y.cpu()), i
        assert float(aux.item()) == float(aux_all[i].item())
        _check_y_same_indices(x, base["gate"], base["bias"], base["W1"], base["W2"], k, 1.0,
                              idx.cpu().numpy(), y.cpu(), f"device pipeline micro-batch {i}")


# ============================================================ Gumbel router

def _uniforms(T, E, seed):
    gen = torch.Generator().manual_seed(seed)
    return torch.rand((T, E), generator=gen, dtype=torch.float32)


@pytest.mark.parametrize("T,H,E,k,tau", [(1000, 512, 12, 3, 1.0), (777, 256, 64, 6, 0.5),
                                         (300, 1024, 8, 2, 2.0), (5000, 256, 128, 2, 1.0),
                                         # the persistent router (more 128-token tiles
                                         # than SMs), noise written back to TMEM
                                         (20000, 384, 72, 4, 0.7)])
def test_route_gumbel_against_oracle(T, H, E, k, tau):
    gen = torch.Generator().manual_seed(T + E)
    x = torch.randn((T, H), generator=gen).to(torch.bfloat16)
    gate = (torch.randn((H, E), generator=gen) / H ** 0.5).to(torch.bfloat16)
    b = torch.randn(E, generator=gen) * 0.5
    u = _uniforms(T, E, seed=T)
    s = _shape(T, H, E, k, 64, 1.0)
    ws = moe.Workspace(s)
    idx = _zeros((T, k), torch.int32)
    w = _zeros((T, k), torch.float32)
    routed = _zeros(E, torch.int32)
    P = _zeros(E, torch.float32)
    aux = _zeros(1, torch.float32)
    sc = _zeros((T, E), torch.float32)
    st = _status()
    moe.moe_route_gumbel(s, x.to(DEV), gate.to(DEV), b.to(DEV), u.to(DEV), tau, idx, w, routed,
                         P, aux, sc, st, ws)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    lg = oracle_logits_chunked(x, gate, b)
    r = O.route_gumbel(lg, u.numpy(), tau, k)
    z = (lg.astype(np.float64) + O.gumbel_noise(u.numpy())) / tau
    gerr = gumbel_fp32_error(u.numpy(), tau)
    assert (np.abs(sc.cpu().numpy() - z) <= 1e-4 * (1 + np.abs(z).max()) + gerr).all()
    gidx = idx.cpu().numpy()
    mism = routing_flips(gidx, r.idx, topk_margins(z, k), f"gumbel router E={E}",
                         slack=1 + np.abs(z).max(), extra=gerr.max(axis=1))
    ok = np.setdiff1d(np.arange(T), mism)
    # a weight is a softmax of the chosen scores: |dw| <= max_j |dz_j|
    w_tol = 1e-5 + gerr.max(axis=1)[ok, None]
    assert (np.abs(w.cpu().numpy()[ok] - r.w[ok]) <= w_tol).all()
    stt, _ = assert_dispatch_on_gpu_indices(gidx, r.p, E, 1, routed=routed.cpu().numpy(),
                                            aux=float(aux.item()), aux_rel=1e-4)
    assert np.allclose(P.cpu().numpy(), stt.P, rtol=1e-4, atol=1e-6)


def test_layer_gumbel_against_oracle():
    w = W.custom(1000, 256, 12, 3, 320, 1.0, "zipf", name="gumbel_layer")
    inp = W.make_inputs(w, seed=31)
    u = _uniforms(w.T, w.E, seed=32)
    tau = 0.7
    s = _shape(w.T, w.H, w.E, w.k, w.h, w.cf)
    ws = moe.Workspace(s)
    y = _zeros((w.T, w.H), torch.bfloat16)
    idx = _zeros((w.T, w.k), torch.int32)
    dest = _zeros((w.T, w.k), torch.int32)
    st = _status()
    dv = {n: v.to(DEV) for n, v in inp.items() if v is not None}
    moe.moe_layer_fwd_gumbel(s, dv["x"], dv["gate"], dv["bias"], u.to(DEV), tau, dv["W1"], dv["W2"],
                             y, topk_idx=idx, dest_row=dest, dev_status=st, ws=ws)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    lg = oracle_logits_chunked(inp["x"], inp["gate"], inp["bias"])
    r = O.route_gumbel(lg, u.numpy(), tau, w.k)
    d = O.dispatch_plan(r.idx, w.E, O.capacity(w.T, w.E, w.k, w.cf))
    gidx = idx.cpu().numpy()
    z = (lg.astype(np.float64) + O.gumbel_noise(u.numpy())) / tau
    routing_flips(gidx, r.idx, topk_margins(z, w.k), "gumbel layer", slack=1 + np.abs(z).max(),
                  extra=gumbel_fp32_error(u.numpy(), tau).max(axis=1))
    assert_dispatch_on_gpu_indices(gidx, r.p, w.E, O.capacity(w.T, w.E, w.k, w.cf),
                                   dest_row=dest.cpu().numpy())
    rows = np.arange(w.T)
    same = (gidx == r.idx).all(1) & ((dest.cpu().numpy() >= 0) == (d.dest_row >= 0)).all(1)
    rows = rows[same]
    kept = d.dest_row[rows] >= 0
    ref = O.token_outputs(np64(inp["x"][torch.from_numpy(rows)]), r.idx[rows], r.w[rows], kept,
                          _Lazy64(inp["W1"]), _Lazy64(inp["W2"]))
    assert_ffn_close(np64(y.cpu()[torch.from_numpy(rows)]), ref, "gumbel layer y")


def test_layer_gumbel_full_size_sampled():
    """The many-expert workload at full size with the training router (the
    scores written back to TMEM once): routing and the permutation in full,
    outputs on 512 sampled tokens."""
    w = W.get("many_expert")
    inp = W.make_inputs(w, seed=0)
    u = _uniforms(w.T, w.E, seed=5)
    tau = 1.0
    s = _shape(w.T, w.H, w.E, w.k, w.h, w.cf)
    ws = moe.Workspace(s)
    y = _zeros((w.T, w.H), torch.bfloat16)
    idx = _zeros((w.T, w.k), torch.int32)
    dest = _zeros((w.T, w.k), torch.int32)
    st = _status()
    dv = {n: v.to(DEV) for n, v in inp.items() if v is not None}
    moe.moe_layer_fwd_gumbel(s, dv["x"], dv["gate"], dv["bias"], u.to(DEV), tau, dv["W1"], dv["W2"],
                             y, topk_idx=idx, dest_row=dest, dev_status=st, ws=ws)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    lg = oracle_logits_chunked(inp["x"], inp["gate"], inp["bias"])
    r = O.route_gumbel(lg, u.numpy(), tau, w.k)
    d = O.dispatch_plan(r.idx, w.E, O.capacity(w.T, w.E, w.k, w.cf))
    gidx = idx.cpu().numpy()
    z = (lg.astype(np.float64) + O.gumbel_noise(u.numpy())) / tau
    routing_flips(gidx, r.idx, topk_margins(z, w.k), "gumbel many_expert",
                  slack=1 + np.abs(z).max(), extra=gumbel_fp32_error(u.numpy(), tau).max(axis=1))
    assert_dispatch_on_gpu_indices(gidx, r.p, w.E, O.capacity(w.T, w.E, w.k, w.cf),
                                   dest_row=dest.cpu().numpy())
    rows = W.sample_rows(w.T, 512, seed=3).numpy()
    same = (gidx[rows] == r.idx[rows]).all(1) & \
        ((dest.cpu().numpy()[rows] >= 0) == (d.dest_row[rows] >= 0)).all(1)
    assert same.mean() > 0.99
    rows = rows[same]
    kept = d.dest_row[rows] >= 0
    ref = O.token_outputs(np64(inp["x"][torch.from_numpy(rows)]), r.idx[rows], r.w[rows], kept,
                          _Lazy64(inp["W1"]), _Lazy64(inp["W2"]))
    assert_ffn_close(np64(y.cpu()[torch.from_numpy(rows)]), ref, "gumbel many_expert y")


def test_layer_captured_in_a_cuda_graph():
    """moe_layer_fwd enqueues only asynchronous work (no allocation, no host
    synchronisation), so it can be captured in a CUDA graph: replays with
    new tokens copied into the captured input give the direct calls' bits."""
    w = W.custom(1000, 256, 12, 3, 320, 1.0, "zipf", name="graph")
    s = _shape(w.T, w.H, w.E, w.k, w.h, w.cf)
    base = W.make_inputs(w, seed=41)
    dv = {n: base[n].to(DEV) for n in ("gate", "W1", "W2", "bias")}
    ws = moe.Workspace(s)
    x_static = base["x"].to(DEV)
    y_static = _zeros((w.T, w.H), torch.bfloat16)
    aux_static = _zeros(1, torch.float32)

    def layer():
        moe.moe_layer_fwd(s, x_static, dv["gate"], dv["bias"], dv["W1"], dv["W2"], y_static,
                          aux=aux_static, ws=ws)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(2):
            layer()
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        layer()
    ws_direct = moe.Workspace(s)
    for seed in (42, 43, 44):
        x = W.make_inputs(w, seed=seed, with_weights=False)["x"].to(DEV)
        x_static.copy_(x)
        g.replay()
        y = _zeros((w.T, w.H), torch.bfloat16)
        aux = _zeros(1, torch.float32)
        idx = _zeros((w.T, w.k), torch.int32)
        moe.moe_layer_fwd(s, x, dv["gate"], dv["bias"], dv["W1"], dv["W2"], y, aux=aux,
                          topk_idx=idx, ws=ws_direct)
        torch.cuda.synchronize()
        assert torch.equal(y_static, y), seed
        assert torch.equal(aux_static, aux), seed
        # and the replayed outputs against the oracle
        _check_y_same_indices(x.cpu(), base["gate"], base["bias"], base["W1"], base["W2"], w.k,
                              w.cf, idx.cpu().numpy(), y_static.cpu(), f"graph replay {seed}")
