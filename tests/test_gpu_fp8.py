"""FP8 (e4m3) dispatch and expert FFN on the GPU vs the oracle's FP8 functions
(MoE comm bottleneck page, section 5.3: FP8 hidden states on the dispatch).

Bit for bit: quantised weights and their column scales, the FP8 dispatch
(permutation, e4m3 rows, row scales). Within the stated tolerances: the FP8
expert FFN and the FP8 layer output, whose GEMMs accumulate in fp32 on the
GPU and in float64 in the oracle."""
import numpy as np
import pytest
import torch

import top_routing_expert_gb300 as moe
import workloads as W
from oracle import moe_oracle as O
from tests._helpers import (NEAR_TIE, assert_dispatch_on_gpu_indices, assert_ffn_close,
                            assert_fp8_out_close, fill_nan_bf16, np64, oracle_logits_chunked,
                            routing_flips, topk_margins)

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    moe.build()
    moe.load_library()


def _zeros(shape, dtype):
    return torch.zeros(shape, dtype=dtype, device=DEV)


def _status():
    return torch.zeros(1, dtype=torch.int32, device=DEV)


def e4m3_values(b: torch.Tensor) -> np.ndarray:
    """e4m3 bytes -> float64 values (decoded by torch's float8_e4m3fn)."""
    return b.detach().cpu().contiguous().view(torch.float8_e4m3fn).float().numpy().astype(np.float64)


def e4m3_bytes(q: np.ndarray) -> torch.Tensor:
    """float64 values that are e4m3-exact -> their bytes (CPU uint8)."""
    t = torch.from_numpy(np.ascontiguousarray(q, np.float32)).to(torch.float8_e4m3fn)
    back = t.float().numpy().astype(np.float64)
    assert np.array_equal(back, np.asarray(q, np.float64)), "value not representable in e4m3"
    return t.view(torch.uint8)


def _special_columns(W: torch.Tensor):
    """Plants a zero column, a wide-range column (subnormal e4m3 results) and
    a column of exact round-to-nearest-even ties (amax 448, so inv = 1)."""
    E, K, N = W.shape
    W[0, :, 0] = 0
    col = torch.full((K,), 2.0 ** -12)
    col[K // 2] = 1000.0
    W[min(1, E - 1), :, 1] = col.to(torch.bfloat16)
    ties = torch.tensor([448.0, 1.0625, 1.1875, -1.0625, 3 * 2.0 ** -10, 2.0 ** -10, 2.0 ** -11,
                         -0.0, 17.0, 18.0, 19.0, -300.0], dtype=torch.float32)
    c = torch.zeros(K)
    c[:len(ties)] = ties
    W[E - 1, :, 2] = c.to(torch.bfloat16)


# ======================================================= weights ====

@pytest.mark.parametrize("E,K,N", [(3, 192, 320), (1, 128, 64), (5, 256, 1024)])
def test_quantize_weights_bit_exact(E, K, N):
    gen = torch.Generator().manual_seed(E * K + N)
    Wt = (torch.randn((E, K, N), generator=gen) / K ** 0.5).to(torch.bfloat16)
    _special_columns(Wt)
    Wq = _zeros((E, N, K), torch.uint8)
    ws = torch.full((E, N), -1.0, device=DEV)
    moe.moe_quantize_weights_fp8(Wt.to(DEV), Wq, ws)
    torch.cuda.synchronize()
    got_q = e4m3_values(Wq)
    got_s = ws.cpu().numpy().astype(np.float64)
    for e in range(E):
        q, s = O.quantize_weights_fp8(np64(Wt[e]))
        assert np.array_equal(got_q[e], q), f"expert {e}: {np.count_nonzero(got_q[e] != q)} bytes differ"
        assert np.array_equal(got_s[e], s), f"expert {e} scales"
    assert got_s[0, 0] == 0 and (got_q[0, 0] == 0).all()          # zero column
    assert (np.abs(got_q) <= O.E4M3_MAX).all()


# ====================================================== dispatch ====

@pytest.mark.parametrize("T,H,E,k,cf,skew", [
    (512, 256, 8, 2, 1.25, 0.0),
    (1000, 192, 12, 3, 1.0, 1.5),       # ragged tiles, drops
    (300, 64, 4, 4, 0.5, 0.0),          # k = E, heavy drops
])
def test_permute_fp8_bit_exact(T, H, E, k, cf, skew):
    gen = torch.Generator().manual_seed(T + E)
    x = torch.randn((T, H), generator=gen).to(torch.bfloat16)
    x[3] = 0                                              # zero row: scale 0
    x[7] *= 1e-4
    x[7, 5] = 200.0                                       # wide-range row
    idx = W.make_topk_idx(T, E, k, skew=skew, seed=T)
    s = moe.MoeShape.make(T, H, E, k, 64, cf)
    ws = moe.Workspace(s)
    A = T * k
    kept = _zeros(E, torch.int32)
    off = _zeros(E + 1, torch.int32)
    dest = _zeros((T, k), torch.int32)
    src = _zeros(A, torch.int32)
    xq = torch.full((A, H), 0x7F, dtype=torch.uint8, device=DEV)
    xs = torch.full((A,), -1.0, device=DEV)
    st = _status()
    moe.moe_permute_fp8(s, x.to(DEV), idx.to(DEV), kept, off, dest, src, xq, xs, st, ws)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    C = O.capacity(T, E, k, cf)
    d = O.dispatch_plan(idx.numpy(), E, C)
    assert np.array_equal(kept.cpu().numpy(), d.kept_counts)
    assert np.array_equal(off.cpu().numpy(), d.offsets)
    assert np.array_equal(dest.cpu().numpy(), d.dest_row)
    n = int(d.offsets[-1])
    q, sc = O.quantize_rows_fp8(np64(x))
    tok = src.cpu().numpy()[:n]
    assert np.array_equal(tok, d.src_token[:n])
    assert np.array_equal(e4m3_values(xq[:n]), q[tok])
    assert np.array_equal(xs[:n].cpu().numpy().astype(np.float64), sc[tok])
    assert sc[3] == 0


# ==================================================== expert FFN ====

def _quantised_weights(W1: torch.Tensor, W2: torch.Tensor):
    """Oracle-quantised weights as the library's device layout."""
    E = W1.shape[0]
    q1, s1, q2, s2 = [], [], [], []
    for e in range(E):
        a, b = O.quantize_weights_fp8(np64(W1[e]))
        q1.append(a)
        s1.append(b)
        a, b = O.quantize_weights_fp8(np64(W2[e]))
        q2.append(a)
        s2.append(b)
    Q = moe.Fp8Weights.__new__(moe.Fp8Weights)
    Q.W1q = e4m3_bytes(np.stack(q1)).to(DEV)
    Q.w1_scale = torch.from_numpy(np.stack(s1).astype(np.float32)).to(DEV)
    Q.W2q = e4m3_bytes(np.stack(q2)).to(DEV)
    Q.w2_scale = torch.from_numpy(np.stack(s2).astype(np.float32)).to(DEV)
    return Q, list(zip(q1, s1)), list(zip(q2, s2))


@pytest.mark.parametrize("E,H,h,counts", [
    (1, 128, 128, [300]),
    (5, 128, 192, [0, 1, 129, 300, 64]),          # empty / single-row segments, partial N tile
    (3, 512, 320, [256, 0, 383]),                 # K = 512: four 128-deep k-blocks
    (16, 1024, 2816, [512, 512, 384, 300, 200, 150, 100, 90, 50, 30, 10, 5, 2, 1, 0, 0]),
    (6, 192, 192, [0, 1, 129, 4000, 257, 1]),     # K = 192: a half k-block read as zeros
])
def test_expert_ffn_fp8_against_oracle(E, H, h, counts):
    k = min(2, E)
    counts = np.asarray(counts)
    N = int(counts.sum())
    T = max((N + k - 1) // k, 1)
    A = T * k
    gen = torch.Generator().manual_seed(E + H + h)
    xp = torch.randn((N, H), generator=gen).to(torch.bfloat16)
    W1 = (torch.randn((E, H, h), generator=gen) / H ** 0.5).to(torch.bfloat16)
    W2 = (torch.randn((E, h, H), generator=gen) / h ** 0.5).to(torch.bfloat16)
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    xq64, xs64 = O.quantize_rows_fp8(np64(xp))
    xq = torch.full((A, H), 0x7F, dtype=torch.uint8)    # rows past N: NaN bytes, never used
    xq[:N] = e4m3_bytes(xq64)
    xs = torch.zeros(A)
    xs[:N] = torch.from_numpy(xs64.astype(np.float32))
    Q, Q1, Q2 = _quantised_weights(W1, W2)
    s = moe.MoeShape.make(T, H, E, k, h, 1.0)
    ws = moe.Workspace(s, fp8=True)
    act = _zeros((A, h), torch.bfloat16)
    yp = _zeros((A, H), torch.bfloat16)
    st = _status()
    moe.moe_expert_ffn_fp8(s, xq.to(DEV), xs.to(DEV), torch.from_numpy(off).to(DEV), Q, act,
                           y_perm=yp, dev_status=st, ws=ws)
    # the same FFN with e4m3 outputs and 128-column block scales
    yq = torch.full((A, H), 0x7F, dtype=torch.uint8, device=DEV)
    ysc = torch.full((A, (H + 127) // 128), -1.0, device=DEV)
    act2 = _zeros((A, h), torch.bfloat16)
    moe.moe_expert_ffn_fp8(s, xq.to(DEV), xs.to(DEV), torch.from_numpy(off).to(DEV), Q, act2,
                           y_q=yq, y_scale=ysc, dev_status=st, ws=ws)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(act2[:N].cpu(), act[:N].cpu())
    # property: the block quantisation of this run's own bf16 outputs (the
    # definition: amax of the block, 448/amax in fp32, e4m3 round to even)
    yb = yp[:N].float().cpu()
    nb = (H + 127) // 128
    amax = torch.stack([yb[:, 128 * b:128 * (b + 1)].abs().amax(dim=1) for b in range(nb)], dim=1)
    assert torch.equal(ysc[:N].cpu(), amax / 448.0)
    # a true fp32 division (torch evaluates `scalar / tensor` as a reciprocal
    # times the scalar, which is not the correctly rounded quotient)
    inv = torch.where(amax > 0, torch.full_like(amax, 448.0) / amax, torch.zeros_like(amax))
    cols = torch.arange(H) // 128
    want = (yb * inv[:, cols]).to(torch.float8_e4m3fn).view(torch.uint8)
    assert torch.equal(yq[:N].cpu(), want)
    ref_act = np.zeros((N, h))
    ref_y = np.zeros((N, H))
    for e in range(E):
        a, b = int(off[e]), int(off[e + 1])
        if b > a:
            u = (xq64[a:b] @ Q1[e][0].T) * xs64[a:b, None] * Q1[e][1][None, :]
            ref_act[a:b] = O.bf16_round(O.gelu_tanh(u))
            ref_y[a:b] = O.expert_mlp_fp8(xq64[a:b], xs64[a:b], *Q1[e], *Q2[e])
    assert_ffn_close(np64(act[:N]), ref_act, "act")
    assert_ffn_close(np64(yp[:N]), ref_y, "y_perm")
    deq = O.dequantize_blocks_fp8(e4m3_values(yq[:N]), ysc[:N].cpu().numpy().astype(np.float64))
    assert_fp8_out_close(deq, O.dequantize_blocks_fp8(*O.quantize_blocks_fp8(ref_y)),
                         "y_q (dequantised)")


# ========================================================= layer ====

class _LazyQ:
    """Oracle-quantised weights of one expert at a time (float64 copies of
    full-size experts are large); caches the last expert."""

    def __init__(self, Wt):
        self.Wt = Wt
        self.e = None

    def __getitem__(self, e):
        e = int(e)
        if e != self.e:
            self.val = O.quantize_weights_fp8(np64(self.Wt[e]))
            self.e = e
        return self.val


def _layer_fp8_gpu(w, inp):
    s = moe.MoeShape.make(w.T, w.H, w.E, w.k, w.h, w.cf)
    ws = moe.Workspace(s, fp8=True)
    T, E, k = w.T, w.E, w.k
    out = dict(
        y=_zeros((max(T, 1), w.H), torch.bfloat16), aux=_zeros(1, torch.float32),
        topk_idx=_zeros((T, k), torch.int32), topk_w=_zeros((T, k), torch.float32),
        offsets=_zeros(E + 1, torch.int32), dest_row=_zeros((T, k), torch.int32),
        dev_status=_status())
    Q = moe.Fp8Weights(inp["W1"].to(DEV), inp["W2"].to(DEV))
    bias = inp["bias"]
    moe.moe_layer_fwd_fp8(s, inp["x"].to(DEV), inp["gate"].to(DEV),
                          None if bias is None else bias.to(DEV), Q, ws=ws, **out)
    torch.cuda.synchronize()
    return {kk: v.cpu() for kk, v in out.items()}, Q


def _check_layer_fp8(w, inp, g, Q, sample=None, check_experts=None):
    T, E, k = w.T, w.E, w.k
    assert int(g["dev_status"].item()) == 0
    lg = oracle_logits_chunked(inp["x"], inp["gate"], inp["bias"])
    r = O.route_from_logits(lg, k)
    d = O.dispatch_plan(r.idx, E, O.capacity(T, E, k, w.cf))
    gidx = g["topk_idx"].numpy()
    routing_flips(gidx, r.idx, topk_margins(lg, k), f"{w.name} fp8")
    gdest = g["dest_row"].numpy()
    assert_dispatch_on_gpu_indices(gidx, r.p, E, O.capacity(T, E, k, w.cf),
                                   offsets=g["offsets"].numpy(), dest_row=gdest,
                                   aux=float(g["aux"].item()))
    for e in (range(E) if check_experts is None else check_experts):
        q1, s1 = O.quantize_weights_fp8(np64(inp["W1"][e]))
        assert np.array_equal(e4m3_values(Q.W1q[e]), q1)
        assert np.array_equal(Q.w1_scale[e].cpu().numpy().astype(np.float64), s1)
    rows = np.arange(T) if sample is None else np.asarray(sample)
    same = (gidx[rows] == r.idx[rows]).all(1) & ((gdest[rows] >= 0) == (d.dest_row[rows] >= 0)).all(1)
    assert same.mean() > 0.99
    rows = rows[same]
    kept = d.dest_row[rows] >= 0
    ref = O.token_outputs_fp8(np64(inp["x"][torch.from_numpy(rows)]), r.idx[rows], r.w[rows], kept,
                              _LazyQ(inp["W1"]), _LazyQ(inp["W2"]), fp8_combine=True)
    assert_fp8_out_close(np64(g["y"][torch.from_numpy(rows)]), ref, f"{w.name} fp8 y")


@pytest.mark.parametrize("name", ["tiny", "imbalanced"])
def test_layer_fp8_named_small_workloads(name):
    w = W.get(name)
    inp = W.make_inputs(w, seed=0)
    g, Q = _layer_fp8_gpu(w, inp)
    _check_layer_fp8(w, inp, g, Q)


@pytest.mark.parametrize("T,H,E,k,h,cf,bias", [
    (1000, 192, 12, 3, 320, 1.0, "zipf"),
    (1, 64, 4, 2, 64, 1.0, "none"),
    (150, 64, 4, 4, 192, 1.0, "none"),
    (600, 128, 8, 2, 64, 0.02, "zipf"),
])
def test_layer_fp8_edge_shapes(T, H, E, k, h, cf, bias):
    w = W.custom(T, H, E, k, h, cf, bias, name=f"fp8edge{T}_{E}_{k}")
    inp = W.make_inputs(w, seed=T)
    g, Q = _layer_fp8_gpu(w, inp)
    _check_layer_fp8(w, inp, g, Q)


def test_layer_fp8_maximum_experts_and_k():
    w = W.custom(1024, 128, 256, 8, 128, 1.5, "normal1.5", name="fp8maxE")
    inp = W.make_inputs(w, seed=7)
    g, Q = _layer_fp8_gpu(w, inp)
    _check_layer_fp8(w, inp, g, Q, check_experts=[0, 255])


def test_layer_fp8_deterministic_and_chain():
    """Two layer calls give the same bits, and permute_fp8 -> expert_ffn_fp8
    (e4m3 outputs) -> combine_fp8 through the separate entry points gives
    them too."""
    w = W.custom(1000, 256, 12, 3, 320, 1.0, "zipf", name="fp8chain")
    inp = W.make_inputs(w, seed=5)
    g1, Q = _layer_fp8_gpu(w, inp)
    g2, _ = _layer_fp8_gpu(w, inp)
    for key in g1:
        assert torch.equal(g1[key], g2[key]), key
    s = moe.MoeShape.make(w.T, w.H, w.E, w.k, w.h, w.cf)
    ws = moe.Workspace(s, fp8=True)
    T, E, k, A = w.T, w.E, w.k, w.T * w.k
    dv = {n: v.to(DEV) for n, v in inp.items() if v is not None}
    idx = _zeros((T, k), torch.int32)
    wt = _zeros((T, k), torch.float32)
    moe.moe_route(s, dv["x"], dv["gate"], dv["bias"], idx, wt, ws=ws)
    off = _zeros(E + 1, torch.int32)
    dest = _zeros((T, k), torch.int32)
    xq = _zeros((A, w.H), torch.uint8)
    xs = _zeros(A, torch.float32)
    moe.moe_permute_fp8(s, dv["x"], idx, None, off, dest, None, xq, xs, ws=ws)
    act = _zeros((A, w.h), torch.bfloat16)
    yq = _zeros((A, w.H), torch.uint8)
    ysc = _zeros((A, (w.H + 127) // 128), torch.float32)
    moe.moe_expert_ffn_fp8(s, xq, xs, off, Q, act, y_q=yq, y_scale=ysc, ws=ws)
    y = _zeros((T, w.H), torch.bfloat16)
    moe.moe_combine_fp8(s, yq, ysc, dest, wt, y)
    torch.cuda.synchronize()
    assert torch.equal(dest.cpu(), g1["dest_row"])
    assert torch.equal(y.cpu(), g1["y"])


def test_layer_fp8_full_size_sampled():
    """The large-expert workload (32768 tokens, H 4096, 8 experts, h 14336)
    in the benchmark's launch configuration: routing and permutation in
    full, outputs on 256 sampled tokens, W1 quantisation of two experts."""
    w = W.get("large_expert")
    inp = W.make_inputs(w, seed=0)
    g, Q = _layer_fp8_gpu(w, inp)
    _check_layer_fp8(w, inp, g, Q, sample=W.sample_rows(w.T, 256, seed=1).numpy(),
                     check_experts=[0, w.E - 1])


@pytest.mark.parametrize("name,n", [("fine_grained", 256), ("many_expert", 96)])
def test_layer_fp8_full_size_sampled_other_workloads(name, n):
    """The fine-grained and many-expert workloads at full size through the FP8
    layer: routing and permutation in full, outputs on sampled tokens (the
    oracle quantises only the experts those tokens reach)."""
    w = W.get(name)
    inp = W.make_inputs(w, seed=0)
    g, Q = _layer_fp8_gpu(w, inp)
    _check_layer_fp8(w, inp, g, Q, sample=W.sample_rows(w.T, n, seed=2).numpy(),
                     check_experts=[0, w.E // 2, w.E - 1])


def test_fp8_nan_rows_past_the_kept_rows_do_not_leak():
    """Rows of the dispatch buffer past offsets[E] are never read into a
    kept row's output (checked with NaN bytes there)."""
    E, H, h = 2, 128, 128
    counts = [130, 5]
    N = sum(counts)
    T, k = 140, 1
    gen = torch.Generator().manual_seed(3)
    xp = torch.randn((N, H), generator=gen).to(torch.bfloat16)
    W1 = (torch.randn((E, H, h), generator=gen) / H ** 0.5).to(torch.bfloat16)
    W2 = (torch.randn((E, h, H), generator=gen) / h ** 0.5).to(torch.bfloat16)
    xq64, xs64 = O.quantize_rows_fp8(np64(xp))
    xq = torch.full((T * k, H), 0xFF, dtype=torch.uint8)
    xq[:N] = e4m3_bytes(xq64)
    xs = torch.full((T * k,), float("nan"))
    xs[:N] = torch.from_numpy(xs64.astype(np.float32))
    Q, _, _ = _quantised_weights(W1, W2)
    s = moe.MoeShape.make(T, H, E, k, h, 1.0)
    ws = moe.Workspace(s, fp8=True)
    act = _zeros((T * k, h), torch.bfloat16)
    fill_nan_bf16(act)
    yp = _zeros((T * k, H), torch.bfloat16)
    off = torch.tensor([0, 130, 135], dtype=torch.int32)
    moe.moe_expert_ffn_fp8(s, xq.to(DEV), xs.to(DEV), off.to(DEV), Q, act, y_perm=yp, ws=ws)
    torch.cuda.synchronize()
    assert torch.isfinite(yp[:N].float()).all()
    assert torch.isfinite(act[:N].float()).all()


# ======================================================= combine ====

@pytest.mark.parametrize("T,H,k,drop", [(512, 256, 2, 0.0), (1000, 320, 3, 0.3), (77, 64, 8, 0.5),
                                        (4096, 4096, 2, 0.01), (300, 2048, 6, 0.1)])
def test_combine_fp8_against_oracle(T, H, k, drop):
    gen = torch.Generator().manual_seed(T + k + 1)
    N = T * k
    perm = torch.randperm(N, generator=gen).reshape(T, k).to(torch.int32)
    dropm = torch.rand((T, k), generator=gen) < drop
    dest = torch.where(dropm, torch.full_like(perm, -1), perm)
    w = W.make_weights(T, k, seed=T)
    yb = torch.randn((N, H), generator=gen).to(torch.bfloat16)
    yb[:, :64] *= 1e-3                                  # a small block beside large ones
    q, sc = O.quantize_blocks_fp8(np64(yb))
    y = _zeros((T, H), torch.bfloat16)
    fill_nan_bf16(y)
    moe.moe_combine_fp8(moe.MoeShape.make(T, H, max(k, 1), k, 64, 1.0), e4m3_bytes(q).to(DEV),
                        torch.from_numpy(sc.astype(np.float32)).to(DEV), dest.to(DEV), w.to(DEV), y)
    torch.cuda.synchronize()
    d = O.Dispatch(C=0, pos=None, kept_counts=None, offsets=None, dest_row=dest.numpy(),
                   src_token=None, N=N)
    w64 = w.numpy().astype(np.float64)
    deq = O.dequantize_blocks_fp8(q, sc)
    ref = O.combine(deq, d, w64, H)
    got = np64(y.cpu())
    mag = O.combine(np.abs(deq), d, np.abs(w64), H)
    assert (np.abs(got - ref) <= np.abs(ref) * 2.0 ** -7 + mag * 2.0 ** -20).all()
    assert np.mean(got == ref) > 0.98
    assert (got[(dest.numpy() < 0).all(axis=1)] == 0).all()


def test_layer_fp8_host_pipeline_equals_device_layer():
    """moe_layer_fwd_host_fp8 over three micro-batches (copies overlapped with
    the FP8 layer on three streams) gives each micro-batch's
    moe_layer_fwd_fp8 output bit for bit, and each micro-batch's y matches
    the oracle's FP8 layer."""
    w = W.custom(1000, 256, 12, 3, 320, 1.0, "zipf", name="pipe8")
    shape = moe.MoeShape.make(w.T, w.H, w.E, w.k, w.h, w.cf)
    base = W.make_inputs(w, seed=31)
    xs = [W.make_inputs(w, seed=s, with_weights=False)["x"] for s in (32, 33, 34)]
    gate, bias = base["gate"].to(DEV), base["bias"].to(DEV)
    Q = moe.Fp8Weights(base["W1"].to(DEV), base["W2"].to(DEV))
    pipe = moe.HostPipeline(shape, fp8=True)
    x_host = [x.pin_memory() for x in xs]
    y_host = [torch.empty((w.T, w.H), dtype=torch.bfloat16).pin_memory() for _ in xs]
    aux_host = torch.zeros(len(xs), dtype=torch.float32).pin_memory()
    status = _status()
    moe.moe_layer_fwd_host_fp8(pipe, x_host, y_host, gate, bias, Q, aux_host, status).synchronize()
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ws = moe.Workspace(shape, fp8=True)
    for i, x in enumerate(xs):
        y = _zeros((w.T, w.H), torch.bfloat16)
        aux = _zeros(1, torch.float32)
        idx = _zeros((w.T, w.k), torch.int32)
        moe.moe_layer_fwd_fp8(shape, x.to(DEV), gate, bias, Q, y, aux=aux, topk_idx=idx, ws=ws)
        torch.cuda.synchronize()
        assert torch.equal(y.cpu(), y_host[i]), i
        assert float(aux.item()) == float(aux_host[i])
        # each micro-batch's y against the oracle's FP8 layer on the GPU's
        # own indices (flips only on near-ties)
        gidx = idx.cpu().numpy()
        lg = oracle_logits_chunked(x, base["gate"], base["bias"])
        r = O.route_from_logits(lg, w.k)
        routing_flips(gidx, r.idx, topk_margins(lg, w.k), f"fp8 host pipeline {i}")
        d = O.dispatch_plan(gidx, w.E, O.capacity(w.T, w.E, w.k, w.cf))
        ref = O.token_outputs_fp8(np64(x), gidx, O.renormalise(r.p, gidx), d.dest_row >= 0,
                                  _LazyQ(base["W1"]), _LazyQ(base["W2"]), fp8_combine=True)
        assert_fp8_out_close(np64(y_host[i]), ref, f"fp8 host pipeline micro-batch {i}")


def test_layer_fp8_captured_in_a_cuda_graph():
    """The FP8 layer (its memset node included) replays from a CUDA graph with
    the direct call's bits."""
    w = W.custom(1000, 256, 12, 3, 320, 1.0, "zipf", name="graph8")
    s = moe.MoeShape.make(w.T, w.H, w.E, w.k, w.h, w.cf)
    base = W.make_inputs(w, seed=51)
    gate, bias = base["gate"].to(DEV), base["bias"].to(DEV)
    Q = moe.Fp8Weights(base["W1"].to(DEV), base["W2"].to(DEV))
    ws = moe.Workspace(s, fp8=True)
    x_static = base["x"].to(DEV)
    y_static = _zeros((w.T, w.H), torch.bfloat16)

    def layer():
        moe.moe_layer_fwd_fp8(s, x_static, gate, bias, Q, y_static, ws=ws)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(2):
            layer()
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        layer()
    ws_direct = moe.Workspace(s, fp8=True)
    for seed in (52, 53):
        x = W.make_inputs(w, seed=seed, with_weights=False)["x"].to(DEV)
        x_static.copy_(x)
        g.replay()
        y = _zeros((w.T, w.H), torch.bfloat16)
        idx = _zeros((w.T, w.k), torch.int32)
        moe.moe_layer_fwd_fp8(s, x, gate, bias, Q, y, topk_idx=idx, ws=ws_direct)
        torch.cuda.synchronize()
        assert torch.equal(y_static, y), seed
        # the replayed outputs against the oracle's FP8 layer on the GPU's indices
        gidx = idx.cpu().numpy()
        lg = oracle_logits_chunked(x.cpu(), base["gate"], base["bias"])
        r = O.route_from_logits(lg, w.k)
        routing_flips(gidx, r.idx, topk_margins(lg, w.k), f"fp8 graph replay {seed}")
        d = O.dispatch_plan(gidx, w.E, O.capacity(w.T, w.E, w.k, w.cf))
        ref = O.token_outputs_fp8(np64(x.cpu()), gidx, O.renormalise(r.p, gidx), d.dest_row >= 0,
                                  _LazyQ(base["W1"]), _LazyQ(base["W2"]), fp8_combine=True)
        assert_fp8_out_close(np64(y_static.cpu()), ref, f"fp8 graph replay {seed}")
