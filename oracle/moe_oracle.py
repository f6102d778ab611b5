"""CPU oracle for the forward pass of one Mixture-of-Experts layer.

TEST INFRASTRUCTURE ONLY. Nothing in the product library imports, links or
calls this module; only the tests, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it. It
shares no code with the CUDA path.

It is plain numpy in float64. Each function computes one step of the layer
literally, in the order the pages give it, with one library primitive at
most per step (a matmul, a stable sort). Page names used in citations:

* "MoE module notes": dpshk.com/news/5154311, an engineering write-up of a
  production MoE layer (router listing in section 3.1, expert FFN in 3.3,
  the ``MoELayer`` listing in 4.2, inference argmax in 5.2).
* "MoE comm bottleneck": cf-1.com/news/4950847, "拆解MoE的通信瓶颈"
  (layer flow in 1.1, byte formulas in 2.1, worked example in 2.2,
  capacity and drop in 3.1, auxiliary loss in 3.2).

Readings taken where the pages are silent, ambiguous or contradict one
another (each is listed again, with its reason, in the design notes):

R1  Routing is deterministic: no Gumbel noise, temperature 1. The training
    router adds Gumbel noise (module notes 3.1); inference drops it and
    takes top-k of the logits (module notes 5.2).
R2  Top-k is chosen on the fp32 logits, largest first; equal logits go to the
    lower expert index first (the pages give no tie rule).
R3  Weights are the softmax over all E experts, renormalised over the k
    chosen ones (module notes 3.1, point 2), which equals a softmax over the
    k chosen logits (comm bottleneck 3.2 listing).
R4  f_e counts assignments before any drop, over T*k (so sum f = 1);
    P_e is the mean of the full softmax over tokens; aux = E * sum f_e P_e
    with the weight alpha left to the caller (comm bottleneck 3.2).
R5  Capacity C = max(1, ceil(cf * T*k / E)) evaluated in binary64 in exactly
    this operation order (comm bottleneck 3.1 gives the ceil; the module
    notes' listing in 4.2 gives the T*k/E form and the floor at 1).
R6  Within an expert, assignments are served in token order and those at
    position >= C are dropped ("later tokens are dropped", comm bottleneck
    3.1). Surviving weights are not renormalised; a token whose slots are
    all dropped outputs zeros (the combine buffer starts at zero in the
    module notes' ``_scatter_back``).
R7  Expert FFN: act = bf16(gelu_tanh(x W1_e)); y_e = bf16(act W2_e), no
    biases (the module notes' 4.2 listing has bias-free expert weights).
R8  Combine: y[t] = bf16( sum over kept slots, ascending j, of w[t,j] y_e ).
R11 Training router (Gumbel): z = (logits + g)/tau with g from caller-drawn
    uniforms; top-k on z, weights and balance statistics from softmax(z).
R12 FP8 path: e4m3 with per-token-row scales for activations and
    per-output-column scales for weights, formed in fp32 (see the FP8 section).
    The expert outputs on their way to the combine are e4m3 with one scale
    per 128-column block of each row (the last block of a row may be
    narrower), formed from the bf16-rounded outputs.

Parity pins for every function here live in tests/test_oracle_pins.py.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np


# ----------------------------------------------------------------- bf16 ----

def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact value of bf16 bit patterns (uint16) as float64."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    # a signalling-NaN pattern widens to a quiet NaN; that is its value here
    with np.errstate(invalid="ignore"):
        return b.view(np.float32).astype(np.float64)


def f64_to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bf16 (ties to even), as bits.

    bf16 keeps 8 significant bits and fp32's exponent range (normal from
    2^-126, subnormal spacing 2^-133, overflow to inf). The value is rounded
    once, from float64, on that grid.
    """
    v = np.asarray(v, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.float64)
    finite = np.isfinite(v)
    out[~finite] = v[~finite]
    vf = v[finite]
    m, ex = np.frexp(vf)                     # vf = m * 2**ex, 0.5 <= |m| < 1
    ex = np.maximum(ex, -125)                # below 2^-126 the grid is fixed
    q = np.rint(np.ldexp(vf, 8 - ex))        # 8 significant bits, RNE
    with np.errstate(over="ignore"):
        out[finite] = np.ldexp(q, ex - 8)    # may overflow to +-inf
    big = np.isfinite(out) & (np.abs(out) >= 2.0 ** 128)
    out[big] = np.sign(out[big]) * np.inf
    bits = (out.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    return bits


def bf16_round(v: np.ndarray) -> np.ndarray:
    """float64 -> nearest bf16 value, returned as float64."""
    return bf16_bits_to_f64(f64_to_bf16_bits(v))


# --------------------------------------------------------------- router ----

def router_logits(x: np.ndarray, gate: np.ndarray, bias: np.ndarray | None = None) -> np.ndarray:
    """Router logits, fp32 [T,E]: logit[t,e] = sum_h x[t,h] gate[h,e] (+ bias[e]).

    The gate is a Linear layer H -> E (module notes 3.1 router listing,
    ``self.gate(x)``; 4.2 ``nn.Linear(hidden_dim, num_experts)``). x and gate
    are bf16 values given as float64; the sum is taken in float64, rounded
    to fp32, and an fp32 bias is added in fp32.
    """
    acc = np.asarray(x, np.float64) @ np.asarray(gate, np.float64)
    lg = acc.astype(np.float32)
    if bias is not None:
        lg = (lg + np.asarray(bias, np.float32)[None, :]).astype(np.float32)
    return lg


def softmax(logits: np.ndarray) -> np.ndarray:
    """p[t,:] = softmax(logits[t,:]) over all E experts, in float64
    (module notes 3.1, ``F.softmax(..., dim=-1)``; R1: temperature 1)."""
    lg = np.asarray(logits, np.float64)
    if not np.all(np.isfinite(lg)):
        raise ValueError("router logits must be finite")
    z = np.exp(lg - lg.max(axis=1, keepdims=True))
    return z / z.sum(axis=1, keepdims=True)


def topk(logits: np.ndarray, k: int) -> np.ndarray:
    """Indices [T,k] of the k largest fp32 logits per token, largest first,
    equal logits ordered by lower expert index (R2; module notes 5.2 picks
    top-k of the logits, ``torch.topk`` returns them sorted)."""
    lg = np.asarray(logits, np.float32)
    order = np.argsort(-lg, axis=1, kind="stable")
    return order[:, :k].astype(np.int32)


def renormalise(p: np.ndarray, idx: np.ndarray) -> np.ndarray:
    """w[t,j] = p[t, idx[t,j]] / sum_j' p[t, idx[t,j']] (module notes 3.1,
    step 3 of the router and the point on normalising top-k weights)."""
    pk = np.take_along_axis(p, idx.astype(np.int64), axis=1)
    return pk / pk.sum(axis=1, keepdims=True)


@dataclass
class Routing:
    idx: np.ndarray       # [T,k] int32
    w: np.ndarray         # [T,k] float64
    p: np.ndarray         # [T,E] float64


def route_from_logits(logits: np.ndarray, k: int) -> Routing:
    """Softmax, top-k and renormalise, in that order (R1-R3)."""
    p = softmax(logits)
    idx = topk(logits, k)
    return Routing(idx=idx, w=renormalise(p, idx), p=p)


def gumbel_noise(u: np.ndarray) -> np.ndarray:
    """Gumbel noise from uniforms u in [0, 1): g = -log(-log(u + 1e-9) + 1e-9)
    (module notes 3.1 router listing and the 4.2 MoELayer listing; the 1e-9
    terms keep both logarithms finite)."""
    u = np.asarray(u, np.float64)
    return -np.log(-np.log(u + 1e-9) + 1e-9)


def route_gumbel(logits: np.ndarray, u: np.ndarray, temperature: float, k: int) -> Routing:
    """The training router (module notes 3.1): z = (logits + g) / temperature,
    p = softmax(z), top-k of z (the same set as top-k of p), weights p
    renormalised over the k chosen (R11: the balance statistics then use this
    perturbed p, as the 4.2 listing feeds `probs` to its balance loss)."""
    z = (np.asarray(logits, np.float64) + gumbel_noise(u)) / float(temperature)
    if not np.all(np.isfinite(z)):
        raise ValueError("router scores must be finite")
    zz = np.exp(z - z.max(axis=1, keepdims=True))
    p = zz / zz.sum(axis=1, keepdims=True)
    idx = np.argsort(-z, axis=1, kind="stable")[:, :k].astype(np.int32)
    return Routing(idx=idx, w=renormalise(p, idx), p=p)


# ------------------------------------------------------ balance stats ------

@dataclass
class Stats:
    routed: np.ndarray    # [E] int64, assignments per expert before drops
    f: np.ndarray         # [E] float64, routed / (T*k)
    P: np.ndarray         # [E] float64, mean router probability
    aux: float            # E * sum f*P


def load_balance_stats(idx: np.ndarray, p: np.ndarray, E: int) -> Stats:
    """Auxiliary load-balancing statistics, comm bottleneck 3.2:
    aux = N * sum_i f_i P_i with N = E experts, f_i the share of assignments
    that go to expert i and P_i the mean router probability of expert i
    over all tokens (R4)."""
    T, k = idx.shape
    routed = np.bincount(idx.reshape(-1).astype(np.int64), minlength=E)[:E]
    if T == 0:
        return Stats(routed=routed, f=np.zeros(E), P=np.zeros(E), aux=0.0)
    f = routed / float(T * k)
    P = p.mean(axis=0)
    return Stats(routed=routed, f=f, P=P, aux=float(E * np.sum(f * P)))


# ------------------------------------------------- capacity and dispatch ---

def capacity(T: int, E: int, k: int, cf: float) -> int:
    """C = max(1, ceil(cf * (T*k) / E)) in binary64 (R5; comm bottleneck 3.1)."""
    return max(1, int(math.ceil(float(cf) * float(T * k) / float(E))))


@dataclass
class Dispatch:
    C: int
    pos: np.ndarray        # [T,k] int64, arrival position inside the expert
    kept_counts: np.ndarray  # [E] int64
    offsets: np.ndarray    # [E+1] int64, exclusive scan of kept_counts
    dest_row: np.ndarray   # [T,k] int32, row in the expert-major buffer, -1 = dropped
    src_token: np.ndarray  # [N] int32, inverse map of dest_row
    N: int                 # kept assignments


def dispatch_plan(idx: np.ndarray, E: int, C) -> Dispatch:
    """Capacity-bounded, token-ordered dispatch (R6).

    Expert e serves its assignments in token order; the one at arrival
    position pos (number of earlier tokens that chose e) is kept iff
    pos < C. Kept assignments are laid out expert by expert, in token order,
    which is the on-device stand-in for the dispatch all-to-all of comm
    bottleneck 1.1 (tokens grouped by destination expert). A token names an
    expert at most once, so ordering the flattened (t, j) list by expert with
    a stable sort orders each expert's list by token. C may also be given
    per expert (an array [E]; see ep_dispatch_plan).
    """
    T, k = idx.shape
    flat = idx.reshape(-1).astype(np.int64)
    order = np.argsort(flat, kind="stable")
    routed = np.bincount(flat, minlength=E)[:E]
    first = np.concatenate([[0], np.cumsum(routed)[:-1]])
    pos_sorted = np.arange(flat.size, dtype=np.int64) - first[flat[order]]
    pos = np.empty(flat.size, dtype=np.int64)
    pos[order] = pos_sorted
    cap = np.broadcast_to(np.asarray(C, np.int64), (E,))
    kept_counts = np.minimum(routed, cap)
    offsets = np.concatenate([[0], np.cumsum(kept_counts)]).astype(np.int64)
    kept = pos < cap[flat]
    dest = np.where(kept, offsets[flat] + pos, -1).astype(np.int32)
    N = int(offsets[-1])
    src = np.full(N, -1, dtype=np.int32)
    tok = np.repeat(np.arange(T, dtype=np.int32), k)
    src[dest[kept]] = tok[kept]
    return Dispatch(C=C, pos=pos.reshape(T, k), kept_counts=kept_counts,
                    offsets=offsets, dest_row=dest.reshape(T, k),
                    src_token=src, N=N)


def ep_dispatch_plan(idx: np.ndarray, E: int, C: int,
                     routed_before: np.ndarray | None = None) -> Dispatch:
    """One rank's dispatch when the experts live on different ranks (expert
    parallelism: comm bottleneck 1.1 sends each token to the rank holding its
    expert; module notes 4.2, ``_all_to_all_routed``).

    With ``routed_before`` (per expert, how many assignments the ranks that
    come before this one in the global token order made to it), each expert
    serves the whole group's tokens in that global order, rank after rank:
    this rank keeps its assignment at local position pos iff
    routed_before[e] + pos < C, with C the capacity of the group's batch.
    Without it, the rank applies C (then its own batch's capacity) to its own
    tokens alone, as the module notes' listing does (its capacity comes from
    the local batch). The rows are laid out expert-major as dispatch_plan
    does; experts of one destination rank are contiguous."""
    if routed_before is None:
        return dispatch_plan(idx, E, C)
    before = np.asarray(routed_before, np.int64)
    return dispatch_plan(idx, E, np.maximum(C - before, 0))


def ep_send_counts(kept_counts: np.ndarray, world: int) -> np.ndarray:
    """Rows one rank sends to each rank: the kept rows of the E/world
    consecutive experts that rank holds (rank g holds experts
    g*E/world .. (g+1)*E/world - 1)."""
    kc = np.asarray(kept_counts, np.int64)
    return kc.reshape(world, -1).sum(axis=1)


def permute(x: np.ndarray, d: Dispatch) -> np.ndarray:
    """x_perm[dest_row[t,j]] = x[t] for every kept assignment
    (the dispatch step of comm bottleneck 1.1, done as a row gather)."""
    return np.asarray(x)[d.src_token]


# ------------------------------------------------------------ expert FFN ---

def gelu_tanh(u: np.ndarray) -> np.ndarray:
    """GELU, tanh form: 0.5 u (1 + tanh(sqrt(2/pi) (u + 0.044715 u^3)))."""
    u = np.asarray(u, np.float64)
    return 0.5 * u * (1.0 + np.tanh(math.sqrt(2.0 / math.pi) * (u + 0.044715 * u ** 3)))


def expert_mlp(rows: np.ndarray, W1e: np.ndarray, W2e: np.ndarray) -> np.ndarray:
    """One expert on a block of rows: Linear -> GELU -> Linear, no biases
    (module notes 3.3 and the 4.2 listing's einsum/gelu/einsum), with bf16
    rounding of the hidden activation and of the output (R7)."""
    u = np.asarray(rows, np.float64) @ np.asarray(W1e, np.float64)
    act = bf16_round(gelu_tanh(u))
    return bf16_round(act @ np.asarray(W2e, np.float64))


def expert_ffn(x_perm: np.ndarray, offsets: np.ndarray, W1, W2) -> np.ndarray:
    """y_perm for the expert-major buffer: rows [offsets[e], offsets[e+1])
    go through expert e. W1/W2 are indexable per expert ([E,H,h], [E,h,H])."""
    E = len(offsets) - 1
    out = np.zeros((int(offsets[-1]), np.asarray(W2[0]).shape[1]), dtype=np.float64)
    for e in range(E):
        a, b = int(offsets[e]), int(offsets[e + 1])
        if b > a:
            out[a:b] = expert_mlp(x_perm[a:b], W1[e], W2[e])
    return out


def combine(y_perm: np.ndarray, d: Dispatch, w: np.ndarray, H: int) -> np.ndarray:
    """y[t] = bf16( sum_{j kept, ascending} w[t,j] * y_perm[dest_row[t,j]] ),
    zero for a token with no kept slot (R6, R8; the combine step of comm
    bottleneck 1.1: weight by the routing weight, return to the token)."""
    T, k = d.dest_row.shape
    acc = np.zeros((T, H), dtype=np.float64)
    for j in range(k):
        r = d.dest_row[:, j]
        m = r >= 0
        acc[m] += w[m, j][:, None] * y_perm[r[m]]
    return bf16_round(acc)


# ----------------------------------------------------------- whole layer ---

@dataclass
class LayerOut:
    logits: np.ndarray
    routing: Routing
    stats: Stats
    dispatch: Dispatch
    y: np.ndarray          # [T,H] float64 holding bf16 values


def layer_forward(x, gate, bias, W1, W2, k: int, cf: float) -> LayerOut:
    """The whole forward pass, steps in the order of comm bottleneck 1.1:
    router, dispatch, expert FFN, weighted combine (inputs as float64
    arrays holding bf16 values)."""
    x = np.asarray(x, np.float64)
    T, H = x.shape
    E = np.asarray(gate).shape[1]
    lg = router_logits(x, gate, bias)
    r = route_from_logits(lg, k)
    st = load_balance_stats(r.idx, r.p, E)
    d = dispatch_plan(r.idx, E, capacity(T, E, k, cf))
    y_perm = expert_ffn(permute(x, d), d.offsets, W1, W2)
    y = combine(y_perm, d, r.w, H)
    return LayerOut(logits=lg, routing=r, stats=st, dispatch=d, y=y)


def token_outputs(x_rows, idx_rows, w_rows, kept_rows, W1, W2) -> np.ndarray:
    """y for a subset of tokens computed one token at a time, from each
    token's own experts, weights and kept mask. The FFN is row-wise, so this
    equals the rows of ``layer_forward``'s y; it lets full-size workloads be
    checked on sampled tokens."""
    x_rows = np.asarray(x_rows, np.float64)
    n, H = x_rows.shape
    acc = np.zeros((n, H), dtype=np.float64)
    idx_rows = np.asarray(idx_rows)
    for e in np.unique(idx_rows):
        for j in range(idx_rows.shape[1]):
            sel = np.nonzero((idx_rows[:, j] == e) & kept_rows[:, j])[0]
            if sel.size:
                ye = expert_mlp(x_rows[sel], W1[int(e)], W2[int(e)])
                acc[sel] += np.asarray(w_rows)[sel, j][:, None] * ye
    return bf16_round(acc)


# ------------------------------------------------------------------ FP8 ---
# FP8 dispatch and expert FFN (MoE comm bottleneck, section 5.3: FP8 hidden
# states halve the dispatch/combine bytes). R12: e4m3 values (4 significant
# bits, exponent bias 7, largest 448, no infinities) with one fp32 scale per
# token row for activations and one per output column for weights; scales
# and the scaled values are formed in fp32 exactly as written below, so the
# quantised bytes are reproducible bit for bit.

E4M3_MAX = 448.0


def e4m3_round(v: np.ndarray) -> np.ndarray:
    """Nearest e4m3 value (ties to even), saturating at +-448, as float64.
    Normals keep 4 significant bits; below 2^-6 the spacing stays 2^-9."""
    v = np.asarray(v, np.float64)
    m, ex = np.frexp(v)
    ex = np.maximum(ex, -5)
    q = np.ldexp(np.rint(np.ldexp(v, 4 - ex)), ex - 4)
    return np.clip(q, -E4M3_MAX, E4M3_MAX)


def quantize_rows_fp8(a: np.ndarray):
    """Per-row e4m3 quantisation: amax = max|a| over the row, inv =
    fp32(448) / fp32(amax), q = e4m3(fp32(a) * inv), scale = fp32(amax) /
    fp32(448) (all products and quotients in fp32); a zero row gives q = 0,
    scale = 0. Returns (q as float64, scale as float64)."""
    a32 = np.asarray(a, np.float32)
    amax = np.abs(a32).max(axis=1) if a32.shape[1] else np.zeros(a32.shape[0], np.float32)
    amax = amax.astype(np.float32)
    nz = amax > 0
    inv = np.zeros_like(amax)
    inv[nz] = np.float32(E4M3_MAX) / amax[nz]
    scale = (amax / np.float32(E4M3_MAX)).astype(np.float32)
    q = e4m3_round((a32 * inv[:, None]).astype(np.float32))
    return q, scale.astype(np.float64)


def quantize_weights_fp8(W: np.ndarray):
    """One expert's weight [K, N] quantised per output column: returns the
    transposed e4m3 values [N, K] (each output column a row, contiguous over
    K) and the fp32 column scales [N]."""
    return quantize_rows_fp8(np.asarray(W).T)


def expert_mlp_fp8(xq: np.ndarray, xs: np.ndarray, w1q, w1s, w2q, w2s) -> np.ndarray:
    """One expert on e4m3 rows: u = xs * w1s * (xq . w1q^T) (float64),
    act = bf16(gelu_tanh(u)), act quantised per row, y = bf16(as * w2s *
    (act_q . w2q^T))."""
    u = (np.asarray(xq) @ np.asarray(w1q, np.float64).T) * xs[:, None] * np.asarray(w1s)[None, :]
    act = bf16_round(gelu_tanh(u))
    aq, as_ = quantize_rows_fp8(act)
    y = (aq @ np.asarray(w2q, np.float64).T) * as_[:, None] * np.asarray(w2s)[None, :]
    return bf16_round(y)


FP8_BLOCK = 128


def quantize_blocks_fp8(a: np.ndarray, block: int = FP8_BLOCK):
    """Per-(row, column block) e4m3 quantisation: each run of `block`
    columns of a row (the last one may be narrower) is quantised as
    quantize_rows_fp8 quantises a row. Returns (q as float64 [n, m], scales
    as float64 [n, ceil(m / block)])."""
    a = np.asarray(a)
    n, m = a.shape
    nb = -(-m // block)
    q = np.zeros((n, m), np.float64)
    s = np.zeros((n, nb), np.float64)
    for b in range(nb):
        q[:, b * block:(b + 1) * block], s[:, b] = quantize_rows_fp8(a[:, b * block:(b + 1) * block])
    return q, s


def dequantize_blocks_fp8(q: np.ndarray, s: np.ndarray, block: int = FP8_BLOCK) -> np.ndarray:
    """q * scale of its block, as float64."""
    cols = np.arange(q.shape[1]) // block
    return np.asarray(q, np.float64) * np.asarray(s, np.float64)[:, cols]


def token_outputs_fp8(x_rows, idx_rows, w_rows, kept_rows, Q1, Q2,
                      fp8_combine: bool = False) -> np.ndarray:
    """y for a subset of tokens through the FP8 FFN: each token row is
    quantised once (the dispatch), then every kept expert runs
    expert_mlp_fp8; Q1[e] = (w1q, w1s), Q2[e] = (w2q, w2s). With
    fp8_combine the expert outputs reach the combine as 128-column block
    quantised e4m3 (quantize_blocks_fp8) and are dequantised there."""
    x_rows = np.asarray(x_rows, np.float64)
    n, H = x_rows.shape
    xq, xs = quantize_rows_fp8(x_rows)
    acc = np.zeros((n, H), dtype=np.float64)
    idx_rows = np.asarray(idx_rows)
    for e in np.unique(idx_rows):
        for j in range(idx_rows.shape[1]):
            sel = np.nonzero((idx_rows[:, j] == e) & kept_rows[:, j])[0]
            if sel.size:
                w1q, w1s = Q1[int(e)]
                w2q, w2s = Q2[int(e)]
                ye = expert_mlp_fp8(xq[sel], xs[sel], w1q, w1s, w2q, w2s)
                if fp8_combine:
                    ye = dequantize_blocks_fp8(*quantize_blocks_fp8(ye))
                acc[sel] += np.asarray(w_rows)[sel, j][:, None] * ye
    return bf16_round(acc)


# ------------------------------------------------------------ accounting ---

def dispatch_bytes(B: int, k: int, H: int, dtype_bytes: int) -> int:
    """Bytes one MoE layer's dispatch moves: B * top_k * H * dtype size
    (comm bottleneck 2.1); the combine moves about as many."""
    return B * k * H * dtype_bytes


def ffn_flops_per_token_expert(H: int, h: int) -> int:
    """Two matmuls of one token through one expert: 2*2*H*h FLOP
    (comm bottleneck 2.2)."""
    return 4 * H * h


def comm_compute_ratio(h: int, dtype_bytes: int) -> float:
    """Bytes per FLOP of one token-expert: (2*H*dtype) / (4*H*h) = dtype / (2 h)
    (comm bottleneck 2.3)."""
    return dtype_bytes / (2.0 * h)
