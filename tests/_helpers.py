"""Shared test utilities: conversions, tolerance checks and the oracle
applied in chunks for full-size workloads. Test infrastructure only."""
from __future__ import annotations

import numpy as np
import torch

from oracle import moe_oracle as O

# floating-point bars for bf16-in / fp32-accumulate outputs
FFN_MAX_REL = 2e-2      # max|err| <= 2e-2 * max|ref|
FFN_MEAN_REL = 5e-3     # sum|err| <= 5e-3 * sum|ref|   (mean relative error)
W_ABS = 1e-6            # routing weights
STAT_REL = 1e-5         # P and aux
NEAR_TIE = 1e-5         # top-k margin below which a routing flip is logged


def np64(t: torch.Tensor) -> np.ndarray:
    """Exact float64 copy of a (bf16 / fp32) tensor."""
    return t.detach().float().cpu().numpy().astype(np.float64)


def assert_ffn_close(got: np.ndarray, ref: np.ndarray, what: str = "output"):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite values"
    if ref.size == 0:
        return
    err = np.abs(got - ref)
    scale = np.abs(ref).max()
    assert err.max() <= FFN_MAX_REL * scale + 1e-30, \
        f"{what}: max|err| {err.max():.3e} > {FFN_MAX_REL} * {scale:.3e}"
    mean_rel = err.sum() / max(np.abs(ref).sum(), 1e-30)
    assert mean_rel <= FFN_MEAN_REL, f"{what}: mean relative error {mean_rel:.3e}"


# Outputs that pass through e4m3 (the FP8 combine's expert outputs): the GPU
# and the oracle round the same way, but their inputs to an e4m3 rounding may
# differ by one bf16 rounding (fp32 vs float64 accumulation), and a value
# whose two versions straddle an e4m3 midpoint lands one e4m3 step apart - at
# most 2^-3 of its magnitude (4 significant bits). Such flips are rare, so
# the mean bar stays that of the bf16 outputs.
FP8_OUT_MAX_REL = 2.0 ** -3
# at most this share of elements may differ by more than one bf16 step
# (2^-7 relative) plus FP8_FAR_ABS of the largest magnitude
FP8_FAR_FRAC = 0.005
FP8_FAR_ABS = 1e-3


def assert_fp8_out_close(got: np.ndarray, ref: np.ndarray, what: str = "output"):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite values"
    if ref.size == 0:
        return
    err = np.abs(got - ref)
    scale = np.abs(ref).max()
    assert err.max() <= FP8_OUT_MAX_REL * scale + 1e-30, \
        f"{what}: max|err| {err.max():.3e} > {FP8_OUT_MAX_REL} * {scale:.3e}"
    mean_rel = err.sum() / max(np.abs(ref).sum(), 1e-30)
    assert mean_rel <= FFN_MEAN_REL, f"{what}: mean relative error {mean_rel:.3e}"
    # the 2^-3 bound admits the rare straddled e4m3 midpoint; a systematic
    # scale error would move most elements by more than a bf16 step
    far = float(np.mean(err > 2.0 ** -7 * np.abs(ref) + FP8_FAR_ABS * scale))
    print(f"{what}: {100 * far:.3f}% of elements beyond one bf16 step")
    assert far <= FP8_FAR_FRAC, f"{what}: {100 * far:.2f}% of elements beyond one bf16 step"


def oracle_logits_chunked(x: torch.Tensor, gate: torch.Tensor, bias, rows=None,
                          chunk: int = 8192) -> np.ndarray:
    """Oracle router logits for all tokens (or the given rows), computed in
    row chunks so float64 copies stay small. Row-wise, so chunking does not
    change any value."""
    g = np64(gate)
    b = None if bias is None else bias.detach().cpu().numpy().astype(np.float32)
    idx = np.arange(x.shape[0]) if rows is None else np.asarray(rows)
    out = np.empty((len(idx), g.shape[1]), np.float32)
    for s in range(0, len(idx), chunk):
        sel = torch.from_numpy(idx[s:s + chunk])
        out[s:s + chunk] = O.router_logits(np64(x[sel]), g, b)
    return out


def topk_margins(logits: np.ndarray, k: int) -> np.ndarray:
    """Smallest gap between consecutive entries of the sorted top-(k+1)
    logits of each token: the decisions a rounding change can flip."""
    lg = np.asarray(logits, np.float64)
    s = -np.sort(-lg, axis=1)[:, :min(k + 1, lg.shape[1])]
    if s.shape[1] < 2:
        return np.full(lg.shape[0], np.inf)
    return np.min(s[:, :-1] - s[:, 1:], axis=1)


def bf16_tensor(a: np.ndarray) -> torch.Tensor:
    """float64 values that are bf16-exact -> bf16 tensor (CPU)."""
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16)


def fill_nan_bf16(t: torch.Tensor):
    t.view(torch.int16).fill_(0x7FC0)


def routing_flips(gidx: np.ndarray, ref_idx: np.ndarray, margins: np.ndarray, what: str,
                  slack: float = 1.0, extra=None) -> np.ndarray:
    """Tokens whose GPU top-k differs from the oracle's: allowed only on a
    near-tie of the scores (top-k margin < NEAR_TIE * slack, plus twice the
    token's score error bound `extra[t]` when given), logged with their
    count. Returns their indices."""
    mism = np.nonzero((np.asarray(gidx) != np.asarray(ref_idx)).any(axis=1))[0]
    allowed = NEAR_TIE * slack + (0.0 if extra is None else 2.0 * np.asarray(extra)[mism])
    assert (margins[mism] < allowed).all(), (what, mism[:10], margins[mism][:10])
    print(f"{what}: {len(mism)} near-tie routing flips of {len(gidx)} tokens")
    return mism


def gumbel_fp32_error(u: np.ndarray, tau: float) -> np.ndarray:
    """Bound on |z_gpu - z_oracle| that the fp32 evaluation of the Gumbel
    noise g = -log(-log(u + 1e-9) + 1e-9) adds, per element, for fp32
    uniforms u (the oracle evaluates it in float64). In fp32, u + 1e-9
    rounds back to u wherever 1e-9 is below half an ulp of u, so the inner
    value t = -log(u + 1e-9) moves by up to 1e-9, and logf adds a few ulp
    (bounded here by 4 ulp, 8 * 2^-24 * t); the outer log turns an error dt
    into dt / (t + 1e-9), which grows as u approaches 1 (t -> 0). Divided by
    the temperature like the scores. The outer log's own rounding is a few
    ulp of g, inside the relative bound the tests apply to every score."""
    t = -np.log(np.asarray(u, np.float64) + 1e-9)
    return (2e-9 + 8.0 * 2.0 ** -24 * t) / (t + 1e-9) / tau


def assert_dispatch_on_gpu_indices(gidx: np.ndarray, p_ref: np.ndarray, E: int, C: int,
                                   routed=None, kept=None, offsets=None, dest_row=None,
                                   aux=None, aux_rel: float = STAT_REL):
    """Same-indices mode: the counts, capacity drops and permutation are an
    integer function of the top-k indices, so the oracle run on the GPU's
    own indices must reproduce the GPU's values bit for bit, whether or not
    a near-tie flipped a token. aux mixes those counts with the oracle's
    probabilities (float64) and must agree within aux_rel."""
    gidx = np.asarray(gidx)
    st = O.load_balance_stats(gidx, p_ref, E)
    d = O.dispatch_plan(gidx, E, C)
    if routed is not None:
        assert np.array_equal(np.asarray(routed), st.routed), "routed counts"
    if kept is not None:
        assert np.array_equal(np.asarray(kept), d.kept_counts), "kept counts"
    if offsets is not None:
        assert np.array_equal(np.asarray(offsets), d.offsets), "offsets"
    if dest_row is not None:
        assert np.array_equal(np.asarray(dest_row), d.dest_row), "dest_row"
    if aux is not None:
        assert abs(float(aux) - st.aux) <= aux_rel * st.aux, ("aux", float(aux), st.aux)
    return st, d
