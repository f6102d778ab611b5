"""The workspace-free dispatch entry point, for callers that cannot allocate
device memory (a plugin in a runtime that owns all device memory, or code
running while a stream is captured). Its scratch is a static device array
inside the library; this checks it against moe_permute with a caller
workspace, bit for bit, over two calls in a row (the second call must not
see the first call's leftovers). Collected last on purpose."""
import numpy as np
import pytest
import torch

import top_routing_expert_gb300 as moe
import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    moe.build()
    moe.load_library()


def _outputs(T, H, E, k):
    z = lambda shape, dt: torch.zeros(shape, dtype=dt, device=DEV)
    return dict(kept_counts=z(E, torch.int32), offsets=z(E + 1, torch.int32),
                dest_row=z((T, k), torch.int32),
                src_token=torch.full((T * k,), -1, dtype=torch.int32, device=DEV),
                x_perm=z((T * k, H), torch.bfloat16), dev_status=z(1, torch.int32))


def _compare(a, b):
    n = int(a["offsets"][-1].item())
    assert torch.equal(a["kept_counts"], b["kept_counts"])
    assert torch.equal(a["offsets"], b["offsets"])
    assert torch.equal(a["dest_row"], b["dest_row"])
    assert torch.equal(a["src_token"][:n], b["src_token"][:n])
    assert torch.equal(a["x_perm"][:n].view(torch.int16), b["x_perm"][:n].view(torch.int16))
    assert int(a["dev_status"].item()) == int(b["dev_status"].item()) == 0


def test_noalloc_permute_matches_workspace_permute_twice_in_a_row():
    cases = [(1000, 192, 12, 3, 1.0, 0.4, 1),   # ragged, drops
             (4096, 256, 16, 2, 1.0, 0.9, 2)]   # heavy skew, other sizes
    for T, H, E, k, cf, skew, seed in cases:
        s = moe.MoeShape.make(T, H, E, k, 64, cf)
        x = W.make_inputs(W.custom(T, H, E, k, 64, cf), seed=seed, with_weights=False)["x"].to(DEV)
        idx = W.make_topk_idx(T, E, k, seed=seed, skew=skew).to(DEV)
        ref = _outputs(T, H, E, k)
        moe.moe_permute(s, x, idx, ws=moe.Workspace(s), **ref)
        got = _outputs(T, H, E, k)
        moe.moe_permute_noalloc(s, x, idx, **got)
        torch.cuda.synchronize()
        _compare(ref, got)


def test_noalloc_same_shape_new_routing_without_status_and_index_only():
    """The same shape twice with different routing (stale tile counts or
    ranks from the first call would show), a call with no dev_status (the
    status word inside the static array), and an index-only call (x_perm
    NULL, src_token given), each bit for bit against moe_permute."""
    T, H, E, k, cf = 3000, 128, 24, 4, 1.0
    s = moe.MoeShape.make(T, H, E, k, 64, cf)
    ws = moe.Workspace(s)
    x = W.make_inputs(W.custom(T, H, E, k, 64, cf), seed=5, with_weights=False)["x"].to(DEV)
    for seed, skew in ((11, 0.0), (12, 0.7)):
        idx = W.make_topk_idx(T, E, k, seed=seed, skew=skew).to(DEV)
        ref = _outputs(T, H, E, k)
        moe.moe_permute(s, x, idx, ws=ws, **ref)
        got = _outputs(T, H, E, k)
        moe.moe_permute_noalloc(s, x, idx, **got)
        torch.cuda.synchronize()
        _compare(ref, got)
    got = _outputs(T, H, E, k)
    got.pop("dev_status")
    moe.moe_permute_noalloc(s, x, idx, **got)
    torch.cuda.synchronize()
    got["dev_status"] = torch.zeros(1, dtype=torch.int32, device=DEV)
    _compare(ref, got)
    got = _outputs(T, H, E, k)
    got["x_perm"] = None
    moe.moe_permute_noalloc(s, x, idx, **got)
    torch.cuda.synchronize()
    n = int(ref["offsets"][-1].item())
    assert torch.equal(got["dest_row"], ref["dest_row"])
    assert torch.equal(got["src_token"][:n], ref["src_token"][:n])
    assert torch.equal(got["offsets"], ref["offsets"])


def test_noalloc_rejects_shapes_beyond_its_static_scratch():
    T, H, E, k = 131072, 64, 128, 2
    s = moe.MoeShape.make(T, H, E, k, 64, 1.1)   # needs > 1 MiB of scratch
    idx = torch.zeros((T, k), dtype=torch.int32, device=DEV)
    x = torch.zeros((T, H), dtype=torch.bfloat16, device=DEV)
    xp = torch.zeros((T * k, H), dtype=torch.bfloat16, device=DEV)
    offs = torch.zeros(E + 1, dtype=torch.int32, device=DEV)
    with pytest.raises(moe.MoeError) as e:
        moe.moe_permute_noalloc(s, x, idx, None, offs, torch.empty_like(idx), None, xp)
    assert e.value.code == 3
    # the largest accepted shapes sit right at the limit: at E = 256 and
    # k = 8 the scratch is 2*r(4*256*ceil(T/128)) + r(8*T) + 2*r(1024) + 512
    # bytes; the first T past 1 MiB is refused, the one before it runs
    E, k = 256, 8
    r = lambda b: (b + 255) // 256 * 256
    need = lambda T: 2 * r(4 * E * -(-T // 128)) + r(T * k) + 2 * r(4 * E) + 512
    T = max(t for t in range(128, 70000, 128) if need(t) <= 1 << 20)
    assert need(T + 128) > 1 << 20
    for TT, ok in ((T, True), (T + 128, False)):
        s = moe.MoeShape.make(TT, 64, E, k, 64, 1.0)
        idx = W.make_topk_idx(TT, E, k, seed=3).to(DEV)
        x = torch.zeros((TT, 64), dtype=torch.bfloat16, device=DEV)
        out = _outputs(TT, 64, E, k)
        if ok:
            moe.moe_permute_noalloc(s, x, idx, **out)
        else:
            with pytest.raises(moe.MoeError):
                moe.moe_permute_noalloc(s, x, idx, **out)
    # a call right after a refused one still matches moe_permute
    ref = _outputs(T, 64, E, k)
    s = moe.MoeShape.make(T, 64, E, k, 64, 1.0)
    idx = W.make_topk_idx(T, E, k, seed=3).to(DEV)
    x = W.make_inputs(W.custom(T, 64, E, k, 64, 1.0), seed=9, with_weights=False)["x"].to(DEV)
    moe.moe_permute(s, x, idx, ws=moe.Workspace(s), **ref)
    got = _outputs(T, 64, E, k)
    moe.moe_permute_noalloc(s, x, idx, **got)
    torch.cuda.synchronize()
    _compare(ref, got)
