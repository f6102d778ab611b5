"""The C-ABI library without a GPU: it builds, loads, exports every symbol
the header declares, and its host-side logic (capacity, workspace size,
argument checks that run before any launch) behaves. No compute calls."""
import ctypes
import os
import re

import pytest

import top_routing_expert_gb300 as moe
import workloads as W
from oracle import moe_oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    moe.build()
    return moe.load_library()


def declared_functions():
    names = []
    inc = os.path.join(ROOT, "include")
    for f in sorted(os.listdir(inc)):
        if f.endswith(".h"):
            text = open(os.path.join(inc, f)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"\b(moe_\w+)\s*\(", text)
    return sorted(set(names))


def test_header_declares_the_abi():
    names = declared_functions()
    for n in ["moe_route", "moe_permute", "moe_expert_ffn", "moe_combine", "moe_layer_fwd"]:
        assert n in names
    assert set(names) == set(moe.EXPORTED_SYMBOLS)


def declared_signatures():
    """{name: [parameter type strings]} from the header's declarations."""
    text = ""
    inc = os.path.join(ROOT, "include")
    for f in sorted(os.listdir(inc)):
        if f.endswith(".h"):
            text += open(os.path.join(inc, f)).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    sigs = {}
    for m in re.finditer(r"\b(moe_\w+)\s*\(([^;{]*?)\)\s*;", text):
        params = [p.strip() for p in m.group(2).split(",") if p.strip()]
        if params == ["void"]:
            params = []
        sigs[m.group(1)] = params
    return sigs


def test_binding_argument_lists_match_the_header(lib):
    # every ctypes prototype has the header's arity, and scalars keep their C type
    kinds = {"int64_t": ctypes.c_int64, "double": ctypes.c_double, "float": ctypes.c_float,
             "size_t": ctypes.c_size_t}
    sigs = declared_signatures()
    assert set(sigs) == set(moe.EXPORTED_SYMBOLS)
    for name, params in sigs.items():
        argtypes = getattr(lib, name).argtypes or []
        assert len(argtypes) == len(params), (name, len(argtypes), params)
        for p, t in zip(params, argtypes):
            base = p.replace("const", "").split()[0] if "*" not in p else None
            if base in kinds:
                assert t is kinds[base], (name, p, t)
            elif "*" in p:
                assert t is not ctypes.c_float and t is not ctypes.c_double, (name, p, t)


def test_library_exports_every_declared_symbol(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n
    assert lib.moe_abi_version() == 1


@pytest.mark.parametrize("name", W.WORKLOAD_ORDER)
def test_capacity_matches_oracle_on_workloads(lib, name):
    w = W.get(name)
    assert moe.capacity(w.T, w.E, w.k, w.cf) == O.capacity(w.T, w.E, w.k, w.cf)


def test_capacity_edge_cases(lib):
    rng_cases = [(0, 4, 2, 1.0), (1, 256, 1, 0.01), (7, 3, 2, 0.5), (1000, 12, 3, 1.0),
                 (131072, 128, 2, 1.1), (10, 1, 1, 1.1), (3, 7, 3, 3.3)]
    for T, E, k, cf in rng_cases:
        assert moe.capacity(T, E, k, cf) == O.capacity(T, E, k, cf)
    assert moe.capacity(5, 0, 1, 1.0) == -1
    assert moe.capacity(5, 4, 1, float("nan")) == -1
    assert moe.capacity(5, 4, 1, -1.0) == -1


def _shape(T=64, H=128, E=8, k=2, h=128, cf=1.25):
    return moe.MoeShape.make(T, H, E, k, h, cf)


def _status(lib, s):
    n = ctypes.c_size_t()
    return lib.moe_workspace_size(ctypes.byref(s) if s is not None else None, ctypes.byref(n)), n.value


def test_workspace_size_and_shape_checks(lib):
    st, n = _status(lib, _shape())
    assert st == 0 and n > 0
    big = _status(lib, _shape(T=32768, H=4096, E=8, k=2, h=14336))[1]
    # holds at least x_perm, act and y_perm for T*k rows
    assert big >= 65536 * (4096 + 14336 + 4096) * 2
    assert _status(lib, None)[0] == 1                       # NULL
    assert _status(lib, _shape(T=-1))[0] == 2               # SHAPE
    assert _status(lib, _shape(cf=0.0))[0] == 2
    assert _status(lib, _shape(cf=float("inf")))[0] == 2
    assert _status(lib, _shape(E=257))[0] == 3              # UNSUPPORTED
    assert _status(lib, _shape(k=9, E=16))[0] == 3
    assert _status(lib, _shape(k=5, E=4))[0] == 3
    assert _status(lib, _shape(H=100))[0] == 3
    assert _status(lib, _shape(h=96))[0] == 3
    assert _status(lib, _shape(T=2 ** 30, k=2))[0] == 3
    assert _status(lib, _shape(T=0))[0] == 0


FAKE = 0x10000  # never dereferenced: every call below fails its host checks


def test_entry_points_reject_bad_arguments_before_launch(lib):
    s = _shape()
    ws_need = _status(lib, s)[1]
    P = ctypes.c_void_p
    f = P(FAKE)
    # NULL required pointers
    assert lib.moe_route(ctypes.byref(s), None, f, None, f, f, None, None, None, None, None,
                         f, ws_need, None) == 1
    assert lib.moe_layer_fwd(ctypes.byref(s), f, f, None, f, f, None, *[None] * 9,
                             f, ws_need, None, None) == 1
    assert lib.moe_combine(ctypes.byref(s), f, f, f, None, None) == 1
    # misaligned pointers
    assert lib.moe_combine(ctypes.byref(s), P(FAKE + 8), f, f, f, None) == 5
    assert lib.moe_permute(ctypes.byref(s), f, f, None, f, f, None, P(FAKE + 2), None, f,
                           ws_need, None) == 5
    # workspace too small / missing
    assert lib.moe_route_logits(ctypes.byref(s), f, f, f, None, None, None, None, f,
                                ws_need - 1, None) == 4
    assert lib.moe_permute(ctypes.byref(s), f, f, None, f, f, None, f, None, None, 0, None) == 1
    # no x_perm and no src_token: nothing to write the permutation to
    assert lib.moe_permute(ctypes.byref(s), f, f, None, f, f, None, None, None, f, ws_need,
                           None) == 1
    assert lib.moe_expert_ffn_gathered(ctypes.byref(s), f, None, f, f, f, f, f, None, f, ws_need,
                                       None) == 1
    # bad shapes
    bad = _shape(E=300)
    assert lib.moe_expert_ffn(ctypes.byref(bad), f, f, f, f, f, f, f, None, 0, None) == 3
    assert lib.moe_combine(None, f, f, f, f, None) == 1


def test_host_pipeline_entry_rejects_bad_arguments(lib):
    s = _shape()
    P = ctypes.c_void_p
    f = P(FAKE)
    n = ctypes.c_size_t()
    assert lib.moe_host_workspace_size(ctypes.byref(s), ctypes.byref(n)) == 0
    assert n.value > _status(lib, s)[1]          # layer workspace + I/O buffers
    ptrs = (P * 1)(f)
    # NULL streams / events / host pointer lists
    assert lib.moe_layer_fwd_host(ctypes.byref(s), 1, ptrs, ptrs, None, f, None, f, f, None, f,
                                  n.value, None, ptrs) == 1
    assert lib.moe_layer_fwd_host(ctypes.byref(s), 1, None, ptrs, None, f, None, f, f, None, f,
                                  n.value, ptrs, ptrs) == 1
    # workspace too small, negative count, bad shape
    assert lib.moe_layer_fwd_host(ctypes.byref(s), 1, ptrs, ptrs, None, f, None, f, f, None, f,
                                  n.value - 1, ptrs, ptrs) == 4
    assert lib.moe_layer_fwd_host(ctypes.byref(s), -1, ptrs, ptrs, None, f, None, f, f, None, f,
                                  n.value, ptrs, ptrs) == 2
    bad = _shape(H=96)
    assert lib.moe_layer_fwd_host(ctypes.byref(bad), 1, ptrs, ptrs, None, f, None, f, f, None, f,
                                  n.value, ptrs, ptrs) == 3


def test_status_strings(lib):
    for code in range(7):
        assert moe.status_str(code)
    assert moe.status_str(0) == "ok"


def test_fp8_entry_points_reject_bad_arguments(lib):
    s = _shape()
    P = ctypes.c_void_p
    f = P(FAKE)
    n8 = ctypes.c_size_t()
    assert lib.moe_workspace_size_fp8(ctypes.byref(s), ctypes.byref(n8)) == 0
    n = _status(lib, s)[1]
    A = 64 * 2
    # row scales, e4m3 act and its row maxima on top of the bf16 layer's scratch
    assert n8.value >= n + A * 128 + 3 * A * 4
    assert lib.moe_workspace_size_fp8(ctypes.byref(_shape(h=96)), ctypes.byref(n8)) == 3
    # weight quantisation: shape, NULL and alignment checks
    assert lib.moe_quantize_weights_fp8(0, 128, 128, f, f, f, None) == 2
    assert lib.moe_quantize_weights_fp8(8, 96, 128, f, f, f, None) == 3
    assert lib.moe_quantize_weights_fp8(8, 128, 128, None, f, f, None) == 1
    assert lib.moe_quantize_weights_fp8(8, 128, 128, f, P(FAKE + 4), f, None) == 5
    # the FP8 layer needs the FP8 workspace size
    assert lib.moe_layer_fwd_fp8(ctypes.byref(s), f, f, None, f, f, f, f, f, *[None] * 9,
                                 f, n, None, None) == 4
    assert lib.moe_layer_fwd_fp8(ctypes.byref(s), f, f, None, f, None, f, f, f, *[None] * 9,
                                 f, n8.value, None, None) == 1
    assert lib.moe_expert_ffn_fp8(ctypes.byref(s), f, None, f, f, f, f, f, f, f, None, None,
                                  None, f, n8.value, None) == 1
    # outputs: bf16 y_perm, or e4m3 y_q with y_scale - not both, not neither
    assert lib.moe_expert_ffn_fp8(ctypes.byref(s), f, f, f, f, f, f, f, f, f, f, f,
                                  None, f, n8.value, None) == 3
    assert lib.moe_expert_ffn_fp8(ctypes.byref(s), f, f, f, f, f, f, f, f, None, f, None,
                                  None, f, n8.value, None) == 1
    assert lib.moe_expert_ffn_fp8(ctypes.byref(s), f, f, f, f, f, f, f, f, None, None, None,
                                  None, f, n8.value, None) == 1
    assert lib.moe_combine_fp8(ctypes.byref(s), f, None, f, f, f, None) == 1
    assert lib.moe_combine_fp8(ctypes.byref(s), f, P(FAKE + 4), f, f, f, None) == 5
    assert lib.moe_permute_fp8(ctypes.byref(s), f, f, None, f, f, None, f, None, None, f, n,
                               None) == 1


def test_binding_sizes_every_tensor_argument():
    """Every tensor the binding hands to a shaped entry point has a minimum
    element count derived from the shape (the C ABI takes bare pointers and
    cannot check sizes), and the counts follow the header's layouts."""
    import inspect
    src = inspect.getsource(moe)
    names = set(re.findall(r'\ba\([A-Za-z0-9_.]+, torch\.[a-z0-9]+, "([A-Za-z0-9_]+)"\)', src))
    assert len(names) >= 30
    s = moe.MoeShape.make(1000, 384, 12, 3, 320, 1.0)
    A = 1000 * 3
    want = {"x": 1000 * 384, "gate": 384 * 12, "offsets": 13, "dest_row": A, "x_perm": A * 384,
            "act": A * 320, "W1": 12 * 384 * 320, "W2q": 12 * 384 * 320, "w1_scale": 12 * 320,
            "y_scale": A * 3, "noise_u": 1000 * 12, "aux": 1}
    for n in names:
        assert moe._need(s, n) >= 1, n
    for n, v in want.items():
        assert moe._need(s, n) == v, n


def test_expert_parallel_entries_reject_bad_arguments(lib):
    s = _shape()                         # E experts in all
    ws_need = _status(lib, s)[1]
    P = ctypes.c_void_p
    f = P(FAKE)
    args = lambda world, rank, routed_all, T_global, send: (
        ctypes.byref(s), world, rank, routed_all, T_global, f, f, None, f, f, None, f, send, None,
        f, ws_need, None)
    E = s.E
    assert lib.moe_ep_permute(*args(3 if E % 3 else 5, 0, None, 0, f)) == 2   # world must divide E
    assert lib.moe_ep_permute(*args(2, 2, None, 0, f)) == 2                  # rank out of range
    assert lib.moe_ep_permute(*args(2, -1, None, 0, f)) == 2
    assert lib.moe_ep_permute(*args(2, 0, None, 0, None)) == 1              # send_counts required
    assert lib.moe_ep_permute(*args(2, 0, f, s.T - 1, f)) == 2              # T_global < T
    assert lib.moe_ep_permute(*args(2, 0, P(FAKE + 4), s.T, f)) == 5        # misaligned
    # regroup: sizes and pointers
    assert lib.moe_ep_regroup(0, 4, 64, 10, 1, f, f, f, None, None) == 2
    assert lib.moe_ep_regroup(2, 200, 64, 10, 1, f, f, f, None, None) == 3  # > 256 experts
    assert lib.moe_ep_regroup(2, 4, 96, 10, 1, f, f, f, None, None) == 3    # H % 64
    assert lib.moe_ep_regroup(2, 4, 64, 10, 1, None, f, f, None, None) == 1
    assert lib.moe_ep_regroup(2, 4, 64, 10, 1, f, None, f, None, None) == 1
