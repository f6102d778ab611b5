"""Python binding of the GB300 MoE layer-forward library (C ABI in
include/moe_gb300.h). Argument marshalling only: every step of the layer
runs in the library's CUDA kernels, on the current torch CUDA stream.

The functions carry the C names. Tensors must be contiguous CUDA tensors of
the dtypes below; outputs are written in place. A non-OK status raises
``MoeError``. There is no CPU path: without the built library (see
``build()``) importing the native layer fails loudly.
"""
from __future__ import annotations

import ctypes
import functools
import os
from typing import Optional, Sequence

import torch

from ._build import LIB, build  # noqa: F401  (re-exported)

__all__ = [
    "MoeError", "MoeShape", "load_library", "capacity", "workspace_size", "status_str",
    "abi_version", "moe_route", "moe_route_logits", "moe_permute", "moe_expert_ffn",
    "moe_combine", "moe_layer_fwd", "moe_permute_noalloc", "moe_layer_fwd_host",
    "host_workspace_size", "HostPipeline", "moe_route_gumbel", "moe_layer_fwd_gumbel",
    "workspace_size_fp8", "moe_quantize_weights_fp8", "moe_layer_fwd_host_fp8", "moe_permute_fp8", "moe_expert_ffn_fp8",
    "moe_layer_fwd_fp8", "moe_combine_fp8", "Fp8Weights", "moe_expert_ffn_gathered",
    "moe_ep_permute", "moe_ep_regroup", "DevicePipeline", "moe_layer_fwd_pipelined",
    "Workspace", "DEV_BAD_INDEX", "DEV_DUP_INDEX",
    "DEV_NONFINITE", "DEV_TIMEOUT", "LAYER_NUM_EVENTS", "EXPORTED_SYMBOLS", "build",
]

DEV_BAD_INDEX, DEV_DUP_INDEX, DEV_NONFINITE, DEV_TIMEOUT = 1, 2, 4, 8
LAYER_NUM_EVENTS = 7
EXPORTED_SYMBOLS = ["moe_abi_version", "moe_capacity", "moe_workspace_size", "moe_status_str",
                    "moe_route", "moe_route_logits", "moe_permute", "moe_expert_ffn",
                    "moe_combine", "moe_layer_fwd", "moe_permute_noalloc",
                    "moe_host_workspace_size", "moe_layer_fwd_host", "moe_route_gumbel",
                    "moe_layer_fwd_gumbel", "moe_workspace_size_fp8", "moe_quantize_weights_fp8",
                    "moe_permute_fp8", "moe_expert_ffn_fp8", "moe_layer_fwd_fp8",
                    "moe_combine_fp8", "moe_expert_ffn_gathered", "moe_host_workspace_size_fp8",
                    "moe_layer_fwd_host_fp8", "moe_ep_permute", "moe_ep_regroup",
                    "moe_pipelined_workspace_size", "moe_layer_fwd_pipelined"]


class MoeError(RuntimeError):
    def __init__(self, fn: str, code: int, text: str):
        super().__init__(f"{fn} failed: status {code} ({text})")
        self.code = code


class MoeShape(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("H", ctypes.c_int64), ("E", ctypes.c_int64),
                ("top_k", ctypes.c_int64), ("h", ctypes.c_int64),
                ("capacity_factor", ctypes.c_double)]

    @classmethod
    def make(cls, T, H, E, k, h, cf) -> "MoeShape":
        return cls(int(T), int(H), int(E), int(k), int(h), float(cf))


_lib: Optional[ctypes.CDLL] = None
_P = ctypes.c_void_p


def load_library(path: Optional[str] = None) -> ctypes.CDLL:
    """Loads the built library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or os.environ.get("MOE_GB300_LIB", LIB)
    if not os.path.exists(path):
        raise RuntimeError(f"native library {path} is missing: run top_routing_expert_gb300.build()")
    lib = ctypes.CDLL(path)
    S = ctypes.POINTER(MoeShape)
    lib.moe_abi_version.restype = ctypes.c_int
    lib.moe_capacity.restype = ctypes.c_int64
    lib.moe_capacity.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_double]
    lib.moe_workspace_size.restype = ctypes.c_int
    lib.moe_workspace_size.argtypes = [S, ctypes.POINTER(ctypes.c_size_t)]
    lib.moe_status_str.restype = ctypes.c_char_p
    lib.moe_status_str.argtypes = [ctypes.c_int]
    lib.moe_route.restype = ctypes.c_int
    lib.moe_route.argtypes = [S] + [_P] * 11 + [ctypes.c_size_t, _P]
    lib.moe_route_logits.restype = ctypes.c_int
    lib.moe_route_logits.argtypes = [S] + [_P] * 8 + [ctypes.c_size_t, _P]
    lib.moe_permute.restype = ctypes.c_int
    lib.moe_permute.argtypes = [S] + [_P] * 9 + [ctypes.c_size_t, _P]
    lib.moe_expert_ffn.restype = ctypes.c_int
    lib.moe_expert_ffn.argtypes = [S] + [_P] * 8 + [ctypes.c_size_t, _P]
    lib.moe_combine.restype = ctypes.c_int
    lib.moe_combine.argtypes = [S] + [_P] * 5
    lib.moe_layer_fwd.restype = ctypes.c_int
    lib.moe_layer_fwd.argtypes = [S] + [_P] * 16 + [ctypes.c_size_t, _P, _P]
    lib.moe_permute_noalloc.restype = ctypes.c_int
    lib.moe_permute_noalloc.argtypes = [S] + [_P] * 9
    lib.moe_route_gumbel.restype = ctypes.c_int
    lib.moe_route_gumbel.argtypes = [S] + [_P] * 4 + [ctypes.c_float] + [_P] * 8 + [ctypes.c_size_t, _P]
    lib.moe_layer_fwd_gumbel.restype = ctypes.c_int
    lib.moe_layer_fwd_gumbel.argtypes = [S] + [_P] * 4 + [ctypes.c_float] + [_P] * 13 + [ctypes.c_size_t, _P, _P]
    lib.moe_host_workspace_size.restype = ctypes.c_int
    lib.moe_host_workspace_size.argtypes = [S, ctypes.POINTER(ctypes.c_size_t)]
    lib.moe_layer_fwd_host.restype = ctypes.c_int
    lib.moe_layer_fwd_host.argtypes = [S, ctypes.c_int64] + [_P] * 9 + [ctypes.c_size_t, _P, _P]
    lib.moe_host_workspace_size_fp8.restype = ctypes.c_int
    lib.moe_host_workspace_size_fp8.argtypes = [S, ctypes.POINTER(ctypes.c_size_t)]
    lib.moe_layer_fwd_host_fp8.restype = ctypes.c_int
    lib.moe_layer_fwd_host_fp8.argtypes = [S, ctypes.c_int64] + [_P] * 11 + [ctypes.c_size_t, _P, _P]
    lib.moe_workspace_size_fp8.restype = ctypes.c_int
    lib.moe_workspace_size_fp8.argtypes = [S, ctypes.POINTER(ctypes.c_size_t)]
    lib.moe_quantize_weights_fp8.restype = ctypes.c_int
    lib.moe_quantize_weights_fp8.argtypes = [ctypes.c_int64] * 3 + [_P] * 4
    lib.moe_permute_fp8.restype = ctypes.c_int
    lib.moe_permute_fp8.argtypes = [S] + [_P] * 10 + [ctypes.c_size_t, _P]
    lib.moe_expert_ffn_fp8.restype = ctypes.c_int
    lib.moe_expert_ffn_fp8.argtypes = [S] + [_P] * 13 + [ctypes.c_size_t, _P]
    lib.moe_expert_ffn_gathered.restype = ctypes.c_int
    lib.moe_expert_ffn_gathered.argtypes = [S] + [_P] * 9 + [ctypes.c_size_t, _P]
    lib.moe_combine_fp8.restype = ctypes.c_int
    lib.moe_combine_fp8.argtypes = [S] + [_P] * 6
    lib.moe_layer_fwd_fp8.restype = ctypes.c_int
    lib.moe_layer_fwd_fp8.argtypes = [S] + [_P] * 18 + [ctypes.c_size_t, _P, _P]
    lib.moe_pipelined_workspace_size.restype = ctypes.c_int
    lib.moe_pipelined_workspace_size.argtypes = [S, ctypes.POINTER(ctypes.c_size_t)]
    lib.moe_layer_fwd_pipelined.restype = ctypes.c_int
    lib.moe_layer_fwd_pipelined.argtypes = [S, ctypes.c_int64] + [_P] * 9 + [ctypes.c_size_t,
                                                                           _P, _P]
    I64 = ctypes.c_int64
    lib.moe_ep_permute.restype = ctypes.c_int
    lib.moe_ep_permute.argtypes = [S, I64, I64, _P, I64] + [_P] * 10 + [ctypes.c_size_t, _P]
    lib.moe_ep_regroup.restype = ctypes.c_int
    lib.moe_ep_regroup.argtypes = [I64, I64, I64, I64, ctypes.c_int] + [_P] * 5
    _lib = lib
    return lib


# ------------------------------------------------------------ helpers ----

def _ptr(t: Optional[torch.Tensor], dtype=None, name="tensor", numel: Optional[int] = None
         ) -> Optional[int]:
    """Device address of a contiguous CUDA tensor of `dtype` on the current
    device holding at least `numel` elements (the C ABI takes bare pointers
    and cannot check sizes, so an undersized buffer is refused here)."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.get_device() != torch.cuda.current_device():
        raise ValueError(f"{name} is on {t.device}, the current device is "
                         f"cuda:{torch.cuda.current_device()}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if numel is not None and t.numel() < numel:
        raise ValueError(f"{name} holds {t.numel()} elements, the shape needs {numel}")
    return t.data_ptr()


def _need(s: "MoeShape", name: str) -> int:
    """Elements the named argument must hold for shape s (layouts as in
    include/moe_gb300.h)."""
    return _need_table(s.T, s.H, s.E, s.top_k, s.h)[name]


@functools.lru_cache(maxsize=64)
def _need_table(T: int, H: int, E: int, k: int, h: int) -> dict:
    A = T * k
    return {
        "x": T * H, "y": T * H, "gate": H * E, "gate_bias": E, "noise_u": T * E,
        "logits": T * E, "logits_out": T * E, "scores_out": T * E,
        "topk_idx": A, "topk_w": A, "dest_row": A, "src_token": A,
        "routed_counts": E, "P": E, "kept_counts": E, "offsets": E + 1,
        "aux": 1, "dev_status": 1,
        "x_perm": A * H, "y_perm": A * H, "act": A * h, "x_q": A * H, "y_q": A * H,
        "x_scale": A, "y_scale": A * ((H + 127) // 128),
        "W1": E * H * h, "W2": E * h * H, "W1q": E * h * H, "W2q": E * H * h,
        "w1_scale": E * h, "w2_scale": E * H,
    }


class _Args:
    """Argument checks of one shaped entry-point call: the shape, its size
    table and the current device are looked up once, then each tensor is
    checked as `_ptr` does (contiguous CUDA tensor of the dtype on the current
    device, at least the elements the shape needs) and its address returned."""
    __slots__ = ("shape", "need", "dev")

    def __init__(self, shape):
        self.shape = _shape(shape)
        s = self.shape
        self.need = _need_table(s.T, s.H, s.E, s.top_k, s.h)
        self.dev = torch.cuda.current_device()

    def __call__(self, t: Optional[torch.Tensor], dtype, name: str) -> Optional[int]:
        if t is None:
            return None
        if not t.is_cuda or t.get_device() != self.dev or not t.is_contiguous() \
                or t.dtype != dtype or t.numel() < self.need[name]:
            return _ptr(t, dtype, name, self.need[name])   # raises with the reason
        return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(fn: str, code: int):
    if code != 0:
        raise MoeError(fn, code, status_str(code))


def _shape(s) -> MoeShape:
    if isinstance(s, MoeShape):
        return s
    if isinstance(s, dict):
        return MoeShape.make(s["T"], s["H"], s["E"], s["k"], s["h"], s["cf"])
    return MoeShape.make(*s)


# ---------------------------------------------------------- host calls ----

def abi_version() -> int:
    return load_library().moe_abi_version()


def capacity(T: int, E: int, k: int, cf: float) -> int:
    return load_library().moe_capacity(T, E, k, cf)


def status_str(code: int) -> str:
    return load_library().moe_status_str(code).decode()


def workspace_size(shape) -> int:
    n = ctypes.c_size_t(0)
    _check("moe_workspace_size", load_library().moe_workspace_size(ctypes.byref(_shape(shape)), ctypes.byref(n)))
    return n.value


def workspace_size_fp8(shape) -> int:
    n = ctypes.c_size_t(0)
    _check("moe_workspace_size_fp8",
           load_library().moe_workspace_size_fp8(ctypes.byref(_shape(shape)), ctypes.byref(n)))
    return n.value


class Workspace:
    """Caller-owned device scratch for one shape (a torch uint8 tensor);
    fp8=True sizes it for the FP8 entry points too."""

    def __init__(self, shape, device="cuda", fp8: bool = False):
        self.shape = _shape(shape)
        self.nbytes = workspace_size_fp8(self.shape) if fp8 else workspace_size(self.shape)
        self.buf = torch.empty(max(self.nbytes, 256), dtype=torch.uint8, device=device)

    @property
    def ptr(self) -> int:
        return self.buf.data_ptr()


def _ws(ws: Workspace | None, shape: MoeShape):
    if ws is None:
        return None, 0
    return ws.ptr, ws.nbytes


def _events(events):
    if events is None:
        return None
    if len(events) != LAYER_NUM_EVENTS:
        raise ValueError(f"events must hold {LAYER_NUM_EVENTS} torch.cuda.Event")
    return (ctypes.c_void_p * LAYER_NUM_EVENTS)(*[e.cuda_event for e in events])


# ------------------------------------------------------------ kernels ----

def moe_route(shape, x, gate, gate_bias, topk_idx, topk_w, routed_counts=None, P=None,
              aux=None, logits_out=None, dev_status=None, ws: Workspace | None = None,
              stream=None):
    a = _Args(shape)
    s = a.shape
    wp, wn = _ws(ws, s)
    _check("moe_route", load_library().moe_route(
        ctypes.byref(s), a(x, torch.bfloat16, "x"), a(gate, torch.bfloat16, "gate"),
        a(gate_bias, torch.float32, "gate_bias"), a(topk_idx, torch.int32, "topk_idx"),
        a(topk_w, torch.float32, "topk_w"),
        a(routed_counts, torch.int32, "routed_counts"),
        a(P, torch.float32, "P"), a(aux, torch.float32, "aux"),
        a(logits_out, torch.float32, "logits_out"),
        a(dev_status, torch.int32, "dev_status"),
        wp, wn, _stream(stream)))


def moe_route_logits(shape, logits, topk_idx, topk_w, routed_counts=None, P=None, aux=None,
                     dev_status=None, ws: Workspace | None = None, stream=None):
    a = _Args(shape)
    s = a.shape
    wp, wn = _ws(ws, s)
    _check("moe_route_logits", load_library().moe_route_logits(
        ctypes.byref(s), a(logits, torch.float32, "logits"),
        a(topk_idx, torch.int32, "topk_idx"), a(topk_w, torch.float32, "topk_w"),
        a(routed_counts, torch.int32, "routed_counts"), a(P, torch.float32, "P"),
        a(aux, torch.float32, "aux"), a(dev_status, torch.int32, "dev_status"),
        wp, wn, _stream(stream)))


def moe_permute(shape, x, topk_idx, kept_counts, offsets, dest_row, src_token, x_perm,
                dev_status=None, ws: Workspace | None = None, stream=None):
    a = _Args(shape)
    s = a.shape
    wp, wn = _ws(ws, s)
    _check("moe_permute", load_library().moe_permute(
        ctypes.byref(s), a(x, torch.bfloat16, "x"),
        a(topk_idx, torch.int32, "topk_idx"),
        a(kept_counts, torch.int32, "kept_counts"), a(offsets, torch.int32, "offsets"),
        a(dest_row, torch.int32, "dest_row"), a(src_token, torch.int32, "src_token"),
        a(x_perm, torch.bfloat16, "x_perm"), a(dev_status, torch.int32, "dev_status"),
        wp, wn, _stream(stream)))


def moe_expert_ffn(shape, x_perm, offsets, W1, W2, act, y_perm, dev_status=None,
                   ws: Workspace | None = None, stream=None):
    a = _Args(shape)
    s = a.shape
    wp, wn = _ws(ws, s)
    _check("moe_expert_ffn", load_library().moe_expert_ffn(
        ctypes.byref(s), a(x_perm, torch.bfloat16, "x_perm"),
        a(offsets, torch.int32, "offsets"),
        a(W1, torch.bfloat16, "W1"), a(W2, torch.bfloat16, "W2"),
        a(act, torch.bfloat16, "act"), a(y_perm, torch.bfloat16, "y_perm"),
        a(dev_status, torch.int32, "dev_status"), wp, wn, _stream(stream)))


def moe_expert_ffn_gathered(shape, x, src_token, offsets, W1, W2, act, y_perm, dev_status=None,
                            ws: Workspace | None = None, stream=None):
    """moe_expert_ffn on x[src_token] without the permuted copy: GEMM1
    gathers its A rows from x by TMA."""
    a = _Args(shape)
    s = a.shape
    wp, wn = _ws(ws, s)
    _check("moe_expert_ffn_gathered", load_library().moe_expert_ffn_gathered(
        ctypes.byref(s), a(x, torch.bfloat16, "x"),
        a(src_token, torch.int32, "src_token"),
        a(offsets, torch.int32, "offsets"), a(W1, torch.bfloat16, "W1"),
        a(W2, torch.bfloat16, "W2"), a(act, torch.bfloat16, "act"),
        a(y_perm, torch.bfloat16, "y_perm"), a(dev_status, torch.int32, "dev_status"),
        wp, wn, _stream(stream)))


def moe_combine(shape, y_perm, dest_row, topk_w, y, stream=None):
    a = _Args(shape)
    s = a.shape
    _check("moe_combine", load_library().moe_combine(
        ctypes.byref(s), a(y_perm, torch.bfloat16, "y_perm"),
        a(dest_row, torch.int32, "dest_row"),
        a(topk_w, torch.float32, "topk_w"), a(y, torch.bfloat16, "y"), _stream(stream)))


def moe_layer_fwd(shape, x, gate, gate_bias, W1, W2, y, aux=None, topk_idx=None, topk_w=None,
                  routed_counts=None, P=None, kept_counts=None, offsets=None, dest_row=None,
                  dev_status=None, ws: Workspace | None = None, stream=None,
                  events: Optional[Sequence[torch.cuda.Event]] = None):
    a = _Args(shape)
    s = a.shape
    wp, wn = _ws(ws, s)
    ev = _events(events)
    _check("moe_layer_fwd", load_library().moe_layer_fwd(
        ctypes.byref(s), a(x, torch.bfloat16, "x"), a(gate, torch.bfloat16, "gate"),
        a(gate_bias, torch.float32, "gate_bias"), a(W1, torch.bfloat16, "W1"),
        a(W2, torch.bfloat16, "W2"), a(y, torch.bfloat16, "y"),
        a(aux, torch.float32, "aux"),
        a(topk_idx, torch.int32, "topk_idx"), a(topk_w, torch.float32, "topk_w"),
        a(routed_counts, torch.int32, "routed_counts"), a(P, torch.float32, "P"),
        a(kept_counts, torch.int32, "kept_counts"), a(offsets, torch.int32, "offsets"),
        a(dest_row, torch.int32, "dest_row"), a(dev_status, torch.int32, "dev_status"),
        wp, wn, _stream(stream), ev))


def moe_permute_noalloc(shape, x, topk_idx, kept_counts, offsets, dest_row, src_token, x_perm,
                        dev_status=None, stream=None):
    """moe_permute without a workspace, for callers that cannot allocate
    device memory: its scratch is a static 1 MiB device array inside the
    library (one per GPU). Larger shapes raise MoeError (unsupported).
    Calls that overlap on the GPU share that array and must be serialised;
    make the first call on a device before any stream capture."""
    a = _Args(shape)
    s = a.shape
    _check("moe_permute_noalloc", load_library().moe_permute_noalloc(
        ctypes.byref(s), a(x, torch.bfloat16, "x"),
        a(topk_idx, torch.int32, "topk_idx"),
        a(kept_counts, torch.int32, "kept_counts"), a(offsets, torch.int32, "offsets"),
        a(dest_row, torch.int32, "dest_row"), a(src_token, torch.int32, "src_token"),
        a(x_perm, torch.bfloat16, "x_perm"), a(dev_status, torch.int32, "dev_status"),
        _stream(stream)))


def host_workspace_size(shape) -> int:
    n = ctypes.c_size_t(0)
    _check("moe_host_workspace_size",
           load_library().moe_host_workspace_size(ctypes.byref(_shape(shape)), ctypes.byref(n)))
    return n.value


def _host_ptr(t: torch.Tensor, name: str, numel: int) -> int:
    if t.is_cuda:
        raise ValueError(f"{name} must be a host tensor")
    if not t.is_contiguous() or t.dtype != torch.bfloat16:
        raise ValueError(f"{name} must be a contiguous bf16 host tensor")
    if t.numel() < numel:
        raise ValueError(f"{name} holds {t.numel()} elements, the shape needs {numel}")
    return t.data_ptr()


class HostPipeline:
    """Owns what moe_layer_fwd_host needs besides the weights: the device
    workspace, three CUDA streams (compute, copy-in, copy-out) and six
    events. Host token/output tensors should be pinned for the copies to
    overlap the layer. fp8=True sizes it for moe_layer_fwd_host_fp8 (run
    with an Fp8Weights in place of W1 and W2 there)."""

    def __init__(self, shape, device="cuda", fp8: bool = False):
        self.shape = _shape(shape)
        self.fp8 = fp8
        if fp8:
            n = ctypes.c_size_t(0)
            _check("moe_host_workspace_size_fp8", load_library().moe_host_workspace_size_fp8(
                ctypes.byref(self.shape), ctypes.byref(n)))
            self.nbytes = n.value
        else:
            self.nbytes = host_workspace_size(self.shape)
        self.buf = torch.empty(max(self.nbytes, 256), dtype=torch.uint8, device=device)
        self.streams = [torch.cuda.Stream(device=device) for _ in range(3)]
        self.events = [torch.cuda.Event() for _ in range(6)]
        for e in self.events:          # create the handles
            e.record(self.streams[0])

    def run(self, x_host, y_host, gate, gate_bias, W1, W2, aux_host=None, dev_status=None):
        """Enqueues the layer over the micro-batches x_host[i] -> y_host[i]
        (lists of [T,H] bf16 host tensors); returns the copy-out stream,
        which the caller synchronises before reading y_host / aux_host."""
        n = len(x_host)
        if len(y_host) != n:
            raise ValueError("x_host and y_host need the same length")
        TH = self.shape.T * self.shape.H
        xs = (ctypes.c_void_p * max(n, 1))(*[_host_ptr(t, "x_host", TH) for t in x_host])
        ys = (ctypes.c_void_p * max(n, 1))(*[_host_ptr(t, "y_host", TH) for t in y_host])
        aux = None
        if aux_host is not None:
            if aux_host.is_cuda or aux_host.dtype != torch.float32 or aux_host.numel() < n:
                raise ValueError("aux_host must be a float32 host tensor with >= n entries")
            aux = aux_host.data_ptr()
        a = _Args(self.shape)
        st = (ctypes.c_void_p * 3)(*[s.cuda_stream for s in self.streams])
        ev = (ctypes.c_void_p * 6)(*[e.cuda_event for e in self.events])
        if self.fp8:
            q = W1  # an Fp8Weights
            _check("moe_layer_fwd_host_fp8", load_library().moe_layer_fwd_host_fp8(
                ctypes.byref(self.shape), n, xs, ys, aux,
                a(gate, torch.bfloat16, "gate"),
                a(gate_bias, torch.float32, "gate_bias"),
                a(q.W1q, torch.uint8, "W1q"),
                a(q.w1_scale, torch.float32, "w1_scale"),
                a(q.W2q, torch.uint8, "W2q"),
                a(q.w2_scale, torch.float32, "w2_scale"),
                a(dev_status, torch.int32, "dev_status"), self.buf.data_ptr(),
                self.nbytes,
                st, ev))
            return self.streams[2]
        _check("moe_layer_fwd_host", load_library().moe_layer_fwd_host(
            ctypes.byref(self.shape), n, xs, ys, aux,
            a(gate, torch.bfloat16, "gate"),
            a(gate_bias, torch.float32, "gate_bias"),
            a(W1, torch.bfloat16, "W1"),
            a(W2, torch.bfloat16, "W2"),
            a(dev_status, torch.int32, "dev_status"),
            self.buf.data_ptr(), self.nbytes, st, ev))
        return self.streams[2]


def moe_layer_fwd_host(pipeline: HostPipeline, x_host, y_host, gate, gate_bias, W1, W2,
                       aux_host=None, dev_status=None):
    """C-ABI name for HostPipeline.run."""
    return pipeline.run(x_host, y_host, gate, gate_bias, W1, W2, aux_host, dev_status)


def moe_layer_fwd_host_fp8(pipeline: HostPipeline, x_host, y_host, gate, gate_bias,
                           q: "Fp8Weights", aux_host=None, dev_status=None):
    """C-ABI name for HostPipeline(fp8=True).run with quantised weights."""
    if not pipeline.fp8:
        raise ValueError("the pipeline was not made with fp8=True")
    return pipeline.run(x_host, y_host, gate, gate_bias, q, None, aux_host, dev_status)


def moe_route_gumbel(shape, x, gate, gate_bias, noise_u, temperature, topk_idx, topk_w,
                     routed_counts=None, P=None, aux=None, scores_out=None, dev_status=None,
                     ws: Workspace | None = None, stream=None):
    """Training router: top-k of (x.gate + bias + gumbel(noise_u)) / temperature."""
    a = _Args(shape)
    s = a.shape
    wp, wn = _ws(ws, s)
    _check("moe_route_gumbel", load_library().moe_route_gumbel(
        ctypes.byref(s), a(x, torch.bfloat16, "x"), a(gate, torch.bfloat16, "gate"),
        a(gate_bias, torch.float32, "gate_bias"), a(noise_u, torch.float32, "noise_u"),
        float(temperature), a(topk_idx, torch.int32, "topk_idx"),
        a(topk_w, torch.float32, "topk_w"),
        a(routed_counts, torch.int32, "routed_counts"),
        a(P, torch.float32, "P"), a(aux, torch.float32, "aux"),
        a(scores_out, torch.float32, "scores_out"),
        a(dev_status, torch.int32, "dev_status"),
        wp, wn, _stream(stream)))


def moe_layer_fwd_gumbel(shape, x, gate, gate_bias, noise_u, temperature, W1, W2, y, aux=None,
                         topk_idx=None, topk_w=None, routed_counts=None, P=None,
                         kept_counts=None, offsets=None, dest_row=None, dev_status=None,
                         ws: Workspace | None = None, stream=None, events=None):
    """moe_layer_fwd with the Gumbel training router."""
    a = _Args(shape)
    s = a.shape
    wp, wn = _ws(ws, s)
    ev = _events(events)
    _check("moe_layer_fwd_gumbel", load_library().moe_layer_fwd_gumbel(
        ctypes.byref(s), a(x, torch.bfloat16, "x"), a(gate, torch.bfloat16, "gate"),
        a(gate_bias, torch.float32, "gate_bias"), a(noise_u, torch.float32, "noise_u"),
        float(temperature), a(W1, torch.bfloat16, "W1"), a(W2, torch.bfloat16, "W2"),
        a(y, torch.bfloat16, "y"), a(aux, torch.float32, "aux"),
        a(topk_idx, torch.int32, "topk_idx"), a(topk_w, torch.float32, "topk_w"),
        a(routed_counts, torch.int32, "routed_counts"), a(P, torch.float32, "P"),
        a(kept_counts, torch.int32, "kept_counts"), a(offsets, torch.int32, "offsets"),
        a(dest_row, torch.int32, "dest_row"), a(dev_status, torch.int32, "dev_status"),
        wp, wn, _stream(stream), ev))


# --------------------------------------------------------------- FP8 ----

def moe_quantize_weights_fp8(W, Wq, w_scale, stream=None):
    """W [E,K,N] bf16 -> Wq [E,N,K] e4m3 bytes (uint8) and w_scale [E,N] fp32."""
    if W.dim() != 3:
        raise ValueError("W must be [E, K, N]")
    E, K, N = W.shape
    _check("moe_quantize_weights_fp8", load_library().moe_quantize_weights_fp8(
        E, K, N, _ptr(W, torch.bfloat16, "W"), _ptr(Wq, torch.uint8, "Wq", E * K * N),
        _ptr(w_scale, torch.float32, "w_scale", E * N), _stream(stream)))


class Fp8Weights:
    """The expert weights quantised for the FP8 layer: W1q [E,h,H], W2q
    [E,H,h] (e4m3 bytes, each output column a row) and their column scales
    w1_scale [E,h], w2_scale [E,H]."""

    def __init__(self, W1, W2, stream=None):
        E, H, h = W1.shape
        dev = W1.device
        self.W1q = torch.empty((E, h, H), dtype=torch.uint8, device=dev)
        self.w1_scale = torch.empty((E, h), dtype=torch.float32, device=dev)
        self.W2q = torch.empty((E, H, h), dtype=torch.uint8, device=dev)
        self.w2_scale = torch.empty((E, H), dtype=torch.float32, device=dev)
        moe_quantize_weights_fp8(W1, self.W1q, self.w1_scale, stream)
        moe_quantize_weights_fp8(W2, self.W2q, self.w2_scale, stream)


def moe_permute_fp8(shape, x, topk_idx, kept_counts, offsets, dest_row, src_token, x_q, x_scale,
                    dev_status=None, ws: Workspace | None = None, stream=None):
    """moe_permute with an e4m3 payload: x_q [T*k,H] uint8, x_scale [T*k] fp32."""
    a = _Args(shape)
    s = a.shape
    wp, wn = _ws(ws, s)
    _check("moe_permute_fp8", load_library().moe_permute_fp8(
        ctypes.byref(s), a(x, torch.bfloat16, "x"),
        a(topk_idx, torch.int32, "topk_idx"),
        a(kept_counts, torch.int32, "kept_counts"), a(offsets, torch.int32, "offsets"),
        a(dest_row, torch.int32, "dest_row"), a(src_token, torch.int32, "src_token"),
        a(x_q, torch.uint8, "x_q"), a(x_scale, torch.float32, "x_scale"),
        a(dev_status, torch.int32, "dev_status"), wp, wn, _stream(stream)))


def moe_expert_ffn_fp8(shape, x_q, x_scale, offsets, q: Fp8Weights, act, y_perm=None,
                       y_q=None, y_scale=None, dev_status=None, ws: Workspace | None = None,
                       stream=None):
    """Expert FFN on e4m3 rows; outputs bf16 y_perm, or e4m3 y_q [T*k,H]
    (uint8) with y_scale [T*k, ceil(H/128)] block scales. ws must be an
    fp8=True workspace."""
    a = _Args(shape)
    s = a.shape
    wp, wn = _ws(ws, s)
    _check("moe_expert_ffn_fp8", load_library().moe_expert_ffn_fp8(
        ctypes.byref(s), a(x_q, torch.uint8, "x_q"),
        a(x_scale, torch.float32, "x_scale"),
        a(offsets, torch.int32, "offsets"), a(q.W1q, torch.uint8, "W1q"),
        a(q.w1_scale, torch.float32, "w1_scale"), a(q.W2q, torch.uint8, "W2q"),
        a(q.w2_scale, torch.float32, "w2_scale"), a(act, torch.bfloat16, "act"),
        a(y_perm, torch.bfloat16, "y_perm"), a(y_q, torch.uint8, "y_q"),
        a(y_scale, torch.float32, "y_scale"), a(dev_status, torch.int32, "dev_status"),
        wp, wn, _stream(stream)))


def moe_combine_fp8(shape, y_q, y_scale, dest_row, topk_w, y, stream=None):
    """Combine of e4m3 expert outputs with 128-column block scales."""
    a = _Args(shape)
    s = a.shape
    _check("moe_combine_fp8", load_library().moe_combine_fp8(
        ctypes.byref(s), a(y_q, torch.uint8, "y_q"),
        a(y_scale, torch.float32, "y_scale"),
        a(dest_row, torch.int32, "dest_row"), a(topk_w, torch.float32, "topk_w"),
        a(y, torch.bfloat16, "y"), _stream(stream)))


def moe_layer_fwd_fp8(shape, x, gate, gate_bias, q: Fp8Weights, y, aux=None, topk_idx=None,
                      topk_w=None, routed_counts=None, P=None, kept_counts=None, offsets=None,
                      dest_row=None, dev_status=None, ws: Workspace | None = None, stream=None,
                      events=None):
    """moe_layer_fwd with the FP8 dispatch and expert FFN; ws must be an
    fp8=True workspace."""
    a = _Args(shape)
    s = a.shape
    wp, wn = _ws(ws, s)
    ev = _events(events)
    _check("moe_layer_fwd_fp8", load_library().moe_layer_fwd_fp8(
        ctypes.byref(s), a(x, torch.bfloat16, "x"), a(gate, torch.bfloat16, "gate"),
        a(gate_bias, torch.float32, "gate_bias"), a(q.W1q, torch.uint8, "W1q"),
        a(q.w1_scale, torch.float32, "w1_scale"), a(q.W2q, torch.uint8, "W2q"),
        a(q.w2_scale, torch.float32, "w2_scale"), a(y, torch.bfloat16, "y"),
        a(aux, torch.float32, "aux"), a(topk_idx, torch.int32, "topk_idx"),
        a(topk_w, torch.float32, "topk_w"),
        a(routed_counts, torch.int32, "routed_counts"),
        a(P, torch.float32, "P"), a(kept_counts, torch.int32, "kept_counts"),
        a(offsets, torch.int32, "offsets"), a(dest_row, torch.int32, "dest_row"),
        a(dev_status, torch.int32, "dev_status"), wp, wn, _stream(stream), ev))


# ------------------------------------------------- expert parallelism ----

def moe_ep_permute(shape, world, rank, x, topk_idx, kept_counts, offsets, dest_row, src_token,
                   x_perm, send_counts, routed_all=None, T_global=0, dev_status=None,
                   ws: Workspace | None = None, stream=None):
    """moe_permute for one rank of an expert-parallel group: with routed_all
    ([world, E] int32, every rank's routed counts) experts serve the group's
    tokens in global order against the group's capacity (T_global tokens);
    without it the rank applies its own batch's capacity. send_counts
    [world] receives the rows for each rank's experts."""
    a = _Args(shape)
    s = a.shape
    wp, wn = _ws(ws, s)
    ra = None
    if routed_all is not None:
        ra = _ptr(routed_all, torch.int32, "routed_all", int(world) * s.E)
    _check("moe_ep_permute", load_library().moe_ep_permute(
        ctypes.byref(s), int(world), int(rank), ra, int(T_global),
        a(x, torch.bfloat16, "x"), a(topk_idx, torch.int32, "topk_idx"),
        a(kept_counts, torch.int32, "kept_counts"), a(offsets, torch.int32, "offsets"),
        a(dest_row, torch.int32, "dest_row"), a(src_token, torch.int32, "src_token"),
        a(x_perm, torch.bfloat16, "x_perm"),
        _ptr(send_counts, torch.int32, "send_counts", int(world)),
        a(dev_status, torch.int32, "dev_status"), wp, wn, _stream(stream)))


def moe_ep_regroup(world, E_local, counts, src, dst, to_expert_major, local_offsets=None,
                   stream=None):
    """Rows of src [rows, H] between the source-major order of an
    expert-parallel exchange and the expert-major order of this rank's
    experts (to_expert_major=True also fills local_offsets [E_local+1]);
    counts [world, E_local] int32."""
    rows, H = (src.shape[0], src.shape[1]) if src.dim() == 2 else (0, 0)
    if dst.dim() != 2 or dst.shape[0] < rows or dst.shape[1] != H:
        raise ValueError("dst must be [rows, H] like src")
    _check("moe_ep_regroup", load_library().moe_ep_regroup(
        int(world), int(E_local), int(H), int(rows), 1 if to_expert_major else 0,
        _ptr(counts, torch.int32, "counts", int(world) * int(E_local)),
        _ptr(src, torch.bfloat16, "src", rows * H) if rows else None,
        _ptr(dst, torch.bfloat16, "dst", rows * H) if rows else None,
        _ptr(local_offsets, torch.int32, "local_offsets", int(E_local) + 1),
        _stream(stream)))


# --------------------------------------------- on-device micro-batching ----

class DevicePipeline:
    """Owns what moe_layer_fwd_pipelined needs besides the weights: two
    layer workspaces, a dispatch stream (high priority) and an expert stream,
    and four events."""

    def __init__(self, shape, device="cuda"):
        self.shape = _shape(shape)
        n = ctypes.c_size_t(0)
        _check("moe_pipelined_workspace_size", load_library().moe_pipelined_workspace_size(
            ctypes.byref(self.shape), ctypes.byref(n)))
        self.nbytes = n.value
        self.buf = torch.empty(max(self.nbytes, 256), dtype=torch.uint8, device=device)
        hi, _ = torch.cuda.Stream.priority_range()
        self.streams = [torch.cuda.Stream(device=device, priority=hi),
                        torch.cuda.Stream(device=device)]
        self.events = [torch.cuda.Event() for _ in range(4)]
        for e in self.events:          # create the handles
            e.record(self.streams[0])

    def run(self, n_micro, x, gate, gate_bias, W1, W2, y, aux=None, dev_status=None):
        """Enqueues n_micro micro-batches (x, y: [n_micro*T, H] bf16 on the
        device) after the work already queued on the current stream; returns
        the dispatch stream, whose completion means y and aux are done."""
        s = self.shape
        cur = torch.cuda.current_stream()
        for st in self.streams:
            st.wait_stream(cur)
        a = _Args(s)
        n = int(n_micro) * s.T * s.H
        st = (ctypes.c_void_p * 2)(*[q.cuda_stream for q in self.streams])
        ev = (ctypes.c_void_p * 4)(*[e.cuda_event for e in self.events])
        _check("moe_layer_fwd_pipelined", load_library().moe_layer_fwd_pipelined(
            ctypes.byref(s), int(n_micro), _ptr(x, torch.bfloat16, "x", n),
            a(gate, torch.bfloat16, "gate"), a(gate_bias, torch.float32, "gate_bias"),
            a(W1, torch.bfloat16, "W1"), a(W2, torch.bfloat16, "W2"),
            _ptr(y, torch.bfloat16, "y", n),
            _ptr(aux, torch.float32, "aux", int(n_micro)),
            a(dev_status, torch.int32, "dev_status"), self.buf.data_ptr(), self.nbytes, st, ev))
        return self.streams[0]


def moe_layer_fwd_pipelined(pipeline: DevicePipeline, n_micro, x, gate, gate_bias, W1, W2, y,
                            aux=None, dev_status=None):
    """C-ABI name for DevicePipeline.run."""
    return pipeline.run(n_micro, x, gate, gate_bias, W1, W2, y, aux, dev_status)
