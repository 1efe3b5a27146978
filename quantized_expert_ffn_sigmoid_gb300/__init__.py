"""Python binding of libcolimoe (the routed-MoE layer on sm_103a).

Argument marshalling only: every step of the layer runs in the library's
CUDA kernels.  Functions carry the names of the C entry points declared in
``include/coli_moe.h``; tensors are torch CUDA tensors (device memory and
streams come from torch), and calls are enqueued on the current torch stream
unless ``stream`` is given.  There is no CPU fallback: importing this module
raises if the compiled library is missing.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libcolimoe.so")

COLI_OK = 0
COLI_EINVAL = -1
COLI_EALIGN = -2
COLI_EWORKSPACE = -3
COLI_ECUDA = -4
COLI_EUNSUPPORTED = -5
STATUS_NONFINITE = 1
STATUS_BADIDX = 2
STATUS_TIMEOUT = 4

EXPORTS = (
    "coli_moe_workspace_size", "coli_moe_workspace_init", "coli_moe_route",
    "coli_moe_quantize_act", "coli_moe_forward", "coli_moe_dispatch", "coli_moe_experts",
    "coli_moe_status", "coli_moe_strerror", "coli_moe_workspace_layout",
    "coli_moe_forward_dump", "coli_moe_forward_static", "coli_moe_layer",
    "coli_moe_stack_forward",
)
STATIC_WS_BYTES = 24 << 20


class Cfg(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("n_experts", ctypes.c_int32),
                ("n_groups", ctypes.c_int32), ("topk_group", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("inter", ctypes.c_int32),
                ("n_shared", ctypes.c_int32), ("shared_inter", ctypes.c_int32),
                ("weight_bits", ctypes.c_int32), ("routed_scaling_factor", ctypes.c_float),
                ("group_size", ctypes.c_int32), ("ep_rank", ctypes.c_int32), ("ep_size", ctypes.c_int32)]
    _OPTIONAL = ("group_size", "ep_rank", "ep_size")

    @classmethod
    def of(cls, shape, ep_rank: int = 0, ep_size: int = 0) -> "Cfg":
        """From any object with the same field names (e.g. synth.LayerShape);
        a missing group_size means per-row scales.  ``ep_rank`` / ``ep_size``
        select one shard of an expert-parallel layer (0 / 0: the whole layer)."""
        vals = {"ep_rank": ep_rank, "ep_size": ep_size}
        return cls(*(vals[f] if f in vals else getattr(shape, f, 0) if f in cls._OPTIONAL else getattr(shape, f)
                     for f, _ in cls._fields_))


class Weights(ctypes.Structure):
    _fields_ = [("experts", ctypes.c_void_p), ("expert_scales", ctypes.c_void_p),
                ("shared", ctypes.c_void_p), ("shared_scales", ctypes.c_void_p)]


class StackLayer(ctypes.Structure):
    _fields_ = [("cfg", Cfg), ("weights", Weights), ("router_w", ctypes.c_void_p), ("corr_bias", ctypes.c_void_p)]


class WsLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in (
        "status", "n_entries", "entry_expert", "entry_count", "entry_offset", "pair_token",
        "pair_slot_of", "qx", "dx", "qh", "dh", "o", "total")]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                          "(there is no CPU fallback)")
    lib = ctypes.CDLL(LIB_PATH)
    P, S, I32, U32P = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32, ctypes.POINTER(ctypes.c_uint32)
    CP, WP = ctypes.POINTER(Cfg), ctypes.POINTER(Weights)
    sig = {
        "coli_moe_workspace_size": ([CP, I32], ctypes.c_size_t),
        "coli_moe_workspace_init": ([P, S, P], ctypes.c_int),
        "coli_moe_route": ([CP, P, I32, P, P, P, P, P, S, P], ctypes.c_int),
        "coli_moe_quantize_act": ([P, I32, I32, P, P, P], ctypes.c_int),
        "coli_moe_forward": ([CP, WP, P, I32, P, P, P, P, S, P], ctypes.c_int),
        "coli_moe_dispatch": ([CP, P, I32, P, P, S, P], ctypes.c_int),
        "coli_moe_experts": ([CP, WP, I32, P, P, P, S, P], ctypes.c_int),
        "coli_moe_status": ([P, P, U32P], ctypes.c_int),
        "coli_moe_strerror": ([ctypes.c_int], ctypes.c_char_p),
        "coli_moe_workspace_layout": ([CP, I32, ctypes.POINTER(WsLayout)], ctypes.c_int),
        "coli_moe_forward_dump": ([CP, WP, P, I32, P, P, P, P, S, P, P, P], ctypes.c_int),
        "coli_moe_forward_static": ([CP, WP, P, I32, P, P, P, P], ctypes.c_int),
        "coli_moe_layer": ([CP, WP, P, I32, P, P, P, P, P, P, S, P], ctypes.c_int),
        "coli_moe_stack_forward": ([ctypes.POINTER(StackLayer), I32, I32, P, P, I32, P, P, P, P, S, P],
                                   ctypes.c_int),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    return lib


lib = _load()


class ColiError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {lib.coli_moe_strerror(code).decode()} ({code})")
        self.code = code


def _check(rc: int, where: str):
    if rc != COLI_OK:
        raise ColiError(rc, where)


def _ptr(t):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _cfg(cfg) -> Cfg:
    return cfg if isinstance(cfg, Cfg) else Cfg.of(cfg)


def make_weights(experts, expert_scales, shared=None, shared_scales=None) -> Weights:
    """A weights struct from torch tensors (keep the tensors alive)."""
    return Weights(experts.data_ptr(), expert_scales.data_ptr(),
                   shared.data_ptr() if shared is not None else None,
                   shared_scales.data_ptr() if shared_scales is not None else None)


# ----------------------------------------------------------------- entry points
def coli_moe_workspace_size(cfg, max_T: int) -> int:
    return int(lib.coli_moe_workspace_size(ctypes.byref(_cfg(cfg)), int(max_T)))


def coli_moe_workspace_init(ws, stream=None):
    _check(lib.coli_moe_workspace_init(_ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "coli_moe_workspace_init")


def new_workspace(cfg, max_T: int, device="cuda"):
    """Allocate (with torch) and initialise a workspace for up to max_T positions."""
    import torch
    n = coli_moe_workspace_size(cfg, max_T)
    if n == 0:
        raise ColiError(COLI_EINVAL, "coli_moe_workspace_size")
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    coli_moe_workspace_init(ws)
    return ws


def coli_moe_route(cfg, x, router_w, corr_bias, topk_idx, topk_w, ws, stream=None):
    T = x.shape[0]
    _check(lib.coli_moe_route(ctypes.byref(_cfg(cfg)), _ptr(x), T, _ptr(router_w), _ptr(corr_bias),
                              _ptr(topk_idx), _ptr(topk_w), _ptr(ws), ws.numel(), _stream(stream)),
           "coli_moe_route")


def coli_moe_quantize_act(x, q, d, stream=None):
    T, K = x.shape
    _check(lib.coli_moe_quantize_act(_ptr(x), T, K, _ptr(q), _ptr(d), _stream(stream)),
           "coli_moe_quantize_act")


def coli_moe_forward(cfg, weights: Weights, x, topk_idx, topk_w, y, ws, stream=None):
    _check(lib.coli_moe_forward(ctypes.byref(_cfg(cfg)), ctypes.byref(weights), _ptr(x), x.shape[0],
                                _ptr(topk_idx), _ptr(topk_w), _ptr(y), _ptr(ws), ws.numel(),
                                _stream(stream)), "coli_moe_forward")


def coli_moe_layer(cfg, weights: Weights, x, router_w, corr_bias, topk_idx, topk_w, y, ws, stream=None):
    _check(lib.coli_moe_layer(ctypes.byref(_cfg(cfg)), ctypes.byref(weights), _ptr(x), x.shape[0],
                              _ptr(router_w), _ptr(corr_bias), _ptr(topk_idx), _ptr(topk_w), _ptr(y),
                              _ptr(ws), ws.numel(), _stream(stream)), "coli_moe_layer")


def coli_moe_dispatch(cfg, x, topk_idx, ws, stream=None):
    _check(lib.coli_moe_dispatch(ctypes.byref(_cfg(cfg)), _ptr(x), x.shape[0], _ptr(topk_idx),
                                 _ptr(ws), ws.numel(), _stream(stream)), "coli_moe_dispatch")


def coli_moe_experts(cfg, weights: Weights, T: int, topk_w, y, ws, stream=None):
    _check(lib.coli_moe_experts(ctypes.byref(_cfg(cfg)), ctypes.byref(weights), int(T), _ptr(topk_w),
                                _ptr(y), _ptr(ws), ws.numel(), _stream(stream)), "coli_moe_experts")


def coli_moe_forward_dump(cfg, weights: Weights, x, topk_idx, topk_w, y, ws, acc_gu=None, acc_d=None,
                          stream=None):
    _check(lib.coli_moe_forward_dump(ctypes.byref(_cfg(cfg)), ctypes.byref(weights), _ptr(x), x.shape[0],
                                     _ptr(topk_idx), _ptr(topk_w), _ptr(y), _ptr(ws), ws.numel(),
                                     _ptr(acc_gu), _ptr(acc_d), _stream(stream)), "coli_moe_forward_dump")


def coli_moe_status(ws, stream=None) -> int:
    v = ctypes.c_uint32(0)
    _check(lib.coli_moe_status(_ptr(ws), _stream(stream), ctypes.byref(v)), "coli_moe_status")
    return int(v.value)


def coli_moe_strerror(code: int) -> str:
    return lib.coli_moe_strerror(int(code)).decode()


def coli_moe_workspace_layout(cfg, T: int) -> WsLayout:
    out = WsLayout()
    _check(lib.coli_moe_workspace_layout(ctypes.byref(_cfg(cfg)), int(T), ctypes.byref(out)),
           "coli_moe_workspace_layout")
    return out


def coli_moe_forward_static(cfg, weights: Weights, x, topk_idx, topk_w, y, stream=None):
    """coli_moe_forward without a caller workspace: the library's static
    24 MiB device scratch is used instead (for callers that cannot allocate;
    calls must not overlap on the GPU)."""
    _check(lib.coli_moe_forward_static(ctypes.byref(_cfg(cfg)), ctypes.byref(weights), _ptr(x), x.shape[0],
                                       _ptr(topk_idx), _ptr(topk_w), _ptr(y), _stream(stream)),
           "coli_moe_forward_static")


def stack_layers(layers):
    """A ctypes array of StackLayer from (cfg, weights, router_w, corr_bias)
    tuples (keep the tensors alive)."""
    arr = (StackLayer * len(layers))()
    for i, (cfg, w, wr, b) in enumerate(layers):
        arr[i] = StackLayer(_cfg(cfg), w, wr.data_ptr(), b.data_ptr())
    return arr


def coli_moe_stack_forward(layers, xs, residual, topk_idx, topk_w, y, ws, add_output=False, stream=None):
    """One step through a stack of layers (``layers`` from stack_layers):
    xs [L+1, T, H] (xs[0] read, the rest written), residual [L, T, H] or
    None, topk_idx / topk_w [L, T, k] and y [L, T, H] written."""
    n, T = len(layers), xs.shape[1]
    _check(lib.coli_moe_stack_forward(layers, n, T, _ptr(xs), _ptr(residual), int(bool(add_output)),
                                      _ptr(topk_idx), _ptr(topk_w), _ptr(y), _ptr(ws), ws.numel(),
                                      _stream(stream)), "coli_moe_stack_forward")


def capture_stack_step(layers, xs, residual, topk_idx, topk_w, y, ws, add_output=False):
    """The stack step captured once as a CUDA graph (torch.cuda.CUDAGraph);
    ``graph.replay()`` runs it again on the same buffers.  Runs the step once
    first, outside capture (the first call of some kernels sets attributes)."""
    import torch
    coli_moe_stack_forward(layers, xs, residual, topk_idx, topk_w, y, ws, add_output)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="thread_local"):
        coli_moe_stack_forward(layers, xs, residual, topk_idx, topk_w, y, ws, add_output)
    return g
