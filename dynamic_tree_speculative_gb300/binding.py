"""Thin Python binding of the spec-tree C ABI (include/spec_tree.h).

Argument marshalling only: every step of the hot path runs in the CUDA
kernels of libspec_tree.so.  PyTorch supplies device memory and streams.
Importing this module without the built library raises, so a missing native
build can never fall back to anything else.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libspec_tree.so")

BF16, F32 = 0, 1
BUILDER_TOPR, BUILDER_SMART = 0, 1
PROBE_FIRST, PROBE_LAST = 0, 1
ROOT, DET, PROBE, FILL = 0, 1, 2, 3
OK, E_PARAM, E_LAYOUT, E_CUDA = 0, -1, -3, -4
S_NONFINITE_DRAFT, S_NONFINITE_TARGET, S_RESIDUAL_EMPTY = 1, 2, 4
S_OVERFLOW, S_TIMEOUT, S_ROWS, S_LAYERS = 8, 16, 32, 64
MAX_SUPPORT = 1024
SUPPORT_DENSE = 0x40000000   # |S| = V for any vocabulary
DENSE_MAX_K = 64
STATIC_MAX_TREES = 64
DEFAULT_SUPPORT = 128

EXPORTS = ("spec_tree_rows_needed", "spec_tree_check_params", "spec_tree_select_expand", "spec_tree_rank",
           "spec_tree_build", "spec_tree_verify", "spec_tree_layer_state_bytes", "spec_tree_layer_rows",
           "spec_tree_layer", "spec_tree_finish", "spec_tree_layer_static", "spec_tree_smart_fit",
           "spec_tree_wait_selftest", "spec_tree_verify_dense", "spec_tree_strerror")


class SpecTreeError(RuntimeError):
    pass


class c_params(ctypes.Structure):
    _fields_ = [("K", ctypes.c_int32), ("m", ctypes.c_int32), ("W", ctypes.c_int32), ("depth", ctypes.c_int32),
                ("R", ctypes.c_int32), ("support", ctypes.c_int32), ("temperature", ctypes.c_float),
                ("builder", ctypes.c_int32), ("lam", ctypes.c_float), ("beta", ctypes.c_float),
                ("gamma", ctypes.c_float), ("delta", ctypes.c_float), ("rho", ctypes.c_float),
                ("eta", ctypes.c_float), ("alpha", ctypes.c_float), ("verify_order", ctypes.c_int32)]


class c_tree(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "node_token", "node_parent", "node_depth", "node_kind", "node_slot", "node_exp_row", "node_score",
        "n_nodes", "sup_id", "sup_q", "sup_qT", "sup_z", "sup_zT", "probe_pos")] + [
        ("n_rows", ctypes.c_int32), ("max_nodes", ctypes.c_int32), ("sup_stride", ctypes.c_int32),
        ("sched", ctypes.c_void_p)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is not built; run `python -c \"import __graft_entry__ as g; g.build()\"`")
    lib = ctypes.CDLL(LIB_PATH)
    P, T, vp, i32, i64 = ctypes.POINTER(c_params), ctypes.POINTER(c_tree), ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    lib.spec_tree_rows_needed.argtypes = [P]
    lib.spec_tree_check_params.argtypes = [P, i32]
    lib.spec_tree_select_expand.argtypes = [P, i32, i32, i32, vp, i64, vp, T, vp, vp]
    lib.spec_tree_rank.argtypes = [P, i32, i32, T, vp, vp]
    lib.spec_tree_build.argtypes = [P, i32, i32, i32, vp, i64, vp, T, vp, vp]
    lib.spec_tree_verify.argtypes = [P, i32, i32, i32, vp, i64, T, vp, vp, vp, vp, vp, vp, vp, vp]
    lib.spec_tree_verify_dense.argtypes = [P, i32, i32, i32, vp, i64, vp, i64, T, vp, vp, vp, vp, vp, vp, vp, vp]
    lib.spec_tree_layer_state_bytes.argtypes = []
    lib.spec_tree_layer_state_bytes.restype = ctypes.c_size_t
    lib.spec_tree_layer_rows.argtypes = [P, i32]
    lib.spec_tree_layer.argtypes = [P, i32, i32, i32, i32, vp, i64, vp, T, vp, vp, vp, vp, vp]
    lib.spec_tree_finish.argtypes = [P, i32, i32, T, vp, vp, vp]
    lib.spec_tree_layer_static.argtypes = [P, i32, i32, i32, i32, vp, i64, vp, T, vp, vp, vp, vp]
    dp = ctypes.POINTER(ctypes.c_double)
    lib.spec_tree_smart_fit.argtypes = [i32, dp, dp, dp, ctypes.c_double, dp, P, dp, dp]
    lib.spec_tree_wait_selftest.argtypes = [ctypes.c_uint32, vp, vp, vp]
    lib.spec_tree_strerror.argtypes = [i32]
    lib.spec_tree_strerror.restype = ctypes.c_char_p
    for name in EXPORTS:
        if name not in ("spec_tree_strerror", "spec_tree_layer_state_bytes"):
            getattr(lib, name).restype = ctypes.c_int
    return lib


_lib = _load()


@dataclasses.dataclass
class Params:
    K: int
    m: int
    W: int
    depth: int
    R: int
    temperature: float = 1.0
    support: int = 128
    builder: int = BUILDER_TOPR
    lam: float = 0.02
    beta: float = 0.0
    gamma: float = 0.5
    delta: float = 0.01
    rho: float = 1.3
    eta: float = 0.0
    alpha: float = 1.0
    verify_order: int = PROBE_FIRST

    def c(self) -> c_params:
        return c_params(self.K, self.m, self.W, self.depth, self.R, self.support, self.temperature, self.builder,
                        self.lam, self.beta, self.gamma, self.delta, self.rho, self.eta, self.alpha,
                        self.verify_order)

    @staticmethod
    def from_workload(wl) -> "Params":
        return Params(K=wl.K, m=wl.m, W=wl.W, depth=wl.depth, R=wl.R, temperature=wl.temperature,
                      support=wl.support, builder=BUILDER_SMART if wl.builder == "smart" else BUILDER_TOPR,
                      lam=wl.lam, beta=wl.beta, gamma=wl.gamma, delta=wl.delta, rho=wl.rho, eta=wl.eta,
                      alpha=wl.alpha, verify_order=PROBE_LAST if wl.verify_order == "rrsw" else PROBE_FIRST)


def _cp(params) -> c_params:
    """Params or an already marshalled c_params (callers in a loop can marshal once)."""
    return params if isinstance(params, c_params) else params.c()


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(rc: int):
    if rc != OK:
        raise SpecTreeError(f"spec_tree error {rc}: {_lib.spec_tree_strerror(rc).decode()}")


class TreeBuffers:
    """Device buffers of a batch of trees (the spec_tree_t of the C ABI)."""

    def __init__(self, params: Params, B: int, n_rows: Optional[int] = None, device="cuda", V: Optional[int] = None):
        i32, f32 = torch.int32, torch.float32
        self.B = B
        self.n_rows = n_rows if n_rows is not None else rows_needed(params)
        self.max_nodes = params.R + 1
        # support arrays hold |S| = min(support, V) ranks per row, at least 128 wide; a dense
        # support of a vocabulary above MAX_SUPPORT tokens keeps K ranks and the probe
        if params.support == SUPPORT_DENSE:
            self.sup_stride = MAX_SUPPORT if V is None or V <= MAX_SUPPORT else max(DEFAULT_SUPPORT, params.K + 1)
        else:
            self.sup_stride = max(DEFAULT_SUPPORT, params.support or DEFAULT_SUPPORT)
        mk = lambda shape, dt: torch.empty(shape, dtype=dt, device=device)  # noqa: E731
        n = (B, self.max_nodes)
        self.node_token, self.node_parent, self.node_depth = mk(n, i32), mk(n, i32), mk(n, i32)
        self.node_kind, self.node_slot, self.node_exp_row = mk(n, i32), mk(n, i32), mk(n, i32)
        self.node_score = mk(n, f32)
        self.n_nodes = mk((B,), i32)
        r = (B, self.n_rows)
        self.sup_id = mk(r + (self.sup_stride,), i32)
        self.sup_q = mk(r + (self.sup_stride,), f32)
        self.sup_qT = mk(r + (self.sup_stride,), f32)
        self.sup_z, self.sup_zT, self.probe_pos = mk(r, f32), mk(r, f32), mk(r, i32)
        # row counter of the support selection (zero; every call leaves it zero) and the latest
        # call's cut key, a threshold hint for the next call's first rows
        self.sched = torch.zeros((3,), dtype=i32, device=device)

    def c(self) -> c_tree:
        if getattr(self, "_c", None) is None:
            t = c_tree()
            for name, _ in c_tree._fields_[:14]:
                setattr(t, name, getattr(self, name).data_ptr())
            t.n_rows, t.max_nodes, t.sup_stride = self.n_rows, self.max_nodes, self.sup_stride
            t.sched = self.sched.data_ptr()
            self._c = t
        return self._c


def _dtype_code(x: torch.Tensor) -> int:
    if x.dtype == torch.bfloat16:
        return BF16
    if x.dtype == torch.float32:
        return F32
    raise SpecTreeError(f"unsupported logits dtype {x.dtype}")


def _row_stride(x: torch.Tensor, rows_per_tree: int) -> int:
    if x.dim() != 3 or x.stride(2) != 1 or x.stride(1) != x.stride(0) // rows_per_tree or \
            x.stride(0) != rows_per_tree * x.stride(1) or x.shape[1] != rows_per_tree:
        raise SpecTreeError("logits must be [B][rows][row_stride] with contiguous rows")
    return x.stride(1)


def rows_needed(params: Params) -> int:
    return _lib.spec_tree_rows_needed(ctypes.byref(_cp(params)))


def spec_tree_check_params(params: Params, V: int) -> int:
    return _lib.spec_tree_check_params(ctypes.byref(_cp(params)), V)


def spec_tree_select_expand(params: Params, V: int, draft: torch.Tensor, u_probe: torch.Tensor, tree: TreeBuffers,
                            status: torch.Tensor, stream=None):
    _check(_lib.spec_tree_select_expand(ctypes.byref(_cp(params)), tree.B, V, _dtype_code(draft), _ptr(draft),
                                        _row_stride(draft, tree.n_rows), _ptr(u_probe), ctypes.byref(tree.c()),
                                        _ptr(status), _stream(stream)))


def spec_tree_rank(params: Params, V: int, tree: TreeBuffers, status: torch.Tensor, stream=None):
    _check(_lib.spec_tree_rank(ctypes.byref(_cp(params)), tree.B, V, ctypes.byref(tree.c()), _ptr(status),
                               _stream(stream)))


def spec_tree_build(params: Params, V: int, draft: torch.Tensor, u_probe: torch.Tensor, tree: TreeBuffers,
                    status: torch.Tensor, stream=None):
    _check(_lib.spec_tree_build(ctypes.byref(_cp(params)), tree.B, V, _dtype_code(draft), _ptr(draft),
                                _row_stride(draft, tree.n_rows), _ptr(u_probe), ctypes.byref(tree.c()),
                                _ptr(status), _stream(stream)))


def spec_tree_verify(params: Params, V: int, target: torch.Tensor, tree: TreeBuffers, u_verify: torch.Tensor,
                     u_bonus: torch.Tensor, accept_len: torch.Tensor, out_tok: torch.Tensor,
                     out_node: torch.Tensor, margins: Optional[torch.Tensor], status: torch.Tensor, stream=None):
    _check(_lib.spec_tree_verify(ctypes.byref(_cp(params)), tree.B, V, _dtype_code(target), _ptr(target),
                                 _row_stride(target, tree.max_nodes), ctypes.byref(tree.c()), _ptr(u_verify),
                                 _ptr(u_bonus), _ptr(accept_len), _ptr(out_tok), _ptr(out_node), _ptr(margins),
                                 _ptr(status), _stream(stream)))


def spec_tree_verify_dense(params: Params, V: int, target: torch.Tensor, draft: torch.Tensor, tree: TreeBuffers,
                           u_verify: torch.Tensor, u_bonus: torch.Tensor, accept_len: torch.Tensor,
                           out_tok: torch.Tensor, out_node: torch.Tensor, margins: Optional[torch.Tensor],
                           status: torch.Tensor, stream=None):
    """spec_tree_verify for trees built on the dense support of a vocabulary above MAX_SUPPORT tokens: it
    reads the node's draft row (the tensor the tree was built from) for the tail law."""
    _check(_lib.spec_tree_verify_dense(ctypes.byref(_cp(params)), tree.B, V, _dtype_code(target), _ptr(target),
                                       _row_stride(target, tree.max_nodes), _ptr(draft),
                                       _row_stride(draft, tree.n_rows), ctypes.byref(tree.c()), _ptr(u_verify),
                                       _ptr(u_bonus), _ptr(accept_len), _ptr(out_tok), _ptr(out_node),
                                       _ptr(margins), _ptr(status), _stream(stream)))


def is_dense(params: Params, V: int) -> bool:
    """The dense support of a vocabulary too large for the support arrays (verify with spec_tree_verify_dense)."""
    return params.support == SUPPORT_DENSE and V > MAX_SUPPORT


def spec_tree_layer_state_bytes() -> int:
    return _lib.spec_tree_layer_state_bytes()


def spec_tree_layer_rows(params: Params, layer: int) -> int:
    return _lib.spec_tree_layer_rows(ctypes.byref(_cp(params)), layer)


class LayerState:
    """Caller-owned per-tree state of the layer-by-layer builder, and the frontier it names."""

    def __init__(self, params: Params, B: int, device="cuda"):
        self.B = B
        self.state = torch.empty((B, spec_tree_layer_state_bytes()), dtype=torch.uint8, device=device)
        self.frontier_token = torch.empty((B, params.W), dtype=torch.int32, device=device)
        self.frontier_parent = torch.empty((B, params.W), dtype=torch.int32, device=device)


def spec_tree_layer(params: Params, V: int, layer: int, layer_draft: torch.Tensor, u_probe: torch.Tensor,
                    tree: TreeBuffers, state: LayerState, status: torch.Tensor, stream=None):
    rows = spec_tree_layer_rows(params, layer)
    _check(_lib.spec_tree_layer(ctypes.byref(_cp(params)), tree.B, V, layer, _dtype_code(layer_draft),
                                _ptr(layer_draft), _row_stride(layer_draft, rows), _ptr(u_probe),
                                ctypes.byref(tree.c()), _ptr(state.state), _ptr(state.frontier_token),
                                _ptr(state.frontier_parent), _ptr(status), _stream(stream)))


def spec_tree_finish(params: Params, V: int, tree: TreeBuffers, state: LayerState, status: torch.Tensor,
                     stream=None):
    _check(_lib.spec_tree_finish(ctypes.byref(_cp(params)), tree.B, V, ctypes.byref(tree.c()), _ptr(state.state),
                                 _ptr(status), _stream(stream)))


def spec_tree_layer_static(params: Params, V: int, layer: int, layer_draft: torch.Tensor, u_probe: torch.Tensor,
                           tree: TreeBuffers, frontier_token: Optional[torch.Tensor],
                           frontier_parent: Optional[torch.Tensor], status: torch.Tensor, stream=None):
    """spec_tree_layer with the builder's state inside the library (no state buffer to allocate); the
    last layer's call also writes the node arrays.  At most STATIC_MAX_TREES trees; builds must not
    overlap on the GPU."""
    rows = spec_tree_layer_rows(params, layer)
    _check(_lib.spec_tree_layer_static(ctypes.byref(_cp(params)), tree.B, V, layer, _dtype_code(layer_draft),
                                       _ptr(layer_draft), _row_stride(layer_draft, rows), _ptr(u_probe),
                                       ctypes.byref(tree.c()), _ptr(frontier_token), _ptr(frontier_parent),
                                       _ptr(status), _stream(stream)))


@dataclasses.dataclass
class CostFit:
    lam: float
    gamma: float
    delta: float
    rho: float
    rms_draft: float
    rms_verify: float

    def apply(self, params: Params) -> Params:
        """params with the fitted SMART cost coefficients (beta = eta = 0)."""
        return dataclasses.replace(params, lam=self.lam, beta=0.0, gamma=self.gamma, delta=self.delta,
                                   rho=self.rho, eta=0.0)


def spec_tree_smart_fit(sizes, t_draft, t_verify, t_base: float, weights=None) -> CostFit:
    """Fit the SMART cost model to profiled step times (host only, no GPU)."""
    def arr(x):
        a = (ctypes.c_double * len(x))(*[float(v) for v in x])
        return ctypes.cast(a, ctypes.POINTER(ctypes.c_double)), a

    n = len(sizes)
    if len(t_draft) != n or len(t_verify) != n or (weights is not None and len(weights) != n):
        raise SpecTreeError("sizes, timings and weights must have the same length")
    (pn, _an), (pd, _ad), (pv, _av) = arr(sizes), arr(t_draft), arr(t_verify)
    pw, _aw = arr(weights) if weights is not None else (None, None)
    coef = (ctypes.c_double * 4)()
    rms = (ctypes.c_double * 2)()
    _check(_lib.spec_tree_smart_fit(n, pn, pd, pv, float(t_base), pw, None,
                                    ctypes.cast(coef, ctypes.POINTER(ctypes.c_double)),
                                    ctypes.cast(rms, ctypes.POINTER(ctypes.c_double))))
    return CostFit(lam=coef[0], gamma=coef[1], delta=coef[2], rho=coef[3], rms_draft=rms[0], rms_verify=rms[1])


class VerifyOutputs:
    def __init__(self, params: Params, B: int, device="cuda"):
        self.accept_len = torch.empty((B,), dtype=torch.int32, device=device)
        self.out_tok = torch.empty((B, params.depth + 1), dtype=torch.int32, device=device)
        self.out_node = torch.empty((B, params.depth + 1), dtype=torch.int32, device=device)
        self.margins = torch.zeros((2,), dtype=torch.int32, device=device)


def spec_tree_wait_selftest(polls: int, status: torch.Tensor, result: torch.Tensor, stream=None):
    """Let one CTA-scope and one cluster-scope bounded wait run out (`polls` polls each) on a barrier
    nothing arrives on; result (4 x int32 on the device) = gave up / polls made, per CTA."""
    _check(_lib.spec_tree_wait_selftest(polls, _ptr(status), _ptr(result), _stream(stream)))
