"""spec_tree_layer_static: the layer-by-layer builder for callers that cannot allocate.

Some callers cannot allocate device memory: a draft loop running inside a host
runtime that reserved all device memory up front and hands its plugins no
allocator, or a decode loop that must not call cudaMalloc/cudaFree because they
can synchronise the device mid-step.  For them spec_tree_layer_static keeps the
builder's per-tree state in a fixed array inside the library instead of a
caller buffer.  This test checks, through the C ABI, that it builds the same
trees as spec_tree_layer + spec_tree_finish with a caller-owned state: node
arrays and score bits, every expanded support row and every frontier, bit for
bit (the tolerance of the other layer-mode tests), on two builds in a row, so
that the second one runs over what the first left in the shared array.  It also
checks that a batch above the array's limit is refused before any launch, that
a whole build changes the device's free memory by nothing (after a first build
has loaded the library's module and its array), that a one-layer build (whose
only call is also the last) matches too, and that an empty batch on the last
layer is accepted.

The file is named to be collected last, so that a failure here comes after
every other test has run.
"""
import numpy as np
import pytest
import torch

from dynamic_tree_speculative_gb300 import binding as B
from dynamic_tree_speculative_gb300 import workloads as WL

pytestmark = pytest.mark.gpu

import parity  # noqa: E402  (loads the native library; fails loudly if absent)

NODE_FIELDS = ("node_token", "node_parent", "node_depth", "node_kind", "node_slot", "node_exp_row", "n_nodes")
SUP_FIELDS = ("sup_id", "sup_q", "sup_qT", "sup_z", "sup_zT", "probe_pos")


def _row0(wl, layer):
    return 0 if layer == 0 else 1 + (layer - 1) * wl.W


def _tree(params, wl):
    tree = B.TreeBuffers(params, wl.B)
    # rows no call expands keep these values in both trees
    tree.sup_id.fill_(-5)
    tree.probe_pos.fill_(-2)
    for t in (tree.sup_q, tree.sup_qT, tree.sup_z, tree.sup_zT):
        t.fill_(float("nan"))
    tree.node_score.fill_(float("nan"))
    return tree


def _build(case, static):
    """One layer-by-layer build; returns the tree (host arrays) and each call's frontier."""
    wl = case.wl
    params = B.Params.from_workload(wl)
    tree = _tree(params, wl)
    state = None if static else B.LayerState(params, wl.B)  # the existing entry points' caller-owned state
    ftok = torch.full((wl.B, wl.W), -7, dtype=torch.int32, device="cuda")
    fpar = torch.full((wl.B, wl.W), -7, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    draft, u = case.draft.cuda(), case.u_probe.cuda()
    fronts = []
    for layer in range(wl.depth):
        rows, r0 = B.spec_tree_layer_rows(params, layer), _row0(wl, layer)
        d, uu = draft[:, r0:r0 + rows].contiguous(), u[:, r0:r0 + rows].contiguous()
        if static:
            B.spec_tree_layer_static(params, wl.V, layer, d, uu, tree, ftok, fpar, status)
            fronts.append((ftok.cpu().numpy().copy(), fpar.cpu().numpy().copy()))
        else:
            B.spec_tree_layer(params, wl.V, layer, d, uu, tree, state, status)
            fronts.append((state.frontier_token.cpu().numpy().copy(), state.frontier_parent.cpu().numpy().copy()))
    if not static:
        B.spec_tree_finish(params, wl.V, tree, state, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, int(status.item())
    host = {k: getattr(tree, k).cpu().numpy() for k in NODE_FIELDS + SUP_FIELDS + ("node_score",)}
    return params, host, fronts


def _same(wl, params, a, b):
    for f in NODE_FIELDS:
        assert np.array_equal(a[f], b[f]), f
    assert np.array_equal(a["node_score"].view(np.int32), b["node_score"].view(np.int32))
    rows = [r for layer in range(wl.depth)
            for r in range(_row0(wl, layer), _row0(wl, layer) + B.spec_tree_layer_rows(params, layer))]
    S = min(wl.support, wl.V)
    for f in SUP_FIELDS:
        x, y = a[f][:, rows], b[f][:, rows]
        if f in ("sup_id", "sup_q", "sup_qT"):
            x, y = x[..., :S], y[..., :S]
        assert np.array_equal(x.view(np.int32), y.view(np.int32)), f


def test_static_state_equals_caller_state_twice_in_a_row():
    # first build: the full limit of trees at the Vicuna-like vocabulary; second build:
    # fewer, deeper trees on other logits, over what the first build left in the array
    builds = [WL.WORKLOADS["vicuna"].with_(B=B.STATIC_MAX_TREES, V=6000, depth=4, R=24),
              WL.WORKLOADS["vicuna"].with_(B=8, V=32000, depth=8, R=60)]
    for i, wl in enumerate(builds):
        case = parity.make_case(wl, 40 + i)
        params, ref, ref_fronts = _build(case, static=False)
        _, got, got_fronts = _build(case, static=True)
        _same(wl, params, got, ref)
        for layer in range(wl.depth):
            assert np.array_equal(got_fronts[layer][0], ref_fronts[layer][0]), (i, layer)
            assert np.array_equal(got_fronts[layer][1], ref_fronts[layer][1]), (i, layer)
        assert (got["n_nodes"] > 1).all()


def test_static_state_refuses_too_many_trees():
    wl = WL.WORKLOADS["vicuna"].with_(B=B.STATIC_MAX_TREES + 1, V=3000, depth=2, R=8)
    params = B.Params.from_workload(wl)
    tree = B.TreeBuffers(params, wl.B)
    d = torch.zeros((wl.B, 1, wl.V), dtype=torch.bfloat16, device="cuda")
    u = torch.zeros((wl.B, 1), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(B.SpecTreeError, match="error -1"):
        B.spec_tree_layer_static(params, wl.V, 0, d, u, tree, None, None, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0


def test_static_build_allocates_nothing():
    """A whole static build leaves the device's free memory unchanged (every input, output and
    frontier buffer allocated beforehand; a first build has loaded the module and its array)."""
    wl = WL.WORKLOADS["vicuna"].with_(B=16, V=8000, depth=4, R=24)
    case = parity.make_case(wl, 44)
    params = B.Params.from_workload(wl)
    tree = _tree(params, wl)
    ftok = torch.full((wl.B, wl.W), -7, dtype=torch.int32, device="cuda")
    fpar = torch.full((wl.B, wl.W), -7, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    draft, u = case.draft.cuda(), case.u_probe.cuda()
    layers = []
    for layer in range(wl.depth):
        rows, r0 = B.spec_tree_layer_rows(params, layer), _row0(wl, layer)
        layers.append((layer, draft[:, r0:r0 + rows].contiguous(), u[:, r0:r0 + rows].contiguous()))

    def build():
        for layer, d, uu in layers:
            B.spec_tree_layer_static(params, wl.V, layer, d, uu, tree, ftok, fpar, status)

    build()
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    build()
    torch.cuda.synchronize()
    free1 = torch.cuda.mem_get_info()[0]
    assert free1 == free0, (free0, free1)
    assert int(status.item()) == 0 and (tree.n_nodes.cpu() > 1).all()


def test_static_one_layer_build():
    """depth 1: the first call is also the last, so it expands the root and cuts the tree."""
    wl = WL.WORKLOADS["vicuna"].with_(B=8, V=6000, depth=1, R=8)
    case = parity.make_case(wl, 45)
    params, ref, ref_fronts = _build(case, static=False)
    _, got, got_fronts = _build(case, static=True)
    _same(wl, params, got, ref)
    assert (got["n_nodes"] == wl.R + 1).all()


def test_static_empty_batch_on_the_last_layer():
    """B = 0 on the last layer: only the argument checks run, and they pass."""
    import ctypes
    wl = WL.WORKLOADS["vicuna"].with_(B=4, V=6000, depth=3, R=12)
    params = B.Params.from_workload(wl)
    tree = B.TreeBuffers(params, wl.B)
    d = torch.zeros((wl.B, wl.W, wl.V), dtype=torch.bfloat16, device="cuda")
    u = torch.zeros((wl.B, wl.W), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = B._lib.spec_tree_layer_static(ctypes.byref(params.c()), 0, wl.V, wl.depth - 1, B.BF16,
                                       ctypes.c_void_p(d.data_ptr()), wl.V, ctypes.c_void_p(u.data_ptr()),
                                       ctypes.byref(tree.c()), None, None, ctypes.c_void_p(status.data_ptr()), None)
    torch.cuda.synchronize()
    assert rc == B.OK and int(status.item()) == 0
