"""C-ABI library: loads, exports every declared symbol, host-side checks (no GPU needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def binding():
    from dynamic_tree_speculative_gb300 import binding as B
    return B


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "spec_tree.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(spec_tree_\w+)\s*\(", src, flags=re.M)))


def test_every_declared_symbol_is_exported(binding):
    names = _declared_functions()
    assert len(names) >= 7
    lib = ctypes.CDLL(binding.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert set(binding.EXPORTS) <= set(names)


def test_rows_needed(binding):
    P = binding.Params
    assert binding.rows_needed(P(K=8, m=1, W=8, depth=8, R=60)) == 57
    assert binding.rows_needed(P(K=6, m=1, W=6, depth=6, R=32)) == 31
    assert binding.rows_needed(P(K=8, m=1, W=8, depth=8, R=60, builder=binding.BUILDER_SMART)) == 61


@pytest.mark.parametrize("kw,V,ok", [
    (dict(K=8, m=1, W=8, depth=8, R=60), 128256, True),
    (dict(K=8, m=8, W=8, depth=8, R=60), 128256, True),     # m = K: one-hot Top-K tree
    (dict(K=8, m=9, W=8, depth=8, R=60), 128256, False),    # m > K
    (dict(K=8, m=1, W=8, depth=8, R=60, verify_order=1), 128256, True),   # probe last
    (dict(K=8, m=1, W=8, depth=8, R=60, verify_order=2), 128256, False),  # unknown order
    (dict(K=8, m=1, W=8, depth=8, R=60), 5, False),         # K > |S| = V
    (dict(K=4, m=1, W=4, depth=3, R=8), 32, True),
    (dict(K=8, m=1, W=8, depth=0, R=60), 1000, False),      # depth < 1
    (dict(K=8, m=1, W=8, depth=8, R=0), 1000, False),       # R < 1
    (dict(K=8, m=1, W=8, depth=8, R=60, temperature=0.0), 1000, False),
    (dict(K=8, m=1, W=8, depth=8, R=60, support=129), 1000, True),    # wide supports: 129 .. 1024
    (dict(K=8, m=1, W=8, depth=8, R=60, support=1024), 128256, True),
    (dict(K=8, m=1, W=8, depth=8, R=60, support=1025), 128256, False),
    (dict(K=128, m=1, W=1, depth=2, R=8, support=0), 128256, True),   # support 0 means 128 ...
    (dict(K=129, m=1, W=1, depth=2, R=8, support=0), 128256, False),  # ... so K = 129 > |S|
    (dict(K=100, m=1, W=1, depth=2, R=8, support=0), 100, True),      # |S| = min(128, V)
    (dict(K=16, m=1, W=16, depth=9, R=60), 1000, False),    # candidates > 2048
    (dict(K=8, m=1, W=8, depth=8, R=600), 1000, False),     # R + 1 > 512
    (dict(K=2, m=0, W=1, depth=1, R=1), 2, True),
])
def test_param_checks(binding, kw, V, ok):
    rc = binding.spec_tree_check_params(binding.Params(**kw), V)
    assert (rc == binding.OK) == ok


def test_bad_arguments_fail_before_any_launch(binding):
    """Host checks return codes without touching CUDA (works with no GPU)."""
    lib = binding._lib
    p = binding.Params(K=8, m=1, W=8, depth=8, R=60).c()
    t = binding.c_tree()
    # null tree
    assert lib.spec_tree_build(ctypes.byref(p), 1, 1000, binding.BF16, ctypes.c_void_p(16), 1000,
                               ctypes.c_void_p(16), None, None, None) == binding.E_PARAM
    # misaligned rows: row_stride * 2 bytes not a multiple of 16
    for name, _ in binding.c_tree._fields_[:14]:
        setattr(t, name, 256)
    t.n_rows, t.max_nodes, t.sup_stride = 57, 61, 128
    assert lib.spec_tree_select_expand(ctypes.byref(p), 1, 1001, binding.BF16, ctypes.c_void_p(256), 1001,
                                       ctypes.c_void_p(256), ctypes.byref(t), None, None) == binding.E_LAYOUT
    # unaligned base pointer
    assert lib.spec_tree_select_expand(ctypes.byref(p), 1, 1000, binding.BF16, ctypes.c_void_p(258), 1008,
                                       ctypes.c_void_p(256), ctypes.byref(t), None, None) == binding.E_LAYOUT
    # unknown dtype
    assert lib.spec_tree_select_expand(ctypes.byref(p), 1, 1000, 7, ctypes.c_void_p(256), 1008,
                                       ctypes.c_void_p(256), ctypes.byref(t), None, None) == binding.E_LAYOUT
    # too few rows per tree
    t.n_rows = 56
    assert lib.spec_tree_select_expand(ctypes.byref(p), 1, 1000, binding.BF16, ctypes.c_void_p(256), 1008,
                                       ctypes.c_void_p(256), ctypes.byref(t), None, None) == binding.E_PARAM
    # verify: null outputs
    t.n_rows = 57
    assert lib.spec_tree_verify(ctypes.byref(p), 1, 1000, binding.BF16, ctypes.c_void_p(256), 1008,
                                ctypes.byref(t), ctypes.c_void_p(256), ctypes.c_void_p(256), None, None, None,
                                None, None, None) == binding.E_PARAM
    assert binding._lib.spec_tree_strerror(binding.E_LAYOUT).startswith(b"unsupported")
    # the bounded-wait self-test: null pointers and poll counts out of range
    assert lib.spec_tree_wait_selftest(64, None, ctypes.c_void_p(256), None) == binding.E_PARAM
    assert lib.spec_tree_wait_selftest(0, ctypes.c_void_p(256), ctypes.c_void_p(256), None) == binding.E_PARAM
    assert lib.spec_tree_wait_selftest(65537, ctypes.c_void_p(256), ctypes.c_void_p(256), None) == binding.E_PARAM


def test_layer_rows_and_state(binding):
    P = binding.Params
    p = P(K=2, m=1, W=8, depth=5, R=24)
    assert [binding.spec_tree_layer_rows(p, layer) for layer in range(-1, 6)] == [0, 1, 2, 4, 8, 8, 0]
    assert [binding.spec_tree_layer_rows(P(K=8, m=1, W=8, depth=8, R=60), layer) for layer in range(8)] == \
        [1] + [8] * 7
    # the rows of all calls are the one-shot build's rows
    for kw in (dict(K=2, m=1, W=8, depth=5, R=24), dict(K=6, m=1, W=6, depth=6, R=32)):
        q = P(**kw)
        assert sum(binding.spec_tree_layer_rows(q, layer) for layer in range(q.depth)) <= binding.rows_needed(q)
    assert binding.spec_tree_layer_rows(P(K=8, m=1, W=8, depth=8, R=60, builder=binding.BUILDER_SMART), 0) == 0
    n = binding.spec_tree_layer_state_bytes()
    assert n > 0 and n % 16 == 0
    # the allocation-free entry point reserves 56 KiB of its array per tree for this state
    assert n <= 56 * 1024


def test_layer_mode_bad_arguments(binding):
    lib = binding._lib
    t = binding.c_tree()
    for name, _ in binding.c_tree._fields_[:14]:
        setattr(t, name, 256)
    t.n_rows, t.max_nodes, t.sup_stride = 57, 61, 128
    vp = ctypes.c_void_p

    def layer(p, layer_idx, state):
        return lib.spec_tree_layer(ctypes.byref(p.c()), 1, 1000, layer_idx, binding.BF16, vp(256), 1008, vp(256),
                                   ctypes.byref(t), state, None, None, None, None)

    p = binding.Params(K=8, m=1, W=8, depth=8, R=60)
    assert layer(p, 8, vp(256)) == binding.E_PARAM                       # past the last layer
    assert layer(p, -1, vp(256)) == binding.E_PARAM
    assert layer(p, 0, None) == binding.E_PARAM                          # no state
    assert layer(p, 0, vp(264)) == binding.E_LAYOUT                      # state not 16-byte aligned
    smart = binding.Params(K=8, m=1, W=8, depth=8, R=60, builder=binding.BUILDER_SMART)
    t.n_rows = 61
    assert layer(smart, 0, vp(256)) == binding.E_PARAM                   # top-R builder only
    t.n_rows = 57
    assert lib.spec_tree_finish(ctypes.byref(p.c()), 1, 1000, ctypes.byref(t), None, None, None) == \
        binding.E_PARAM
    assert lib.spec_tree_finish(ctypes.byref(p.c()), 1, 1000, ctypes.byref(t), vp(264), None, None) == \
        binding.E_LAYOUT


def test_layer_static_host_checks(binding):
    """The allocation-free layer call refuses batches above its array and checks arguments before any
    CUDA call (B = 0 runs the checks alone)."""
    lib = binding._lib
    t = binding.c_tree()
    for name, _ in binding.c_tree._fields_[:14]:
        setattr(t, name, 256)
    t.n_rows, t.max_nodes, t.sup_stride = 57, 61, 128
    vp = ctypes.c_void_p
    p = binding.Params(K=8, m=1, W=8, depth=8, R=60)

    def call(B, layer, tree=t, params=p):
        return lib.spec_tree_layer_static(ctypes.byref(params.c()), B, 1000, layer, binding.BF16, vp(256), 1008,
                                          vp(256), ctypes.byref(tree), None, None, None, None)

    assert call(binding.STATIC_MAX_TREES + 1, 0) == binding.E_PARAM
    assert call(-1, 0) == binding.E_PARAM
    assert call(0, 0) == binding.OK and call(0, 7) == binding.OK
    assert call(0, 8) == binding.E_PARAM                                  # past the last layer
    t.max_nodes = 60                                                      # node arrays too small for R + 1
    assert call(0, 6) == binding.OK and call(0, 7) == binding.E_PARAM     # only the last layer writes nodes
    t.max_nodes = 61
    smart = binding.Params(K=8, m=1, W=8, depth=8, R=60, builder=binding.BUILDER_SMART)
    t.n_rows = 61
    assert call(0, 0, params=smart) == binding.E_PARAM                    # top-R builder only


def test_binding_structs_match_the_c_header(binding, tmp_path):
    """The ctypes mirrors of spec_tree_params and spec_tree_t have the header's sizes and field offsets."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    fields = {"spec_tree_params": binding.c_params, "spec_tree_t": binding.c_tree}
    # the C names of the binding's fields (the binding spells lambda as lam)
    cname = {"lam": "lambda"}
    src = ["#include <stddef.h>", "#include <stdio.h>", '#include "spec_tree.h"', "int main(void) {"]
    for st, cls in fields.items():
        src.append(f'  printf("{st} %zu\\n", sizeof({st}));')
        for f, _ in cls._fields_:
            c = cname.get(f, f)
            src.append(f'  printf("{st}.{f} %zu\\n", offsetof({st}, {c}));')
    src.append('  printf("SPEC_TREE_STATIC_MAX_TREES %d\\n", (int)SPEC_TREE_STATIC_MAX_TREES);')
    src += ["  return 0;", "}"]
    c_file, exe = tmp_path / "abi.c", tmp_path / "abi"
    c_file.write_text("\n".join(src) + "\n")
    subprocess.run([cc, "-I", os.path.join(ROOT, "include"), str(c_file), "-o", str(exe)], check=True)
    got = dict(line.split() for line in subprocess.run([str(exe)], capture_output=True, text=True,
                                                       check=True).stdout.splitlines())
    assert int(got["SPEC_TREE_STATIC_MAX_TREES"]) == binding.STATIC_MAX_TREES
    for st, cls in fields.items():
        assert int(got[st]) == ctypes.sizeof(cls), st
        for f, _ in cls._fields_:
            assert int(got[f"{st}.{f}"]) == getattr(cls, f).offset, (st, f)
