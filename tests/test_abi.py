"""The C ABI library builds, loads without a GPU, exports every symbol that
include/*.h declares, and rejects bad arguments on the host before launching."""
import ctypes

import pytest

import skvtest


@pytest.fixture(scope="module")
def lib():
    from sparse_kv_long_gb300 import _build
    _build.build()
    import sparse_kv_long_gb300 as skv
    return skv.lib()


def test_header_declares_the_hot_path():
    names = skvtest.declared_symbols()
    for must in ["skv_sketch_project", "skv_sketch_query", "skv_pool_keys", "skv_index_score",
                 "skv_topk_select", "skv_sparse_attend_decode", "skv_host_register"]:
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in skvtest.declared_symbols() if not hasattr(lib, n)]
    assert not missing, missing


def test_version_and_status_strings(lib):
    assert lib.skv_version() == 1
    assert lib.skv_status_string(0) == b"ok"
    assert lib.skv_status_string(1) == b"invalid argument"


def test_host_side_argument_checks(lib):
    P = ctypes.c_void_p
    # r must be 64
    assert lib.skv_sketch_project(P(16), 4, 2, 256, 32, P(16), None, None, P(16), None) == 1
    # negative batch
    assert lib.skv_index_score(0, -1, 256, P(16), P(16), 10, P(16), 1, 0, 0, P(16), None, None, None) == 1
    # k must be >= 1
    assert lib.skv_topk_select(1, P(16), 10, P(16), 0, 0, 0, 1, P(16), 10, P(16), P(16), 1 << 20,
                               None, None) == 1
    # max_rows too small for S + k + W
    assert lib.skv_topk_select(1, P(16), 10, P(16), 4, 2, 2, 1, P(16), 7, P(16), P(16), 1 << 20,
                               None, None) == 1
    # pooled mode takes no sinks or tail
    assert lib.skv_topk_select(1, P(16), 10, P(16), 4, 1, 0, 4, P(16), 100, P(16), P(16), 1 << 20,
                               None, None) == 1
    # head dim other than 256 is not implemented by the attention kernel
    assert lib.skv_attend_workspace_size(1, 8, 2, 128, 64) == 0
    assert lib.skv_sparse_attend_decode(0, 1, 8, 2, 128, P(16), P(16), P(16), None, None, 0, 10,
                                        P(16), 16, P(16), 1.0, P(16), P(16), 1 << 20, None, None) == 2
    # empty inputs are a no-op success
    assert lib.skv_sketch_project(P(16), 0, 2, 256, 64, P(16), None, None, P(16), None) == 0
    assert lib.skv_pool_keys(P(16), 0, 64, 128, 4, 0, 4, P(16), None) == 0
    assert lib.skv_pool_keys(P(16), 1, 64, 128, 4, 10, 8, P(16), None) == 1  # past capacity
    assert lib.skv_topk_workspace_size(8) > 0
    # gather probe: rows of a multiple of 16 bytes from an aligned base; none is a no-op
    assert lib.skv_gather_read(P(16), P(16), 4, 24, P(16), None) == 1
    assert lib.skv_gather_read(P(8), P(16), 4, 32, P(16), None) == 1
    assert lib.skv_gather_read(P(16), P(16), -1, 32, P(16), None) == 1
    assert lib.skv_gather_read(P(16), P(16), 0, 32, P(16), None) == 0


def test_prefill_argument_checks(lib):
    P = ctypes.c_void_p
    # scores: odd key stride, stride below n_blocks, negative nq; empty is a no-op
    assert lib.skv_prefill_index_scores(4, P(16), P(16), 10, P(16), 11, None, None) == 1
    assert lib.skv_prefill_index_scores(4, P(16), P(16), 10, P(16), 8, None, None) == 1
    assert lib.skv_prefill_index_scores(-1, P(16), P(16), 10, P(16), 10, None, None) == 1
    assert lib.skv_prefill_index_scores(0, P(16), P(16), 10, P(16), 10, None, None) == 0
    assert lib.skv_prefill_index_scores(4, P(16), P(16), 10, P(12), 10, None, None) == 1  # keys not 8-aligned
    # attention: head dim 256 only, Hq % Hkv, chunk >= 1; nq == 0 is a no-op
    args = lambda nq, Hq, Hkv, d, chunk: (nq, Hq, Hkv, d, P(16), P(16), P(16), 100, P(16), P(16), chunk,
                                          P(16), 8, P(16), 1.0, P(16), P(16), None, None)
    assert lib.skv_prefill_attend(*args(2, 16, 2, 128, 64)) == 1
    assert lib.skv_prefill_attend(*args(2, 16, 3, 256, 64)) == 1
    assert lib.skv_prefill_attend(*args(2, 16, 2, 256, 0)) == 1
    assert lib.skv_prefill_attend(*args(0, 16, 2, 256, 64)) == 0


def test_layer_step_struct_matches_the_header(lib, tmp_path):
    """The binding's LayerStep has the size and field offsets that a C
    compiler gives skv_layer_step (include/sparsekv.h)."""
    import shutil
    import subprocess

    import sparse_kv_long_gb300 as skv
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    names = [f[0] for f in skv.LayerStep._fields_]
    src = tmp_path / "layout.c"
    body = "".join(f'  printf("{n} %zu\\n", offsetof(skv_layer_step, {n}));\n' for n in names)
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "sparsekv.h"\nint main(void) {\n'
                   '  printf("size %zu\\n", sizeof(skv_layer_step));\n' + body + "  return 0;\n}\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-I", str(skvtest.ROOT) + "/include", str(src), "-o", str(exe)], check=True)
    got = dict(line.split() for line in subprocess.run([str(exe)], capture_output=True, text=True,
                                                       check=True).stdout.splitlines())
    assert int(got["size"]) == ctypes.sizeof(skv.LayerStep)
    for n in names:
        assert int(got[n]) == getattr(skv.LayerStep, n).offset, n


def test_layer_step_argument_checks(lib):
    import sparse_kv_long_gb300 as skv
    a = skv.LayerStep()
    a.B, a.Hq, a.Hkv, a.d, a.r, a.n_cap, a.k, a.S, a.W = 2, 24, 4, 256, 64, 1000, 64, 4, 16
    ws = ctypes.c_void_p(256)
    assert lib.skv_decode_layer_step(ctypes.byref(a), ws, 1 << 30, None, None) == 1  # null pointers
    a.r = 32
    assert lib.skv_decode_layer_step_workspace_size(ctypes.byref(a)) == 0             # rank must be 64
    a.r, a.W = 64, 0
    assert lib.skv_decode_layer_step_workspace_size(ctypes.byref(a)) == 0             # the tail holds the new token
    a.W, a.policy, a.Hs = 16, 1, 10
    assert lib.skv_decode_layer_step_workspace_size(ctypes.byref(a)) == 0             # fewer hot slots than picks
    assert lib.skv_decode_layer_step(None, ws, 1 << 30, None, None) == 1
