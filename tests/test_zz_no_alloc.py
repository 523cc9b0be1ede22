"""The no-allocation top-k entry point against the regular one.

skv_topk_select_noalloc exists for callers that cannot hand the library any
scratch memory (an engine that has reserved all device memory for its own KV
pools, or a decode loop that must not call cudaMalloc).  It keeps its scratch
in a fixed device array inside the library.  This test calls it through the C
ABI several times in a row (4, 3, then the full 32 requests, then 3 again), on
different inputs, and checks that each result equals
what skv_topk_select returns with a caller-provided workspace (selections are
integer results, so equality is exact).  It also checks that a batch larger
than the fixed capacity is refused before any launch.

The file name makes pytest collect it last.
"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def skv():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from sparse_kv_long_gb300 import _build
    _build.build()
    import sparse_kv_long_gb300 as m
    fn = m.lib().skv_topk_select_noalloc
    P, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    fn.argtypes = [i32, P, i64, P, i32, i32, i32, i32, P, i32, P, P, P]
    fn.restype = i32
    return m


def _noalloc(skv, okeys, lengths, k, S, W, ratio, idx, count, status):
    B, n_cap = okeys.shape
    return skv.lib().skv_topk_select_noalloc(
        B, okeys.data_ptr(), n_cap, lengths.data_ptr(), k, S, W, ratio, idx.data_ptr(), idx.shape[1],
        count.data_ptr(), status.data_ptr(), torch.cuda.current_stream().cuda_stream)


def test_noalloc_matches_workspace_version_on_two_calls(skv):
    rng = np.random.default_rng(4242)
    cases = [
        dict(lengths=[250_000, 9000, 3136, 40_000], k=2048, S=64, W=1024, ratio=1, alphabet=None),
        dict(lengths=[70_001, 3137, 12_345], k=512, S=0, W=0, ratio=4, alphabet=5),  # heavy ties
        # the capacity of the fixed array (32 requests), then a smaller call
        # again: what a larger call left in the array must not leak into it
        dict(lengths=list(rng.integers(3137, 30_000, 32)), k=1024, S=32, W=256, ratio=1, alphabet=None),
        dict(lengths=[20_000, 5000, 8191], k=300, S=4, W=8, ratio=1, alphabet=7),
    ]
    for case in cases:
        L = np.array(case["lengths"], np.int32)
        B = len(L)
        ratio = case["ratio"]
        n_cap = int(L.max()) if ratio == 1 else int(L.max()) // ratio + 1
        if case["alphabet"] is None:
            keys = rng.integers(0, 2 ** 32, (B, n_cap), dtype=np.uint64).astype(np.uint32)
        else:
            keys = (0x80000000 + rng.integers(0, case["alphabet"], (B, n_cap))).astype(np.uint32)
        k, S, W = case["k"], case["S"], case["W"]
        max_rows = S + k + W if ratio == 1 else ratio * k + ratio - 1
        okeys = torch.from_numpy(keys.view(np.int32)).cuda()
        Ld = torch.from_numpy(L).cuda()
        idx_a = torch.full((B, max_rows), -1, dtype=torch.int32, device="cuda")
        cnt_a = torch.zeros((B,), dtype=torch.int32, device="cuda")
        ws = torch.zeros((skv.topk_workspace_size(B),), dtype=torch.uint8, device="cuda")
        skv.topk_select(okeys, Ld, k, idx_a, cnt_a, ws, S=S, W=W, ratio=ratio)
        idx_b = torch.full((B, max_rows), -1, dtype=torch.int32, device="cuda")
        cnt_b = torch.zeros((B,), dtype=torch.int32, device="cuda")
        st = torch.zeros((1,), dtype=torch.int32, device="cuda")
        assert _noalloc(skv, okeys, Ld, k, S, W, ratio, idx_b, cnt_b, st) == 0
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        assert torch.equal(cnt_a, cnt_b)
        for b in range(B):
            n = int(cnt_a[b])
            assert torch.equal(idx_a[b, :n], idx_b[b, :n])


def test_noalloc_refuses_batches_beyond_capacity(skv):
    okeys = torch.zeros((33, 100), dtype=torch.int32, device="cuda")
    L = torch.full((33,), 100, dtype=torch.int32, device="cuda")
    idx = torch.zeros((33, 20), dtype=torch.int32, device="cuda")
    cnt = torch.zeros((33,), dtype=torch.int32, device="cuda")
    st = torch.zeros((1,), dtype=torch.int32, device="cuda")
    assert _noalloc(skv, okeys, L, 4, 2, 2, 1, idx, cnt, st) == 4  # SKV_ENOMEM
