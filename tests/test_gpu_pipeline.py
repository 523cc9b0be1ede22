"""End-to-end parity of the chained decode step (a1..a6) with the oracle.

tiny workload (1 x 8192, fp32 sketch, bf16 KV): everything runs on the GPU
from the raw keys; selections may differ from the oracle's only within 1e-3
relative of the k-th score; attention within 2e-3 of the oracle on the
GPU-selected rows; every planted token is selected.

sketch workload at reduced size (ragged batch, int4 sketch, int8 KV): the
GPU scorer, top-k and attention consume the oracle's sketch bytes, q8 and
int8 rows (identical bytes on both sides), so the index sets must be
bit-exact.
"""
import math

import numpy as np
import pytest
import torch

import skvtest as T
import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def skv():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from sparse_kv_long_gb300 import _build
    _build.build()
    import sparse_kv_long_gb300 as m
    return m


def test_tiny_workload_end_to_end(skv, orc):
    w = wl.TINY
    x = wl.tiny_inputs(w)
    B, Tn, Hq, Hkv, d, r = w.B, w.T, w.Hq, w.Hkv, w.d, w.r
    # ---- GPU chain ----
    K = T.bf16_dev(x["K"].reshape(B * Tn, Hkv, d))
    V = T.bf16_dev(x["V"].reshape(B * Tn, Hkv, d))
    q = T.bf16_dev(x["q"])
    U = T.dev(x["basis"])
    L = T.dev(x["lengths"])
    sk = torch.zeros((B * Tn, Hkv * r), dtype=torch.float32, device="cuda")
    skv.sketch_project(K, U, None, sk)
    qp = torch.zeros((B, Hkv * r), dtype=torch.float32, device="cuda")
    skv.sketch_query(q, Hkv, U, None, qp)
    okeys = torch.zeros((B, Tn), dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    skv.index_score(skv.SKETCH_F32, qp, sk.view(B, Tn, Hkv * r), L, okeys, S=w.S, W=w.W, status=st)
    idx = torch.zeros((B, w.max_rows), dtype=torch.int32, device="cuda")
    cnt = torch.zeros((B,), dtype=torch.int32, device="cuda")
    ws = torch.zeros((skv.topk_workspace_size(B),), dtype=torch.uint8, device="cuda")
    skv.topk_select(okeys, L, w.k, idx, cnt, ws, S=w.S, W=w.W, status=st)
    out = torch.zeros((B, Hq, d), dtype=torch.float32, device="cuda")
    aws = torch.zeros((skv.attend_workspace_size(B, Hq, Hkv, d, w.max_rows),), dtype=torch.uint8, device="cuda")
    skv.sparse_attend_decode(skv.KV_BF16, q, K, V, idx, cnt, 1 / math.sqrt(d), out, aws, Hkv,
                             req_row_stride=Tn, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    gidx, gcnt = T.host(idx), T.host(cnt)
    # ---- oracle chain ----
    s_ref = orc.sketch_project(x["K"].reshape(B * Tn, Hkv, d), x["basis"])["s"].reshape(B, Tn, Hkv * r)
    qp_ref = orc.sketch_query(x["q"], Hkv, x["basis"], None, int8=False)["qp"]
    sc = orc.index_score(orc.SKETCH_F32, qp_ref, s_ref, x["lengths"], S=w.S, W=w.W)
    ridx, rcnt = orc.topk_select(sc["okey"], x["lengths"], w.k, S=w.S, W=w.W)
    assert gcnt[0] == rcnt[0] == w.max_rows
    cand = np.sort(sc["fscore"][0, w.S:Tn - w.W])[::-1]
    kth = cand[w.k - 1]
    diff = T.assert_sets_within_tolerance(gidx[0, :gcnt[0]], ridx[0, :rcnt[0]], lambda t: sc["fscore"][0, t], kth)
    assert np.all(np.diff(gidx[0, :gcnt[0]]) > 0)  # ascending
    sel = set(gidx[0, :gcnt[0]].tolist())
    assert all(int(p) in sel for p in x["planted"][0]), "a planted token was missed"
    ref = orc.attend(orc.KV_BF16, x["q"], x["K"].reshape(B * Tn, -1), x["V"].reshape(B * Tn, -1), gidx, gcnt,
                     1 / math.sqrt(d), Hkv, d, d, req_row_stride=Tn)
    err = np.max(np.abs(T.host(out) - ref))
    assert err < 2e-3, err
    print(f"tiny: {diff} tokens differ near the k-th score; max abs err {err:.2e}")


@pytest.mark.parametrize("lengths", [[9000, 5000, 3136, 3137], [40000]])
def test_sketch_workload_small_bit_exact_sets(skv, orc, lengths):
    B, Hq, Hkv, d, r, k, S, W = len(lengths), 24, 4, 256, 64, 2048, 64, 1024
    x = wl.sketch_inputs_cpu(B, lengths, Hq, Hkv, d, r, seed=11 + len(lengths))
    Tcap = int(max(lengths))
    L = x["lengths"]
    # oracle bytes
    sk = orc.sketch_project(x["K"].reshape(B * Tcap, Hkv, d), x["basis"], x["c"])["q4"].reshape(B, Tcap, Hkv * r // 2)
    qq = orc.sketch_query(x["q"], Hkv, x["basis"], x["c"])
    k8, ks = orc.quant_int8_rows(x["K"].reshape(B * Tcap, Hkv, d))
    v8, vs = orc.quant_int8_rows(x["V"].reshape(B * Tcap, Hkv, d))
    sc = orc.index_score(orc.SKETCH_INT4, qq["q8"], sk, L, S=S, W=W)
    ridx, rcnt = orc.topk_select(sc["okey"], L, k, S=S, W=W)
    # GPU on the same bytes
    okeys = torch.zeros((B, Tcap), dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    Ld = T.dev(L)
    skv.index_score(skv.SKETCH_INT4, T.dev(qq["q8"]), T.dev(sk), Ld, okeys, S=S, W=W, status=st)
    max_rows = S + k + W
    idx = torch.zeros((B, max_rows), dtype=torch.int32, device="cuda")
    cnt = torch.zeros((B,), dtype=torch.int32, device="cuda")
    ws = torch.zeros((skv.topk_workspace_size(B),), dtype=torch.uint8, device="cuda")
    skv.topk_select(okeys, Ld, k, idx, cnt, ws, S=S, W=W, status=st)
    out = torch.zeros((B, Hq, d), dtype=torch.float32, device="cuda")
    aws = torch.zeros((skv.attend_workspace_size(B, Hq, Hkv, d, max_rows),), dtype=torch.uint8, device="cuda")
    skv.sparse_attend_decode(skv.KV_INT8, T.bf16_dev(x["q"]), T.dev(k8), T.dev(v8), idx, cnt, 1 / 16.0, out, aws,
                             Hkv, k_scale=T.f16_dev(ks), v_scale=T.f16_dev(vs), req_row_stride=Tcap, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    gidx, gcnt = T.host(idx), T.host(cnt)
    assert np.array_equal(gcnt, rcnt)
    for b in range(B):
        assert np.array_equal(gidx[b, :gcnt[b]], ridx[b, :rcnt[b]])
    ref = orc.attend(orc.KV_INT8, x["q"], k8.reshape(B * Tcap, -1), v8.reshape(B * Tcap, -1), ridx, rcnt, 1 / 16.0,
                     Hkv, d, d, k_scale=ks, v_scale=vs, req_row_stride=Tcap)
    err = np.max(np.abs(T.host(out) - ref))
    assert err < 2e-3, err
