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
import mmap

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


@pytest.mark.parametrize("kv_host", [False, True], ids=["hbm", "host"])
def test_pooled_workload_small_end_to_end(skv, orc, kv_host):
    """Pooled indexer (ratio 4) -> fused score+select -> block expansion ->
    bf16 attention, 16 query / 2 KV heads.  Pooled keys bit-exact; selections
    may differ only within 1e-3 relative of the k-th block score; attention
    within 2e-3 of the oracle on the GPU-selected rows.  With kv_host the raw
    indexer keys and the K/V rows are read zero-copy from registered host
    memory (only the pooled keys live in HBM)."""
    B, Hq, Hkv, d, d_idx, kb = 2, 16, 2, 256, 128, 512
    lengths = [40003, 12000]
    x = wl.pooled_inputs_cpu(B, lengths, Hq, Hkv, d, d_idx, seed=23)
    L = x["lengths"]
    Tcap = x["K"].shape[1]
    Tcap4 = x["idx_keys"].shape[1]
    nb_cap = Tcap4 // 4
    mm = None
    if kv_host:
        parts = [np.ascontiguousarray(x["idx_keys"]), np.ascontiguousarray(x["K"]), np.ascontiguousarray(x["V"])]
        sizes = [a.nbytes for a in parts]
        mm = mmap.mmap(-1, sum(sizes))
        harr = np.frombuffer(mm, dtype=np.uint8, count=sum(sizes))
        off = 0
        for a in parts:
            harr[off:off + a.nbytes] = a.view(np.uint8).reshape(-1)
            off += a.nbytes
        alias = skv.host_register(harr.ctypes.data, harr.nbytes)
        keys = skv.HostView(alias, x["idx_keys"].shape, 2)
        Kd = skv.HostView(alias + sizes[0], (B * Tcap, Hkv, d), 2)
        Vd = skv.HostView(alias + sizes[0] + sizes[1], (B * Tcap, Hkv, d), 2)
    else:
        keys = T.bf16_dev(x["idx_keys"])
        Kd = T.bf16_dev(x["K"].reshape(B * Tcap, Hkv, d))
        Vd = T.bf16_dev(x["V"].reshape(B * Tcap, Hkv, d))
    try:
        _pooled_chain_check(skv, orc, x, B, Hq, Hkv, d, d_idx, kb, L, Tcap, nb_cap, keys, Kd, Vd)
    finally:
        if kv_host:
            torch.cuda.synchronize()
            skv.host_unregister(harr.ctypes.data)
            del harr
            mm.close()


def _pooled_chain_check(skv, orc, x, B, Hq, Hkv, d, d_idx, kb, L, Tcap, nb_cap, keys, Kd, Vd):
    # GPU: pool, score + select, attend
    pooled = torch.zeros((B, nb_cap, d_idx), dtype=torch.bfloat16, device="cuda")
    skv.pool_keys(keys, pooled, 0, nb_cap)
    max_rows = 4 * kb + 3
    idx = torch.zeros((B, max_rows), dtype=torch.int32, device="cuda")
    cnt = torch.zeros((B,), dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.zeros((skv.score_select_workspace_size(B),), dtype=torch.uint8, device="cuda")
    skv.score_select(skv.POOLED_BF16, T.bf16_dev(x["q_idx"]), pooled, T.dev(L), kb, idx, cnt, ws, ratio=4,
                     status=st)
    out = torch.zeros((B, Hq, d), dtype=torch.float32, device="cuda")
    aws = torch.zeros((skv.attend_workspace_size(B, Hq, Hkv, d, max_rows),), dtype=torch.uint8, device="cuda")
    skv.sparse_attend_decode(skv.KV_BF16, T.bf16_dev(x["q"]), Kd, Vd, idx, cnt, 1 / math.sqrt(d), out, aws,
                             Hkv, req_row_stride=Tcap, n_pool_rows=B * Tcap, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    # oracle
    pk = np.stack([orc.pool_keys(x["idx_keys"][b], 4) for b in range(B)])
    np.testing.assert_array_equal(T.host(pooled), pk)
    sc = orc.index_score(orc.POOLED_BF16, x["q_idx"], pk, L, ratio=4)
    ridx, rcnt = orc.topk_select(sc["okey"], L, kb, ratio=4, max_rows=max_rows)
    gidx, gcnt = T.host(idx), T.host(cnt)
    assert np.array_equal(gcnt, rcnt)
    for b in range(B):
        nb = int(L[b]) // 4
        kth = np.sort(sc["fscore"][b, :nb])[::-1][kb - 1]
        gblk = set((gidx[b, :4 * kb:4] // 4).tolist())
        rblk = set((ridx[b, :4 * kb:4] // 4).tolist())
        for blk in gblk ^ rblk:
            assert abs(sc["fscore"][b, blk] - kth) <= 1e-3 * abs(kth)
        # the incomplete last block (T mod 4 tokens) is always attended
        tail = int(L[b]) % 4
        np.testing.assert_array_equal(gidx[b, 4 * kb:4 * kb + tail], np.arange(4 * nb, 4 * nb + tail))
    ref = orc.attend(orc.KV_BF16, x["q"], x["K"].reshape(B * Tcap, -1), x["V"].reshape(B * Tcap, -1), gidx, gcnt,
                     1 / math.sqrt(d), Hkv, d, d, req_row_stride=Tcap)
    err = np.max(np.abs(T.host(out) - ref))
    assert err < 2e-3, err


def test_host_clock_workload_small_end_to_end(skv, orc):
    """Host int4 tier behind a windowed-CLOCK hot buffer: int4 score + select
    -> CLOCK resolve (misses fetched zero-copy from registered host memory and
    requantised to int8) -> int8 attention over the request's HBM pool of
    sinks, tail ring and hot slots, over several decode steps with a drifting
    query.  Index sets, row ids and the pool bit-exact; attention within 2e-3."""
    B, Hq, Hkv, d, r, k, S, W = 2, 24, 4, 256, 64, 512, 64, 256
    lengths = [20000, 12001]
    x = wl.sketch_inputs_cpu(B, lengths, Hq, Hkv, d, r, seed=31)
    L = x["lengths"]
    Tcap = int(max(lengths))
    Hs = 3 * k // 2                     # hot slots (>= k; 2.5 % of 250K tokens at full size)
    R = S + W + Hs
    max_rows = S + k + W
    sk = orc.sketch_project(x["K"].reshape(B * Tcap, Hkv, d), x["basis"], x["c"])["q4"].reshape(B, Tcap, -1)
    host = np.stack([orc.quant_int4_rows(x["K"]), orc.quant_int4_rows(x["V"])], axis=3)  # [B][Tcap][Hkv][2][136]
    k8all, ksall = orc.quant_int8_rows(x["K"])
    v8all, vsall = orc.quant_int8_rows(x["V"])
    # HBM pool per request: sinks, tail ring (token t at S + t mod W), hot slots (zero)
    k8 = np.zeros((B, R, Hkv, d), np.int8)
    v8 = np.zeros((B, R, Hkv, d), np.int8)
    ks = np.zeros((B, R, Hkv), np.uint16)
    vs = np.zeros((B, R, Hkv), np.uint16)
    for b in range(B):
        Tb = int(L[b])
        for t in list(range(S)) + list(range(Tb - W, Tb)):
            row = t if t < S else S + t % W
            k8[b, row], v8[b, row], ks[b, row], vs[b, row] = k8all[b, t], v8all[b, t], ksall[b, t], vsall[b, t]
    mm = mmap.mmap(-1, host.nbytes)
    harr = np.frombuffer(mm, dtype=np.uint8, count=host.nbytes)
    harr[:] = host.reshape(-1)
    alias = skv.host_register(harr.ctypes.data, host.nbytes)
    try:
        g = {n: T.dev(a) for n, a in (("k8", k8), ("v8", v8))}
        g["ks"], g["vs"] = T.f16_dev(ks), T.f16_dev(vs)
        g_tok = torch.full((B, Hs), -1, dtype=torch.int32, device="cuda")
        g_ref = torch.zeros((B, Hs), dtype=torch.uint8, device="cuda")
        g_use = torch.full((B, Hs), -1, dtype=torch.int32, device="cuda")
        g_tslot = torch.full((B, Tcap), -1, dtype=torch.int32, device="cuda")
        g_hand = torch.zeros((B,), dtype=torch.int32, device="cuda")
        g_step = torch.zeros((2,), dtype=torch.int32, device="cuda")
        states = [orc.ClockState(Hs, Tcap) for _ in range(B)]
        Ld, skd = T.dev(L), T.dev(sk)
        ws = torch.zeros((skv.score_select_workspace_size(B),), dtype=torch.uint8, device="cuda")
        aws = torch.zeros((skv.attend_workspace_size(B, Hq, Hkv, d, max_rows),), dtype=torch.uint8, device="cuda")
        rng = np.random.default_rng(5)
        qf = wl.bf16_bits_to_f32(x["q"])
        misses = []
        for step in range(6):
            # drifting query: q_s = unit(q_{s-1} + eta * xi) * |q_{s-1}|, per head
            if step:
                xi = rng.standard_normal(qf.shape).astype(np.float32)
                nq = np.linalg.norm(qf, axis=-1, keepdims=True)
                qn = qf + 0.35 * nq / math.sqrt(d) * xi
                qf = (qn / np.linalg.norm(qn, axis=-1, keepdims=True) * nq).astype(np.float32)
            qb = wl.to_bf16_bits(qf)
            qq = orc.sketch_query(qb, Hkv, x["basis"], x["c"])
            idx = torch.zeros((B, max_rows), dtype=torch.int32, device="cuda")
            cnt = torch.zeros((B,), dtype=torch.int32, device="cuda")
            st = torch.zeros(1, dtype=torch.int32, device="cuda")
            skv.score_select(skv.SKETCH_INT4, T.dev(qq["q8"]), skd, Ld, k, idx, cnt, ws, S=S, W=W, status=st)
            rows = torch.zeros((B, max_rows), dtype=torch.int32, device="cuda")
            nmiss = torch.zeros((B,), dtype=torch.int32, device="cuda")
            skv.resolve_rows_clock(Ld, idx, cnt, g_step, S, W, Hs, g_tok, g_ref, g_use, g_tslot, g_hand, alias,
                                   g["k8"], g["v8"], g["ks"], g["vs"], R, rows, nmiss, status=st)
            out = torch.zeros((B, Hq, d), dtype=torch.float32, device="cuda")
            skv.sparse_attend_decode(skv.KV_INT8, T.bf16_dev(qb), g["k8"].view(B * R, Hkv, d),
                                     g["v8"].view(B * R, Hkv, d), rows, cnt, 1 / 16.0, out, aws, Hkv,
                                     k_scale=g["ks"].view(B * R, Hkv), v_scale=g["vs"].view(B * R, Hkv),
                                     req_row_stride=R, status=st)
            torch.cuda.synchronize()
            assert int(st.item()) == 0
            sc = orc.index_score(orc.SKETCH_INT4, qq["q8"], sk, L, S=S, W=W)
            ridx, rcnt = orc.topk_select(sc["okey"], L, k, S=S, W=W)
            gidx, gcnt, grows = T.host(idx), T.host(cnt), T.host(rows)
            assert np.array_equal(gcnt, rcnt)
            rrows = np.zeros_like(grows)
            step_miss = []
            for b in range(B):
                n = int(rcnt[b])
                assert np.array_equal(gidx[b, :n], ridx[b, :n])
                rr, m = states[b].resolve(int(L[b]), S, W, ridx[b, :n], step, host[b], k8[b], v8[b], ks[b], vs[b],
                                          Hkv, d)
                rrows[b, :n] = rr
                assert np.array_equal(grows[b, :n], rr)
                assert int(nmiss[b].item()) == m
                step_miss.append(m)
            misses.append(step_miss)
            np.testing.assert_array_equal(T.host(g["k8"]), k8)
            np.testing.assert_array_equal(T.host(g["vs"]), vs)
            ref = orc.attend(orc.KV_INT8, qb, k8.reshape(B * R, -1), v8.reshape(B * R, -1), rrows, rcnt, 1 / 16.0,
                             Hkv, d, d, k_scale=ks.reshape(B * R, Hkv), v_scale=vs.reshape(B * R, Hkv),
                             req_row_stride=R)
            err = np.max(np.abs(T.host(out) - ref))
            assert err < 2e-3, err
        assert misses[0] == [k, k]                      # cold start: every pick misses
        assert all(0 < m < k for m in misses[-1])       # the drift keeps part of the set hot
    finally:
        skv.host_unregister(harr.ctypes.data)
