"""Parity of the chained layer step (skv_decode_layer_step, called through
the C ABI) with the oracle chain, over several decode steps that each append
a token.

Per step and request: the appended token's int8 K/V rows (and, with the
host tier, its int4 host row) are bit-exact; its sketch codes and the folded
query equal the oracle's except +-1 at rounding ties; the selection is
bit-exact against the oracle's score + top-k on the query the step folded
(the appended token is in the tail, so its sketch row is never scored); with
the host tier the hot-buffer misses and the HBM pool (sinks, tail ring, hot
slots) are bit-exact against the oracle's CLOCK resolve; attention is within
2e-3 of the oracle's fp64 attention over the same rows.
"""
import math
import mmap

import numpy as np
import pytest
import torch

import skvtest as T
import workloads as wl

pytestmark = pytest.mark.gpu

ATOL = 2e-3


@pytest.fixture(scope="module")
def skv():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from sparse_kv_long_gb300 import _build
    _build.build()
    import sparse_kv_long_gb300 as m
    return m


def _drift(rng, qf, eta, d):
    """q_s = unit(q_{s-1} + eta * xi) * |q_{s-1}| per head."""
    xi = rng.standard_normal(qf.shape).astype(np.float32)
    nq = np.linalg.norm(qf, axis=-1, keepdims=True)
    qn = qf + eta * nq / math.sqrt(d) * xi
    return (qn / np.linalg.norm(qn, axis=-1, keepdims=True) * nq).astype(np.float32)


def _check_fold_and_selection(orc, x, qb, q8_gpu, sk, L, k, S, W, gidx, gcnt, Hkv):
    ref_q = orc.sketch_query(qb, Hkv, x["basis"], x["c"])
    T.assert_codes_match_except_ties(q8_gpu, ref_q["q8"], ref_q["x"])
    sc = orc.index_score(orc.SKETCH_INT4, q8_gpu, sk, L, S=S, W=W)
    ridx, rcnt = orc.topk_select(sc["okey"], L, k, S=S, W=W)
    assert np.array_equal(gcnt, rcnt)
    for b in range(len(L)):
        assert np.array_equal(gidx[b, :gcnt[b]], ridx[b, :rcnt[b]])
    return ridx, rcnt


@pytest.mark.parametrize("lengths", [[9000, 5000, 3137], [2500, 40_000], [500, 1090, 70_001]],
                         ids=["ragged", "dense_and_sparse", "shorter_than_sinks_and_tail"])
def test_layer_step_resident_matches_oracle_chain(skv, orc, lengths):
    B, Hq, Hkv, d, r, k, S, W = len(lengths), 24, 4, 256, 64, 2048, 64, 1024
    n_steps = 3
    final = [t + n_steps - 1 for t in lengths]
    x = wl.sketch_inputs_cpu(B, final, Hq, Hkv, d, r, seed=77 + B)
    n_cap = int(max(final)) + 5
    Tf = int(max(final))
    # the oracle's caches of every token; the device starts with the tokens
    # before the first step's current token, the rest filled with a pattern
    sk_all = orc.sketch_project(x["K"].reshape(B * Tf, Hkv, d), x["basis"], x["c"])
    q4_all = sk_all["q4"].reshape(B, Tf, -1)
    k8_all, ks_all = orc.quant_int8_rows(x["K"])
    v8_all, vs_all = orc.quant_int8_rows(x["V"])
    sk = np.full((B, n_cap, Hkv * r // 2), 0x5A, np.uint8)
    k8 = np.full((B, n_cap, Hkv, d), 0x33, np.int8)
    v8 = np.full((B, n_cap, Hkv, d), 0x33, np.int8)
    ks = np.full((B, n_cap, Hkv), 0x3C00, np.uint16)
    vs = np.full((B, n_cap, Hkv), 0x3C00, np.uint16)
    for b, t0 in enumerate(lengths):
        sk[b, :t0 - 1] = q4_all[b, :t0 - 1]
        k8[b, :t0 - 1], ks[b, :t0 - 1] = k8_all[b, :t0 - 1], ks_all[b, :t0 - 1]
        v8[b, :t0 - 1], vs[b, :t0 - 1] = v8_all[b, :t0 - 1], vs_all[b, :t0 - 1]
    g_sk, g_k8, g_v8 = T.dev(sk), T.dev(k8.reshape(B * n_cap, Hkv, d)), T.dev(v8.reshape(B * n_cap, Hkv, d))
    g_ks, g_vs = T.f16_dev(ks.reshape(B * n_cap, Hkv)), T.f16_dev(vs.reshape(B * n_cap, Hkv))
    U, c = T.dev(x["basis"]), T.dev(x["c"])
    max_rows = S + k + W
    idx = torch.zeros((B, max_rows), dtype=torch.int32, device="cuda")
    cnt = torch.zeros((B,), dtype=torch.int32, device="cuda")
    q8 = torch.zeros((B, Hkv * r), dtype=torch.int8, device="cuda")
    out = torch.zeros((B, Hq, d), dtype=torch.float32, device="cuda")
    rng = np.random.default_rng(9)
    qf = wl.bf16_bits_to_f32(x["q"])
    ws = None
    for step in range(n_steps):
        if step:
            qf = _drift(rng, qf, 0.3, d)
        qb = wl.to_bf16_bits(qf)
        L = np.array([t + step for t in lengths], np.int32)
        cur = L - 1
        nk = np.stack([x["K"][b, cur[b]] for b in range(B)])
        nv = np.stack([x["V"][b, cur[b]] for b in range(B)])
        g_q, g_nk, g_nv, g_L = T.bf16_dev(qb), T.bf16_dev(nk), T.bf16_dev(nv), T.dev(L)
        args = skv.layer_step_args(q=g_q, new_k=g_nk, new_v=g_nv, lengths=g_L, basis=U, c=c, sketch=g_sk, k8=g_k8,
                                   k_scale=g_ks, v8=g_v8, v_scale=g_vs, idx=idx, count=cnt, out=out, k=k, S=S, W=W,
                                   softmax_scale=1 / 16.0, q8_out=q8)
        if ws is None:
            ws = torch.zeros((skv.decode_layer_step_workspace_size(args),), dtype=torch.uint8, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        skv.decode_layer_step(args, ws, status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        # the appended token: int8 rows bit-exact, sketch codes up to rounding ties
        hk8, hv8 = T.host(g_k8).reshape(B, n_cap, Hkv, d), T.host(g_v8).reshape(B, n_cap, Hkv, d)
        hks, hvs = T.host(g_ks).reshape(B, n_cap, Hkv), T.host(g_vs).reshape(B, n_cap, Hkv)
        hsk = T.host(g_sk)
        for b in range(B):
            t = cur[b]
            assert np.array_equal(hk8[b, t], k8_all[b, t]) and np.array_equal(hks[b, t], ks_all[b, t])
            assert np.array_equal(hv8[b, t], v8_all[b, t]) and np.array_equal(hvs[b, t], vs_all[b, t])
            T.assert_codes_match_except_ties(T.unpack_int4(hsk[b, t]), T.unpack_int4(q4_all[b, t]),
                                             sk_all["x"].reshape(B, Tf, -1)[b, t])
            k8[b, t], ks[b, t], v8[b, t], vs[b, t] = k8_all[b, t], ks_all[b, t], v8_all[b, t], vs_all[b, t]
            sk[b, t] = hsk[b, t]
        assert np.array_equal(hk8, k8) and np.array_equal(hsk, sk)  # nothing else was written
        gidx, gcnt = T.host(idx), T.host(cnt)
        ridx, rcnt = _check_fold_and_selection(orc, x, qb, T.host(q8), sk, L, k, S, W, gidx, gcnt, Hkv)
        ref = orc.attend(orc.KV_INT8, qb, k8.reshape(B * n_cap, -1), v8.reshape(B * n_cap, -1), ridx, rcnt, 1 / 16.0,
                         Hkv, d, d, k_scale=ks.reshape(B * n_cap, Hkv), v_scale=vs.reshape(B * n_cap, Hkv),
                         req_row_stride=n_cap)
        err = np.max(np.abs(T.host(out) - ref))
        assert err < ATOL, (step, err)


def test_layer_step_host_clock_matches_oracle_chain(skv, orc):
    """Host int4 tier in registered host memory behind the windowed-CLOCK hot
    buffer: the step writes the token's int4 host row and its int8 tail-ring
    row, selects, resolves (misses fetched zero-copy) and attends."""
    B, Hq, Hkv, d, r, k, S, W = 2, 24, 4, 256, 64, 512, 64, 256
    lengths = [20000, 12001]
    n_steps = 4
    final = [t + n_steps - 1 for t in lengths]
    x = wl.sketch_inputs_cpu(B, final, Hq, Hkv, d, r, seed=131)
    Tf = int(max(final))
    n_cap = Tf + 3
    Hs = 3 * k // 2
    R = S + W + Hs
    max_rows = S + k + W
    rb = orc.int4_row_bytes(d)
    q4_all = orc.sketch_project(x["K"].reshape(B * Tf, Hkv, d), x["basis"], x["c"])["q4"].reshape(B, Tf, -1)
    host_all = np.stack([orc.quant_int4_rows(x["K"]), orc.quant_int4_rows(x["V"])], axis=3)  # [B][Tf][Hkv][2][rb]
    k8_all, ks_all = orc.quant_int8_rows(x["K"])
    v8_all, vs_all = orc.quant_int8_rows(x["V"])
    sk = np.zeros((B, n_cap, Hkv * r // 2), np.uint8)
    sk[:, :Tf] = q4_all
    host = np.full((B, n_cap, Hkv, 2, rb), 0x5C, np.uint8)
    k8 = np.zeros((B, R, Hkv, d), np.int8)
    v8 = np.zeros((B, R, Hkv, d), np.int8)
    ks = np.zeros((B, R, Hkv), np.uint16)
    vs = np.zeros((B, R, Hkv), np.uint16)
    for b, t0 in enumerate(lengths):
        host[b, :t0 - 1] = host_all[b, :t0 - 1]
        for t in list(range(S)) + list(range(t0 - W, t0 - 1)):  # the tail before the first step's token
            row = t if t < S else S + t % W
            k8[b, row], v8[b, row], ks[b, row], vs[b, row] = k8_all[b, t], v8_all[b, t], ks_all[b, t], vs_all[b, t]
    mm = mmap.mmap(-1, host.nbytes)
    harr = np.frombuffer(mm, dtype=np.uint8, count=host.nbytes)
    harr[:] = host.reshape(-1)
    alias = skv.host_register(harr.ctypes.data, host.nbytes)
    hview = harr.reshape(host.shape)
    try:
        g_sk = T.dev(sk)
        g_k8, g_v8 = T.dev(k8.reshape(B * R, Hkv, d)), T.dev(v8.reshape(B * R, Hkv, d))
        g_ks, g_vs = T.f16_dev(ks.reshape(B * R, Hkv)), T.f16_dev(vs.reshape(B * R, Hkv))
        g_tok = torch.full((B, Hs), -1, dtype=torch.int32, device="cuda")
        g_ref = torch.zeros((B, Hs), dtype=torch.uint8, device="cuda")
        g_use = torch.full((B, Hs), -1, dtype=torch.int32, device="cuda")
        g_tslot = torch.full((B, n_cap), -1, dtype=torch.int32, device="cuda")
        g_hand = torch.zeros((B,), dtype=torch.int32, device="cuda")
        g_step = torch.zeros((2,), dtype=torch.int32, device="cuda")
        states = [orc.ClockState(Hs, n_cap) for _ in range(B)]
        U, c = T.dev(x["basis"]), T.dev(x["c"])
        idx = torch.zeros((B, max_rows), dtype=torch.int32, device="cuda")
        cnt = torch.zeros((B,), dtype=torch.int32, device="cuda")
        nmiss = torch.zeros((B,), dtype=torch.int32, device="cuda")
        q8 = torch.zeros((B, Hkv * r), dtype=torch.int8, device="cuda")
        out = torch.zeros((B, Hq, d), dtype=torch.float32, device="cuda")
        rng = np.random.default_rng(12)
        qf = wl.bf16_bits_to_f32(x["q"])
        ws = None
        misses = []
        for step in range(n_steps):
            if step:
                qf = _drift(rng, qf, 0.35, d)
            qb = wl.to_bf16_bits(qf)
            L = np.array([t + step for t in lengths], np.int32)
            cur = L - 1
            nk = np.stack([x["K"][b, cur[b]] for b in range(B)])
            nv = np.stack([x["V"][b, cur[b]] for b in range(B)])
            # the struct holds raw addresses: keep the tensors alive until the step has run
            g_q, g_nk, g_nv, g_L = T.bf16_dev(qb), T.bf16_dev(nk), T.bf16_dev(nv), T.dev(L)
            args = skv.layer_step_args(q=g_q, new_k=g_nk, new_v=g_nv,
                                       lengths=g_L, basis=U, c=c, sketch=g_sk, k8=g_k8, k_scale=g_ks, v8=g_v8,
                                       v_scale=g_vs, idx=idx, count=cnt, out=out, k=k, S=S, W=W,
                                       softmax_scale=1 / 16.0, policy=skv.HOST_CLOCK, Hs=Hs, host_rows=alias,
                                       step=g_step, slot_token=g_tok, ref=g_ref, use_step=g_use, token_slot=g_tslot,
                                       hand=g_hand, n_miss=nmiss, q8_out=q8)
            if ws is None:
                ws = torch.zeros((skv.decode_layer_step_workspace_size(args),), dtype=torch.uint8, device="cuda")
            st = torch.zeros(1, dtype=torch.int32, device="cuda")
            skv.decode_layer_step(args, ws, status=st)
            torch.cuda.synchronize()
            assert int(st.item()) == 0
            # the appended token: int4 host row and int8 tail-ring row bit-exact
            for b in range(B):
                t = cur[b]
                assert np.array_equal(hview[b, t], host_all[b, t]), (step, b)
                host[b, t] = host_all[b, t]
                row = S + t % W
                k8[b, row], v8[b, row], ks[b, row], vs[b, row] = k8_all[b, t], v8_all[b, t], ks_all[b, t], vs_all[b, t]
            gidx, gcnt = T.host(idx), T.host(cnt)
            ridx, rcnt = _check_fold_and_selection(orc, x, qb, T.host(q8), sk[:, :n_cap], L, k, S, W, gidx, gcnt, Hkv)
            rrows = np.zeros((B, max_rows), np.int32)
            step_miss = []
            for b in range(B):
                n = int(rcnt[b])
                rr, m = states[b].resolve(int(L[b]), S, W, ridx[b, :n], step, host[b], k8[b], v8[b], ks[b], vs[b],
                                          Hkv, d)
                rrows[b, :n] = rr
                assert int(nmiss[b].item()) == m
                step_miss.append(m)
            misses.append(step_miss)
            np.testing.assert_array_equal(T.host(g_k8).reshape(k8.shape), k8)
            np.testing.assert_array_equal(T.host(g_vs).reshape(vs.shape), vs)
            np.testing.assert_array_equal(T.host(g_tok), np.stack([s.slot_token for s in states]))
            ref = orc.attend(orc.KV_INT8, qb, k8.reshape(B * R, -1), v8.reshape(B * R, -1), rrows, rcnt, 1 / 16.0,
                             Hkv, d, d, k_scale=ks.reshape(B * R, Hkv), v_scale=vs.reshape(B * R, Hkv),
                             req_row_stride=R)
            err = np.max(np.abs(T.host(out) - ref))
            assert err < ATOL, (step, err)
        assert misses[0] == [k, k]                     # cold start: every pick misses
        assert all(0 < m < k for m in misses[-1])      # the drift keeps part of the set hot
        assert np.all(hview[:, Tf:] == 0x5C)           # host rows past the appended tokens untouched
    finally:
        skv.host_unregister(harr.ctypes.data)
