"""Full-size parity in the benchmark's launch configuration.

One layer-step of the sketch workload -- 8 requests x 250,000 tokens, 24
query / 4 KV heads, head dim 256, int8 K/V, int4 rank-64 sketch, top 2048 +
64 sinks + 1024 tail -- built and launched by the very code the benchmark
times (bench.SketchWorkloadGPU: fused prepare, fused score + select,
attention), then checked against the oracle:

* prepare: the folded query q8 and the appended token's sketch codes equal
  the oracle's except +-1 at rounding ties; its int8 K/V rows are bit-exact;
* selection: bit-exact for every request against the oracle's score + top-k
  on the same sketch bytes and q8 (all 248,912 candidates per request);
* attention: every output within 2e-3 of the fp64 oracle on the selected rows.
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


def test_sketch_workload_full_size_layer_step(skv, orc):
    import bench
    B, Tn, Hq, Hkv, d, r = bench.W_B, bench.W_T, bench.W_HQ, bench.W_HKV, bench.W_D, bench.W_R
    k, S, W = bench.W_K, bench.W_S, bench.W_W
    w = bench.SketchWorkloadGPU(torch, skv, wl, torch.device("cuda", 0), layers=1)
    w.layer(0)
    torch.cuda.synchronize()
    assert int(w.status.item()) == 0
    U, c = T.host(w.U), T.host(w.c)
    q, nk, nv = T.host(w.q[0]), T.host(w.newk[0]), T.host(w.newv[0])

    # a1 + a2 + int8 append of the current token (row T-1 of every request)
    ref_q = orc.sketch_query(q, Hkv, U, c)
    T.assert_codes_match_except_ties(T.host(w.q8), ref_q["q8"], ref_q["x"])
    ref_sk = orc.sketch_project(nk, U, c)
    sk = T.host(w.sk[0])                                          # [B][T][128] int4 codes
    rk8, rks = orc.quant_int8_rows(nk)
    rv8, rvs = orc.quant_int8_rows(nv)
    last = torch.arange(B, device="cuda") * Tn + (Tn - 1)
    for b in range(B):
        T.assert_codes_match_except_ties(T.unpack_int4(sk[b, Tn - 1]), T.unpack_int4(ref_sk["q4"][b]),
                                         ref_sk["x"][b].ravel())
    np.testing.assert_array_equal(T.host(w.k8[0][last]), rk8)
    np.testing.assert_array_equal(T.host(w.v8[0][last]), rv8)
    np.testing.assert_array_equal(T.host(w.ks[0][last]), rks)
    np.testing.assert_array_equal(T.host(w.vs[0][last]), rvs)

    # a3 + a4 on the same bytes
    L = np.full((B,), Tn, np.int32)
    sc = orc.index_score(orc.SKETCH_INT4, T.host(w.q8), sk, L, S=S, W=W)
    ridx, rcnt = orc.topk_select(sc["okey"], L, k, S=S, W=W)
    gidx, gcnt = T.host(w.idx), T.host(w.cnt)
    np.testing.assert_array_equal(gcnt, rcnt)
    np.testing.assert_array_equal(gidx, ridx)

    # a6 on the selected rows
    n = S + k + W
    phys = (torch.arange(B, device="cuda")[:, None] * Tn + w.idx.long()).reshape(-1)
    k8s, v8s = T.host(w.k8[0][phys]), T.host(w.v8[0][phys])
    kss, vss = T.host(w.ks[0][phys]), T.host(w.vs[0][phys])
    rows = np.tile(np.arange(n, dtype=np.int32), (B, 1))
    ref = orc.attend(orc.KV_INT8, q, k8s.reshape(B * n, -1), v8s.reshape(B * n, -1), rows, gcnt, 1 / math.sqrt(d),
                     Hkv, d, d, k_scale=kss, v_scale=vss, req_row_stride=n)
    err = np.max(np.abs(T.host(w.out[0]) - ref))
    assert err < 2e-3, err


@pytest.mark.parametrize("kv_host", [False, True], ids=["hbm", "host"])
def test_pooled_workload_full_size_layer_step(skv, orc, kv_host):
    """One layer-step of the pooled workload -- 4 requests x 1,048,576 tokens,
    16 query / 2 KV heads, bf16 K/V, 128-dim indexer keys pooled by 4, top 512
    blocks -- built and launched by the benchmark's own code, K/V (and the raw
    indexer keys) in HBM or in registered host memory read zero-copy:

    * pooled keys: all 262,144 blocks per request bit-exact (the one the
      current token completes was pooled again inside the step);
    * selection: equal counts; block sets differ only where the oracle's fp32
      score is within 1e-3 relative of the 512-th; each block expands to its
      4 tokens in ascending order;
    * attention: every output within 2e-3 of the fp64 oracle on the GPU's rows.
    """
    import bench
    w = bench.PooledWorkloadGPU(torch, skv, wl, torch.device("cuda", 0), layers=1, kv_host=kv_host)
    try:
        P = w.P
        B, Tn, Hkv, d, di = P.B, P.T, P.Hkv, P.d, P.d_idx
        w.layer(0)
        torch.cuda.synchronize()
        assert int(w.status.item()) == 0
        kv_bytes = B * Tn * Hkv * d * 2
        if kv_host:
            raw_all = w.hosts[0].arr.view(np.uint16)
            raw = raw_all[kv_bytes:].reshape(B, Tn, di)               # after K and V, in uint16 units
        else:
            raw = T.host(w.keys[0])
        pooled = T.host(w.pooled[0])
        for b in range(B):
            np.testing.assert_array_equal(pooled[b], orc.pool_keys(raw[b], P.ratio))

        L = np.full((B,), Tn, np.int32)
        sc = orc.index_score(orc.POOLED_BF16, T.host(w.qidx[0]), pooled, L, ratio=P.ratio)
        ridx, rcnt = orc.topk_select(sc["okey"], L, P.k_blocks, ratio=P.ratio, max_rows=P.max_rows)
        gidx, gcnt = T.host(w.idx), T.host(w.cnt)
        np.testing.assert_array_equal(gcnt, rcnt)
        n = int(gcnt[0])
        assert n == P.ratio * P.k_blocks
        for b in range(B):
            g = gidx[b, :n].reshape(-1, P.ratio)
            np.testing.assert_array_equal(g - g[:, :1], np.tile(np.arange(P.ratio), (g.shape[0], 1)))
            assert np.all(g[:, 0] % P.ratio == 0) and np.all(np.diff(g[:, 0]) > 0)
            kth = np.sort(sc["fscore"][b, :w.nb])[::-1][P.k_blocks - 1]
            gb, rb = set((g[:, 0] // P.ratio).tolist()), set((ridx[b, :n:P.ratio] // P.ratio).tolist())
            for blk in gb ^ rb:
                assert abs(sc["fscore"][b, blk] - kth) <= 1e-3 * abs(kth)

        # attention on the GPU-selected rows, gathered for the oracle
        if kv_host:
            hk = raw_all[:kv_bytes // 2].reshape(B, Tn, Hkv, d)
            hv = raw_all[kv_bytes // 2:kv_bytes].reshape(B, Tn, Hkv, d)
            ks = np.stack([hk[b, gidx[b, :n]] for b in range(B)])
            vs = np.stack([hv[b, gidx[b, :n]] for b in range(B)])
        else:
            phys = (torch.arange(B, device="cuda")[:, None] * Tn + w.idx[:, :n].long()).reshape(-1)
            ks, vs = T.host(w.K[0][phys]), T.host(w.V[0][phys])
        rows = np.tile(np.arange(n, dtype=np.int32), (B, 1))
        ref = orc.attend(orc.KV_BF16, T.host(w.q[0]), ks.reshape(B * n, -1), vs.reshape(B * n, -1), rows, gcnt,
                         1 / math.sqrt(d), Hkv, d, d, req_row_stride=n)
        err = np.max(np.abs(T.host(w.out) - ref))
        assert err < 2e-3, err
    finally:
        torch.cuda.synchronize()
        w.close()


def test_host_clock_workload_full_size_layer_step(skv, orc):
    """One layer-step of the host-tier workload -- 8 requests x 250,000 tokens,
    int4 K/V rows in registered host memory, HBM holding the sketch, 64 sinks,
    the 1,024-token tail ring and 6,250 CLOCK hot slots per request -- built
    and launched by the benchmark's own code, from a cold hot buffer:

    * selection bit-exact against the oracle on the same sketch bytes and q8;
    * resolver: row ids, misses and every CLOCK state word equal the oracle's
      state machine, and the hot slots it filled (host int4 rows requantised
      to int8) are bit-exact;
    * attention within 2e-3 of the fp64 oracle on the resolved rows.
    """
    import bench
    B, Tn, Hkv, d = bench.W_B, bench.W_T, bench.W_HKV, bench.W_D
    k, S, W = bench.W_K, bench.W_S, bench.W_W
    w = bench.HostClockWorkloadGPU(torch, skv, wl, torch.device("cuda", 0), layers=1, n_steps=2, eta=0.35)
    try:
        R, Hs = w.R, w.Hs
        k8c = T.host(w.k8[0]).reshape(B, R, Hkv, d).copy()
        v8c = T.host(w.v8[0]).reshape(B, R, Hkv, d).copy()
        ksc = T.host(w.ks[0]).reshape(B, R, Hkv).copy()
        vsc = T.host(w.vs[0]).reshape(B, R, Hkv).copy()
        w.set_step(0)
        w.layer(0, lambda name: None)
        torch.cuda.synchronize()
        assert int(w.status.item()) == 0
        L = np.full((B,), Tn, np.int32)
        sc = orc.index_score(orc.SKETCH_INT4, T.host(w.q8), T.host(w.sk[0]), L, S=S, W=W)
        ridx, rcnt = orc.topk_select(sc["okey"], L, k, S=S, W=W)
        gidx, gcnt, grows = T.host(w.idx), T.host(w.cnt), T.host(w.rows)
        np.testing.assert_array_equal(gcnt, rcnt)
        np.testing.assert_array_equal(gidx, ridx)
        host = w.hosts[0].arr.reshape(B, Tn, w.tok_bytes)
        tok, ref, use, tslot, hand = (T.host(w.tok[0]), T.host(w.ref[0]), T.host(w.use[0]), T.host(w.tslot[0]),
                                      T.host(w.hand[0]))
        k8g, v8g = T.host(w.k8[0]).reshape(B, R, Hkv, d), T.host(w.v8[0]).reshape(B, R, Hkv, d)
        for b in range(B):
            n = int(rcnt[b])
            st = orc.ClockState(Hs, Tn)
            rr, m = st.resolve(Tn, S, W, ridx[b, :n], 0, host[b], k8c[b], v8c[b], ksc[b], vsc[b], Hkv, d)
            np.testing.assert_array_equal(grows[b, :n], rr, err_msg=f"rows b={b}")
            assert int(w.nmiss[0, b].item()) == m
            np.testing.assert_array_equal(tok[b], st.slot_token)
            np.testing.assert_array_equal(ref[b], st.ref)
            np.testing.assert_array_equal(use[b], st.use_step)
            np.testing.assert_array_equal(tslot[b], st.token_slot)
            assert int(hand[b]) == int(st.hand[0])
            np.testing.assert_array_equal(k8g[b, S + W:], k8c[b, S + W:])     # the hot slots
            np.testing.assert_array_equal(v8g[b, S + W:], v8c[b, S + W:])
        ks_g, vs_g = T.host(w.ks[0]), T.host(w.vs[0])
        ref_out = orc.attend(orc.KV_INT8, T.host(w.q[0]), k8g.reshape(B * R, -1), v8g.reshape(B * R, -1), grows,
                             gcnt, 1 / math.sqrt(d), Hkv, d, d, k_scale=ks_g, v_scale=vs_g, req_row_stride=R)
        err = np.max(np.abs(T.host(w.out) - ref_out))
        assert err < 2e-3, err
    finally:
        torch.cuda.synchronize()
        w.close()


def test_mla_lru_workload_full_size_layer_step(skv, orc):
    """One layer-step of the latent-row workload -- 32 requests x 142,000
    tokens, fp8 rows of 576, 128 absorbed heads, indexer over raw 128-dim
    bf16 keys, pages of 64 with the oldest 70 % host-only, 4,096 LRU hot
    slots -- built and launched by the benchmark's own code:

    * selection: counts equal; sets differ only within 1e-3 relative of the
      oracle's 2,048-th score;
    * resolver: row ids, misses and the pool bytes it wrote equal the
      oracle's LRU state machine on the GPU's picks;
    * attention of four requests (all 128 heads) within 2e-3 of the fp64
      oracle on the resolved rows.
    """
    import bench
    w = bench.MlaLruWorkloadGPU(torch, skv, wl, torch.device("cuda", 0), layers=1, n_steps=2)
    try:
        B, Tn, K, P, D, DV = w.B, w.T, w.K, w.PAGE, w.D, w.DV
        pool0 = T.host(w.pool[0]).copy()
        w.set_step(0)
        w.layer(0, lambda name: None)
        torch.cuda.synchronize()
        assert int(w.status.item()) == 0
        L = np.full((B,), Tn, np.int32)
        sc = orc.index_score(orc.POOLED_BF16, T.host(w.qidx[0]), T.host(w.keys[0]), L, ratio=1)
        ridx, rcnt = orc.topk_select(sc["okey"], L, K, ratio=1)
        gidx, gcnt, grows = T.host(w.idx), T.host(w.cnt), T.host(w.rows)
        np.testing.assert_array_equal(gcnt, rcnt)
        for b in range(B):
            kth = np.sort(sc["fscore"][b, :Tn])[::-1][K - 1]
            for t in set(gidx[b].tolist()) ^ set(ridx[b].tolist()):
                assert abs(sc["fscore"][b, t] - kth) <= 1e-3 * abs(kth), (b, t)
        bt = T.host(w.bt)
        host = w.hosts[0].arr.reshape(B, Tn, D)
        for b in range(B):
            st = orc.LruState(w.SLOTS, Tn)
            rr, m = st.resolve(gidx[b], P, bt[b], w.hot_base + b * w.hot_stride, 0, host[b], pool0, D)
            np.testing.assert_array_equal(grows[b], rr, err_msg=f"rows b={b}")
            assert int(w.nmiss[0, b].item()) == m
        pool1 = T.host(w.pool[0])
        np.testing.assert_array_equal(pool1, pool0)
        q = T.host(w.q[0])
        for b in (0, 7, 19, 31):
            ref_out = orc.attend(orc.KV_FP8, q[b:b + 1], pool1, pool1, grows[b:b + 1], gcnt[b:b + 1],
                                 1 / math.sqrt(D), 1, D, DV, k_pitch=D, v_pitch=D)
            err = np.max(np.abs(T.host(w.out[b:b + 1]) - ref_out))
            assert err < 2e-3, (b, err)
    finally:
        torch.cuda.synchronize()
        w.close()


def _repeat_selection(launch, idx, cnt, status, reps, check_every=50):
    """Run launch() reps times; the status word stays 0 and every result
    equals the first (a selection is deterministic, so any difference is a
    race between the request's CTAs)."""
    launch()
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    idx0, cnt0 = idx.clone(), cnt.clone()
    for r in range(reps):
        launch()
        if r % check_every == check_every - 1:
            torch.cuda.synchronize()
            assert int(status.item()) == 0, f"status {int(status.item())} after {r + 2} launches"
            assert torch.equal(cnt, cnt0) and torch.equal(idx, idx0), f"result changed after {r + 2} launches"


def test_pooled_selection_repeated_launches(skv):
    """The pooled workload's fused selection (4 x 1,048,576 tokens, 32-bit
    keys: two barriers and the final poll) launched 600 times on one
    workspace: no wait runs out and the picks never change.  A missing
    barrier between the last non-final pass's read of its bin count and the
    final pass's clearing of the shared histogram made this fail within a
    few hundred launches."""
    import bench
    w = bench.PooledWorkloadGPU(torch, skv, wl, torch.device("cuda", 0), layers=1)
    try:
        P = w.P

        def launch():
            skv.score_select(skv.POOLED_BF16, w.qidx[0], w.pooled[0], w.lengths, P.k_blocks, w.idx, w.cnt, w.tws,
                             ratio=P.ratio, status=w.status)

        _repeat_selection(launch, w.idx, w.cnt, w.status, 600)
    finally:
        torch.cuda.synchronize()
        w.close()


@pytest.mark.parametrize("mode", ["f32", "int4"])
def test_sketch_selection_repeated_launches(skv, mode):
    """fp32 sketch keys (three radix passes) and int4 sketch keys (two) over
    8 requests x 120,000 candidates, 600 launches on one workspace."""
    B, Tn, width, k = 8, 120_000, 64 if mode == "f32" else 256, 2048
    g = torch.Generator(device="cuda").manual_seed(11)
    L = torch.full((B,), Tn, dtype=torch.int32, device="cuda")
    if mode == "f32":
        q = torch.randn((B, width), generator=g, device="cuda")
        keys = torch.randn((B, Tn, width), generator=g, device="cuda")
        m = skv.SKETCH_F32
    else:
        q = torch.randint(-127, 128, (B, width), generator=g, device="cuda", dtype=torch.int32).to(torch.int8)
        keys = torch.randint(0, 256, (B, Tn, width // 2), generator=g, device="cuda", dtype=torch.int32).to(torch.uint8)
        m = skv.SKETCH_INT4
    idx = torch.zeros((B, 64 + k + 1024), dtype=torch.int32, device="cuda")
    cnt = torch.zeros((B,), dtype=torch.int32, device="cuda")
    ws = torch.zeros((skv.score_select_workspace_size(B),), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")

    def launch():
        skv.score_select(m, q, keys, L, k, idx, cnt, ws, S=64, W=1024, status=st)

    _repeat_selection(launch, idx, cnt, st, 600)
