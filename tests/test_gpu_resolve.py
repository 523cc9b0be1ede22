"""Parity of the a5 resolvers and the host-tier encoding (through the C ABI)
with the CPU oracle: windowed CLOCK over a host int4 tier and the block-table
LRU hot buffer, over a sequence of decode steps with drifting selections.

Bar: bit-exact -- row ids, miss counts, every word of the resolver state and
every byte written to the pools, after every step.
"""
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


def status_word():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


class HostBuffer:
    """Anonymous-mmap host memory registered with the library (zero-copy)."""

    def __init__(self, skv, data: np.ndarray):
        self.skv = skv
        self.nbytes = data.nbytes
        self.mm = mmap.mmap(-1, max(self.nbytes, 4096))
        self.arr = np.frombuffer(self.mm, dtype=np.uint8, count=self.nbytes)
        self.arr[:] = data.reshape(-1).view(np.uint8)
        self.addr = self.arr.ctypes.data
        self.alias = skv.host_register(self.addr, self.nbytes)

    def close(self):
        self.skv.host_unregister(self.addr)
        del self.arr
        self.mm.close()


# ---------------------------------------------------------------------------
# host-tier encoding
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("n,Hkv,d", [(1, 1, 256), (257, 4, 256), (33, 2, 512)])
def test_quantize_int4_rows_bit_exact(skv, orc, n, Hkv, d):
    rng = np.random.default_rng(7 + n)
    x = rng.standard_normal((n, Hkv, d)).astype(np.float32) * rng.uniform(0.01, 50, (n, Hkv, 1))
    x[0, 0, :64] = 0.0                       # a zero group -> zero scale and codes
    if n > 1:
        x[1, 0, 5] = 1e4                     # one outlier dominates its group
    bits = wl.to_bf16_bits(x.astype(np.float32))
    rb = orc.int4_row_bytes(d)
    ref = orc.quant_int4_rows(bits)          # [n][Hkv][rb]
    # host-tier layout: [n][Hkv][K|V][rb]; write this tensor as the V half
    out = torch.full((n, Hkv, 2, rb), 0xAB, dtype=torch.uint8, device="cuda")
    skv.quantize_int4_rows(T.bf16_dev(bits), out[:, :, 1], token_pitch=Hkv * 2 * rb, head_pitch=2 * rb)
    got = T.host(out)
    np.testing.assert_array_equal(got[:, :, 1], ref)
    assert (got[:, :, 0] == 0xAB).all()      # the K half is untouched


# ---------------------------------------------------------------------------
# CLOCK over a host int4 tier
# ---------------------------------------------------------------------------

def _clock_case(orc, seed, B, Hkv, d, S, W, Hs, k, lengths, t_cap, n_steps, keep):
    rng = np.random.default_rng(seed)
    K = wl.to_bf16_bits(rng.standard_normal((B, t_cap, Hkv, d)).astype(np.float32))
    V = wl.to_bf16_bits(rng.standard_normal((B, t_cap, Hkv, d)).astype(np.float32))
    host = np.stack([orc.quant_int4_rows(K), orc.quant_int4_rows(V)], axis=3)  # [B][t_cap][Hkv][2][rb]
    seqs = [wl.pick_sequence(rng, S, int(lengths[b]) - W, k, n_steps, keep) for b in range(B)]
    return host, seqs


def _selection(S, W, Tb, picks):
    return np.concatenate([np.arange(S), picks, np.arange(Tb - W, Tb)]).astype(np.int32)


@pytest.mark.parametrize("Hs,k,keep,where", [(150, 96, 0.8, "device"), (96, 96, 0.5, "device"),
                                             (31, 20, 0.7, "host"), (7, 5, 0.4, "device"),
                                             (150, 60, 0.0, "host")])
def test_clock_resolve_matches_oracle(skv, orc, Hs, k, keep, where):
    B, Hkv, d, S, W = 3, 2, 256, 16, 64
    lengths = np.array([2500, 3000, 1900], np.int32)
    t_cap, n_steps = 3072, 9
    host, seqs = _clock_case(orc, 11 + Hs + k, B, Hkv, d, S, W, Hs, k, lengths, t_cap, n_steps, keep)
    R = S + W + Hs + 5                       # rows per request in the HBM pool
    max_rows = S + W + k + 3
    rng = np.random.default_rng(3)
    k8 = rng.integers(-127, 128, (B, R, Hkv, d), dtype=np.int8)
    v8 = rng.integers(-127, 128, (B, R, Hkv, d), dtype=np.int8)
    ks = rng.integers(0, 0x3c00, (B, R, Hkv), dtype=np.uint16)
    vs = rng.integers(0, 0x3c00, (B, R, Hkv), dtype=np.uint16)
    states = [orc.ClockState(Hs, t_cap) for _ in range(B)]

    g_k8, g_v8, g_ks, g_vs = T.dev(k8), T.dev(v8), T.f16_dev(ks), T.f16_dev(vs)
    g_tok = torch.full((B, Hs), -1, dtype=torch.int32, device="cuda")
    g_ref = torch.zeros((B, Hs), dtype=torch.uint8, device="cuda")
    g_use = torch.full((B, Hs), -1, dtype=torch.int32, device="cuda")
    g_tslot = torch.full((B, t_cap), -1, dtype=torch.int32, device="cuda")
    g_hand = torch.zeros((B,), dtype=torch.int32, device="cuda")
    g_step = torch.zeros((2,), dtype=torch.int32, device="cuda")   # [step, ticket], advanced by each call
    g_len = T.dev(lengths)
    hb = None
    if where == "host":
        hb = HostBuffer(skv, host)
        host_arg = hb.alias
    else:
        host_arg = T.dev(host)
    try:
        for step in range(n_steps):
            idx = np.full((B, max_rows), -7, np.int32)
            count = np.zeros((B,), np.int32)
            for b in range(B):
                sel = _selection(S, W, int(lengths[b]), seqs[b][step])
                idx[b, :len(sel)] = sel
                count[b] = len(sel)
            rows = torch.full((B, max_rows), -9, dtype=torch.int32, device="cuda")
            nmiss = torch.zeros((B,), dtype=torch.int32, device="cuda")
            st = status_word()
            skv.resolve_rows_clock(g_len, T.dev(idx), T.dev(count), g_step, S, W, Hs, g_tok, g_ref, g_use, g_tslot,
                                   g_hand, host_arg, g_k8, g_v8, g_ks, g_vs, R, rows, nmiss, status=st)
            torch.cuda.synchronize()
            assert int(st.item()) == 0
            assert T.host(g_step).tolist() == [step + 1, 0]
            got_rows = T.host(rows)
            for b in range(B):
                n = int(count[b])
                ref_rows, m = states[b].resolve(int(lengths[b]), S, W, idx[b, :n], step, host[b], k8[b], v8[b],
                                                ks[b], vs[b], Hkv, d)
                np.testing.assert_array_equal(got_rows[b, :n], ref_rows, err_msg=f"rows b={b} step={step}")
                assert int(nmiss[b].item()) == m
            np.testing.assert_array_equal(T.host(g_tok), np.stack([s.slot_token for s in states]))
            np.testing.assert_array_equal(T.host(g_ref), np.stack([s.ref for s in states]))
            np.testing.assert_array_equal(T.host(g_use), np.stack([s.use_step for s in states]))
            np.testing.assert_array_equal(T.host(g_tslot), np.stack([s.token_slot for s in states]))
            np.testing.assert_array_equal(T.host(g_hand), np.concatenate([s.hand for s in states]))
            np.testing.assert_array_equal(T.host(g_k8), k8)
            np.testing.assert_array_equal(T.host(g_v8), v8)
            np.testing.assert_array_equal(T.host(g_ks), ks)
            np.testing.assert_array_equal(T.host(g_vs), vs)
    finally:
        if hb is not None:
            hb.close()


def test_clock_more_picks_than_slots_is_flagged(skv):
    B, Hkv, d, S, W, Hs = 1, 1, 256, 4, 8, 10
    t_cap = 256
    idx = np.arange(0, 40, dtype=np.int32)[None]          # 4 sinks + 36 picks (T = 200)
    rows = torch.full((B, 40), -9, dtype=torch.int32, device="cuda")
    nmiss = torch.zeros((B,), dtype=torch.int32, device="cuda")
    tok = torch.full((B, Hs), -1, dtype=torch.int32, device="cuda")
    ref = torch.zeros((B, Hs), dtype=torch.uint8, device="cuda")
    use = torch.full((B, Hs), -1, dtype=torch.int32, device="cuda")
    tslot = torch.full((B, t_cap), -1, dtype=torch.int32, device="cuda")
    hand = torch.zeros((B,), dtype=torch.int32, device="cuda")
    R = S + W + Hs
    k8 = torch.zeros((R, Hkv, d), dtype=torch.int8, device="cuda")
    ks = torch.zeros((R, Hkv), dtype=torch.float16, device="cuda")
    host = torch.zeros((t_cap, Hkv, 2, 136), dtype=torch.uint8, device="cuda")
    st = status_word()
    skv.resolve_rows_clock(T.dev(np.array([200], np.int32)), T.dev(idx), T.dev(np.array([40], np.int32)),
                           torch.zeros(2, dtype=torch.int32, device="cuda"), S, W, Hs, tok, ref, use, tslot, hand, host, k8, k8.clone(), ks, ks.clone(), R, rows, nmiss,
                           status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & 8                              # SKV_DEV_COUNT
    assert int(nmiss.item()) == -1
    got = T.host(rows)[0]
    np.testing.assert_array_equal(got[:4], np.arange(4))
    assert (got[4:] == -1).all()
    assert (T.host(tok) == -1).all() and int(hand.item()) == 0


# ---------------------------------------------------------------------------
# LRU hot buffer behind a block table
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("n_slots,k,keep,where", [(128, 64, 0.7, "device"), (64, 64, 0.3, "host"),
                                                  (100, 37, 0.9, "device"), (5, 3, 0.5, "device")])
def test_lru_resolve_matches_oracle(skv, orc, n_slots, k, keep, where):
    B, page, t_cap, row_bytes = 3, 16, 1024, 576
    lengths = np.array([1000, 1024, 700], np.int32)
    n_pages = t_cap // page
    n_steps = 9
    rng = np.random.default_rng(100 + n_slots + k)
    # block table: pages p < floor(0.7 * ceil(T / page)) are host-only
    bt = np.full((B, n_pages), -1, np.int32)
    for b in range(B):
        n_used = -(-int(lengths[b]) // page)
        first = int(np.floor(0.7 * n_used))
        for p in range(first, n_used):
            bt[b, p] = b * n_pages + p
    hot_base = B * n_pages * page
    hot_stride = n_slots + 3
    n_pool_rows = hot_base + B * hot_stride
    pool = rng.integers(0, 256, (n_pool_rows, row_bytes), dtype=np.uint8)
    host = rng.integers(0, 256, (B, t_cap, row_bytes), dtype=np.uint8)
    seqs = [wl.pick_sequence(rng, 0, int(lengths[b]), k, n_steps, keep) for b in range(B)]
    states = [orc.LruState(n_slots, t_cap) for _ in range(B)]

    g_pool = T.dev(pool)
    g_stamp = torch.full((B, n_slots), -1, dtype=torch.int64, device="cuda")
    g_tok = torch.full((B, n_slots), -1, dtype=torch.int32, device="cuda")
    g_tslot = torch.full((B, t_cap), -1, dtype=torch.int32, device="cuda")
    g_order = torch.arange(n_slots, dtype=torch.int32, device="cuda").repeat(B, 1).contiguous()
    g_bt, g_len = T.dev(bt), T.dev(lengths)
    g_step = torch.zeros((2,), dtype=torch.int32, device="cuda")
    hb = None
    if where == "host":
        hb = HostBuffer(skv, host)
        host_arg = hb.alias
    else:
        host_arg = T.dev(host)
    try:
        for step in range(n_steps):
            idx = np.full((B, k + 2), -5, np.int32)
            count = np.full((B,), k, np.int32)
            for b in range(B):
                idx[b, :k] = seqs[b][step]
            rows = torch.full((B, k + 2), -9, dtype=torch.int32, device="cuda")
            nmiss = torch.zeros((B,), dtype=torch.int32, device="cuda")
            st = status_word()
            skv.resolve_rows_lru(g_len, T.dev(idx), T.dev(count), g_step, page, g_bt, hot_base, hot_stride, g_stamp,
                                 g_tok, g_tslot, g_order, host_arg, g_pool, rows, nmiss, status=st)
            torch.cuda.synchronize()
            assert int(st.item()) == 0
            assert T.host(g_step).tolist() == [step + 1, 0]
            got_rows = T.host(rows)
            for b in range(B):
                ref_rows, m = states[b].resolve(idx[b, :k], page, bt[b], hot_base + b * hot_stride, step, host[b],
                                                pool, row_bytes)
                np.testing.assert_array_equal(got_rows[b, :k], ref_rows, err_msg=f"rows b={b} step={step}")
                assert int(nmiss[b].item()) == m
            np.testing.assert_array_equal(T.host(g_stamp), np.stack([s.stamp for s in states]))
            np.testing.assert_array_equal(T.host(g_tok), np.stack([s.slot_token for s in states]))
            np.testing.assert_array_equal(T.host(g_tslot), np.stack([s.token_slot for s in states]))
            np.testing.assert_array_equal(T.host(g_pool), pool)
            # the maintained LRU order is the (stamp, slot) order of the oracle's stamps
            for b in range(B):
                st_b = states[b].stamp
                np.testing.assert_array_equal(T.host(g_order)[b], np.lexsort((np.arange(n_slots), st_b)))
    finally:
        if hb is not None:
            hb.close()


def test_lru_too_few_slots_is_flagged(skv):
    B, page, t_cap, row_bytes, n_slots = 1, 16, 256, 32, 4
    bt = np.full((B, t_cap // page), -1, np.int32)           # everything host-only
    idx = np.arange(0, 60, 6, dtype=np.int32)[None]          # 10 misses, 4 slots
    pool = torch.zeros((n_slots, row_bytes), dtype=torch.uint8, device="cuda")
    host = torch.ones((B, t_cap, row_bytes), dtype=torch.uint8, device="cuda")
    stamp = torch.full((B, n_slots), -1, dtype=torch.int64, device="cuda")
    tok = torch.full((B, n_slots), -1, dtype=torch.int32, device="cuda")
    tslot = torch.full((B, t_cap), -1, dtype=torch.int32, device="cuda")
    order = torch.arange(n_slots, dtype=torch.int32, device="cuda")[None].contiguous()
    rows = torch.full((B, 10), -9, dtype=torch.int32, device="cuda")
    nmiss = torch.zeros((B,), dtype=torch.int32, device="cuda")
    st = status_word()
    skv.resolve_rows_lru(T.dev(np.array([256], np.int32)), T.dev(idx), T.dev(np.array([10], np.int32)),
                         torch.zeros(2, dtype=torch.int32, device="cuda"), page,
                         T.dev(bt), 0, 0, stamp, tok, tslot, order, host, pool, rows, nmiss, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & 8
    assert int(nmiss.item()) == -1
    assert (T.host(rows) == -1).all()
    assert (T.host(pool) == 0).all()


def test_gather_read_probe_runs_on_device_and_host_memory(skv):
    """The scattered-row read probe runs over device memory and over a
    registered host tier and leaves the status clean."""
    import mmap
    rows = torch.tensor([5, 0, 99, 37, 12], dtype=torch.int64, device="cuda")
    sink = torch.zeros((1,), dtype=torch.int64, device="cuda")
    dev_buf = torch.zeros((100 * 1088,), dtype=torch.uint8, device="cuda")
    skv.gather_read(dev_buf, rows, 1088, sink)
    nbytes = 100 * 1088
    mm = mmap.mmap(-1, nbytes)
    harr = np.frombuffer(mm, dtype=np.uint8, count=nbytes)
    harr[:] = 7
    alias = skv.host_register(harr.ctypes.data, nbytes)
    try:
        skv.gather_read(alias, rows, 1088, sink)
        torch.cuda.synchronize()
    finally:
        skv.host_unregister(harr.ctypes.data)
