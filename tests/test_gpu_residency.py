"""Residency transitions under decode, on the GPU, against the oracle.

"vLLM's Hybrid HiSparse ...", *Three residency states, one block pool*: three
requests decode side by side over a pool too small for all of them.  Two
start fully resident, one reuses a prefix that exists only in host memory
(placeholders, its partial last page brought back by a fill).  Every step
appends a token to each request (opening pages takes blocks, and under
pressure the manager releases the oldest pages that already have a host
copy), copies completed pages to host memory (skv_materialize_pages), and
resolves a set of picks with the LRU resolver.  Checked every step:

* row ids, LRU state and miss counts equal the oracle's state machine run on
  the same block table;
* every resolved row holds the picked token's true bytes -- a page released
  before its host copy, or a fill or copy that moved the wrong rows, shows up
  here (host rows of resident pages start as garbage);
* at the end the pool and the host tier equal the oracle's mirrors byte for
  byte, and the resident requests went from full to mixed (the host-prefix
  request is mixed from the start: placeholders plus its resident tail).
"""
import mmap

import numpy as np
import pytest
import torch

import skvtest as T

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def skv():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from sparse_kv_long_gb300 import _build
    _build.build()
    import sparse_kv_long_gb300 as m
    return m


@pytest.mark.parametrize("leased", [False, True], ids=["reserved_hot", "leased_hot"])
def test_pressure_driven_transitions_under_decode(skv, orc, leased):
    """leased: every request's hot buffer is made of blocks leased from the
    same pool as the resident pages (skv_residency_lease_hot and the leased
    resolver); otherwise a reserved region after the pool's blocks."""
    B, page, t_cap, row_bytes = 3, 16, 1024, 576
    max_pages = t_cap // page
    n_slots, k, n_steps = 40, 24, 48
    n_hp = -(-n_slots // page)                  # hot pages per request
    n_blocks = 60 + (B * n_hp if leased else 0)
    start = [500, 400, 300]                     # requests 0, 1 resident; 2 from a host prefix
    rng = np.random.default_rng(77)
    truth = rng.integers(0, 256, (B, t_cap, row_bytes), dtype=np.uint8)
    hot_base, hot_stride = n_blocks * page, n_slots
    n_pool_rows = n_blocks * page if leased else hot_base + B * hot_stride

    r = skv.Residency(n_blocks, page, B, max_pages, tail_pages=1)
    r.add(0, start[0])
    r.add(1, start[1])
    r.add(2, start[2], host_prefix=True)
    assert r.state(2) == skv.RESIDENCY_MIXED   # placeholders plus the resident partial last page
    hot_rows = [None] * B
    g_hot = None
    if leased:
        hb = np.stack([r.lease_hot(b, n_hp) for b in range(B)])
        assert r.free_blocks() == n_blocks - 58 - B * n_hp
        hot_rows = [(hb[b][np.arange(n_slots) // page] * page + np.arange(n_slots) % page).astype(np.int32)
                    for b in range(B)]
        assert len(set(np.concatenate(hot_rows).tolist())) == B * n_slots
        g_hot = T.dev(hb.astype(np.int32))

    # host tier (registered host memory): only request 2's prefix is there at first
    nbytes = B * t_cap * row_bytes
    mm = mmap.mmap(-1, nbytes)
    harr = np.frombuffer(mm, dtype=np.uint8, count=nbytes)
    harr[:] = 0xEE
    host_cpu = harr.reshape(B, t_cap, row_bytes)
    host_cpu[2, :start[2]] = truth[2, :start[2]]
    alias = skv.host_register(harr.ctypes.data, nbytes)
    # pool: resident pages hold their tokens' rows, everything else garbage
    pool_cpu = np.full((n_pool_rows, row_bytes), 0xDD, np.uint8)
    bt = r.block_table()
    n_tok = list(start)
    for b in range(2):
        for p in range(-(-n_tok[b] // page)):
            t0, t1 = p * page, min((p + 1) * page, n_tok[b])
            pool_cpu[bt[b, p] * page:bt[b, p] * page + (t1 - t0)] = truth[b, t0:t1]
    try:
        g_pool = T.dev(pool_cpu)
        g_stamp = torch.full((B, n_slots), -1, dtype=torch.int64, device="cuda")
        g_tok = torch.full((B, n_slots), -1, dtype=torch.int32, device="cuda")
        g_tslot = torch.full((B, t_cap), -1, dtype=torch.int32, device="cuda")
        g_order = torch.arange(n_slots, dtype=torch.int32, device="cuda").repeat(B, 1).contiguous()
        g_step = torch.zeros((2,), dtype=torch.int32, device="cuda")
        st = torch.zeros((1,), dtype=torch.int32, device="cuda")
        states = [orc.LruState(n_slots, t_cap) for _ in range(B)]
        seen = [set() for _ in range(B)]
        n_released = 0

        def fill_all(bt, g_bt):
            # pages whose first rows are host-only come back into their blocks
            # (before anything is appended into them: the copy is whole-page)
            for b in range(B):
                f = r.fills(b)
                if f.size:
                    pairs = np.stack([np.full(f.size, b, np.int32), f], 1).astype(np.int32)
                    skv.fill_pages(T.dev(pairs), page, g_bt, g_pool, alias, t_cap, status=st)
                    for p in f:
                        pool_cpu[bt[b, p] * page:(bt[b, p] + 1) * page] = host_cpu[b, p * page:(p + 1) * page]
                    r.mark_filled(b, f)

        fill_all(bt, T.dev(bt))                 # admission: request 2's partial page
        assert all(r.fills(b).size == 0 for b in range(B))
        for step in range(n_steps):
            # 1. append this step's token of every request; under pressure pages get released
            for b in range(B):
                before = r.block_table()
                r.append(b, 1)
                t = n_tok[b]
                n_tok[b] += 1
                bt = r.block_table()
                n_released += int(((before >= 0) & (bt < 0)).sum())
                blk = bt[b, t // page]
                assert blk >= 0
                prow = blk * page + t % page
                pool_cpu[prow] = truth[b, t]
                g_pool[prow] = T.dev(truth[b, t])
            g_bt = T.dev(bt)
            assert all(r.fills(b).size == 0 for b in range(B))   # appends open fresh pages only
            # 2. completed resident pages get their host copy, then may be released later
            for b in range(B):
                pend = r.pending(b)
                if pend.size:
                    pairs = np.stack([np.full(pend.size, b, np.int32), pend], 1).astype(np.int32)
                    skv.materialize_pages(T.dev(pairs), page, g_bt, g_pool, alias, t_cap, status=st)
                    for p in pend:
                        host_cpu[b, p * page:(p + 1) * page] = pool_cpu[bt[b, p] * page:(bt[b, p] + 1) * page]
                    r.mark_copied(b, pend)
            for b in range(B):
                seen[b].add(r.state(b))
            # 3. resolve this step's picks
            idx = np.full((B, k), -1, np.int32)
            for b in range(B):
                idx[b] = np.sort(rng.choice(n_tok[b], size=k, replace=False))
            rows = torch.full((B, k), -9, dtype=torch.int32, device="cuda")
            nmiss = torch.zeros((B,), dtype=torch.int32, device="cuda")
            skv.resolve_rows_lru(T.dev(np.array(n_tok, np.int32)), T.dev(idx), T.dev(np.full(B, k, np.int32)), g_step,
                                 page, g_bt, hot_base, hot_stride, g_stamp, g_tok, g_tslot, g_order, alias, g_pool,
                                 rows, nmiss, status=st, hot_blocks=g_hot)
            torch.cuda.synchronize()
            assert int(st.item()) == 0
            got = T.host(rows)
            pool_now = T.host(g_pool)
            for b in range(B):
                ref_rows, m = states[b].resolve(idx[b], page, bt[b], hot_base + b * hot_stride, step, host_cpu[b],
                                                pool_cpu, row_bytes, hot_rows=hot_rows[b])
                np.testing.assert_array_equal(got[b], ref_rows, err_msg=f"rows b={b} step={step}")
                assert int(nmiss[b].item()) == m
                np.testing.assert_array_equal(pool_now[got[b]], truth[b, idx[b]], err_msg=f"bytes b={b} step={step}")
        np.testing.assert_array_equal(T.host(g_pool), pool_cpu)
        np.testing.assert_array_equal(host_cpu, harr.reshape(B, t_cap, row_bytes))
        assert n_released > 0
        assert {skv.RESIDENCY_FULL, skv.RESIDENCY_MIXED} <= seen[0] | seen[1]
        assert skv.RESIDENCY_MIXED in seen[2]
    finally:
        torch.cuda.synchronize()
        skv.host_unregister(harr.ctypes.data)


def test_page_copies_flag_bad_pages(skv):
    """A listed page that is out of range or a placeholder sets SKV_DEV_RANGE
    and moves nothing; the valid ones are copied."""
    B, page, t_cap, row_bytes = 2, 4, 16, 32
    bt = T.dev(np.array([[0, -1, 1, -1], [2, 3, -1, -1]], np.int32))
    pool = torch.arange(4 * page * row_bytes, dtype=torch.int64, device="cuda").to(torch.uint8).view(4 * page, row_bytes)
    host = torch.zeros((B, t_cap, row_bytes), dtype=torch.uint8, device="cuda")
    pairs = T.dev(np.array([[0, 2], [0, 1], [1, 7], [5, 0], [1, 1]], np.int32))
    st = torch.zeros((1,), dtype=torch.int32, device="cuda")
    skv.materialize_pages(pairs, page, bt, pool, host, t_cap, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & skv.DEV_RANGE
    h = T.host(host)
    p = T.host(pool)
    np.testing.assert_array_equal(h[0, 8:12], p[4:8])      # (0, 2) -> block 1
    np.testing.assert_array_equal(h[1, 4:8], p[12:16])     # (1, 1) -> block 3
    assert (h[0, :8] == 0).all() and (h[0, 12:] == 0).all() and (h[1, :4] == 0).all() and (h[1, 8:] == 0).all()
