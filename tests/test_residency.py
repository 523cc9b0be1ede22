"""The residency manager's policy, on the host (no GPU).

"vLLM's Hybrid HiSparse ...", *Three residency states, one block pool*: a
request keeps its KV in the pool while there is room, completed prefix pages
get a host copy ahead of need, and under pressure the request gives up its
coldest pages (keeping its tail); a request reusing a host-only prefix starts
with placeholders.  These tests hold the manager to its stated rules:
conservation of blocks, release only of copied pages, never the newest page
or the protected tail, the oldest page of the request with the most resident
pages first, and the three states.
"""
import numpy as np
import pytest

import sparse_kv_long_gb300 as skv
from sparse_kv_long_gb300 import SkvError


@pytest.fixture(scope="module", autouse=True)
def built():
    from sparse_kv_long_gb300 import _build
    _build.build()


def resident(table):
    return int((table >= 0).sum())


def test_full_residency_and_host_copies():
    r = skv.Residency(n_blocks=40, page=16, max_requests=3, max_pages=10)
    r.add(0, 100)                       # 7 pages (6 complete)
    r.add(1, 48)                        # 3 complete pages
    t = r.block_table()
    assert resident(t) == 10 and r.free_blocks() == 30
    assert len(set(t[t >= 0].tolist())) == 10          # distinct blocks
    assert r.state(0) == skv.RESIDENCY_FULL and r.state(2) == -1
    np.testing.assert_array_equal(r.pending(0), np.arange(6))
    np.testing.assert_array_equal(r.pending(1), np.arange(3))
    r.mark_copied(0, [0, 1, 2])
    np.testing.assert_array_equal(r.pending(0), [3, 4, 5])
    with pytest.raises(SkvError):
        r.mark_copied(0, [6])                           # page 6 is not complete
    r.append(0, 12)                                     # completes page 6
    np.testing.assert_array_equal(r.pending(0), [3, 4, 5, 6])
    assert resident(r.block_table()) == 10
    r.append(0, 1)                                      # opens page 7
    assert resident(r.block_table()) == 11
    r.remove(1)
    assert r.free_blocks() == 40 - 8


def test_pressure_releases_the_oldest_copied_page_of_the_largest_request():
    page = 4
    r = skv.Residency(n_blocks=10, page=page, max_requests=2, max_pages=16, tail_pages=2)
    r.add(0, 6 * page)                  # 6 blocks
    r.add(1, 4 * page)                  # 4 blocks: the pool is full
    assert r.free_blocks() == 0
    with pytest.raises(SkvError):       # nothing copied yet: nothing may be released
        r.append(0, 1)
    r.mark_copied(0, r.pending(0))
    r.mark_copied(1, r.pending(1))
    before = r.block_table()
    r.append(1, 1)                      # request 1 opens page 4: request 0 (6 resident) gives page 0
    after = r.block_table()
    assert after[0, 0] == -1 and before[0, 0] == after[1, 4]
    assert r.state(0) == skv.RESIDENCY_MIXED and r.state(1) == skv.RESIDENCY_FULL
    # explicit reclaim: request 0 (5 resident) gives its oldest copied pages, never its last 2
    rel = r.reclaim(10)
    # 0 has pages 1..5 resident (4, 5 protected), 1 has 0..4 (3, 4 protected); ties go to the most resident
    assert rel.tolist() == [[0, 1], [1, 0], [0, 2], [1, 1], [0, 3], [1, 2]]
    t = r.block_table()
    assert (t[0, 4:6] >= 0).all() and (t[1, 3:5] >= 0).all()     # the protected tails stay
    assert r.free_blocks() == 6 and resident(t) == 4
    assert r.reclaim(3).size == 0                                   # nothing left to release


def test_no_residency_start_and_tail_fill():
    page = 8
    r = skv.Residency(n_blocks=8, page=page, max_requests=2, max_pages=32)
    r.add(0, 3 * page)
    r.add(1, 3 * page + 5, host_prefix=False)
    r.remove(1)
    r.add(1, 2 * page + 5, host_prefix=True)            # a partial last page
    t = r.block_table()
    assert (t[1, :2] == -1).all() and t[1, 2] >= 0
    np.testing.assert_array_equal(r.fills(1), [2])
    assert r.pending(1).size == 0                       # a page awaiting its fill is not copied out
    r.append(1, 3)                                      # completes page 2 (still unfilled)
    assert r.pending(1).size == 0
    r.mark_filled(1, [2])
    np.testing.assert_array_equal(r.pending(1), [2])
    assert r.fills(1).size == 0
    r2 = skv.Residency(n_blocks=2, page=page, max_requests=1, max_pages=8)
    r2.add(0, 4 * page, host_prefix=True)               # nothing resident at all
    assert r2.state(0) == skv.RESIDENCY_NONE and r2.free_blocks() == 2
    r2.append(0, 1)                                     # the new token opens a resident page
    assert r2.state(0) == skv.RESIDENCY_MIXED and r2.block_table()[0, 4] >= 0


def test_blocks_are_conserved_over_a_random_sequence():
    rng = np.random.default_rng(3)
    page, nb = 4, 30
    r = skv.Residency(n_blocks=nb, page=page, max_requests=4, max_pages=64, tail_pages=1)
    n_tok = [0, 0, 0, 0]
    for b in range(4):
        r.add(b, 0)
    for step in range(400):
        b = int(rng.integers(0, 4))
        try:
            r.append(b, 1)
            n_tok[b] += 1
        except SkvError:
            pass
        if step % 7 == 0:
            for q in range(4):
                r.mark_copied(q, r.pending(q))
        t = r.block_table()
        used = t[t >= 0]
        assert len(set(used.tolist())) == used.size             # a block has one owner
        assert used.size + r.free_blocks() == nb
        for q in range(4):
            n_pages = -(-n_tok[q] // page)
            if n_pages:
                assert t[q, n_pages - 1] >= 0                     # the newest page stays resident
            assert (t[q, n_pages:] == -1).all()


def test_argument_errors():
    with pytest.raises(SkvError):
        skv.Residency(n_blocks=4, page=0, max_requests=1, max_pages=4)
    r = skv.Residency(n_blocks=4, page=4, max_requests=1, max_pages=4)
    with pytest.raises(SkvError):
        r.add(1, 0)                                     # no such slot
    r.add(0, 4)
    with pytest.raises(SkvError):
        r.add(0, 4)                                     # slot in use
    with pytest.raises(SkvError):
        r.append(0, 100)                                # past max_pages


def test_hot_buffers_are_leased_from_the_pool():
    page = 4
    r = skv.Residency(n_blocks=12, page=page, max_requests=2, max_pages=16, tail_pages=1)
    r.add(0, 8 * page)                                  # 8 blocks
    hb0 = r.lease_hot(0, 2)                             # 2 more: 10 used, 2 free
    assert r.free_blocks() == 2 and len(set(hb0.tolist()) | set(r.block_table()[0, :8].tolist())) == 10
    with pytest.raises(SkvError):
        r.lease_hot(0, 1)                               # one lease per request
    r.add(1, 0)
    with pytest.raises(SkvError):
        r.lease_hot(1, 3)                               # 2 free and nothing copied: cannot lease 3
    assert r.free_blocks() == 2                         # a failed lease takes nothing
    r.mark_copied(0, r.pending(0))
    hb1 = r.lease_hot(1, 3)                             # request 0 gives its oldest copied page
    t = r.block_table()
    assert t[0, 0] == -1 and r.free_blocks() == 0
    assert not (set(hb1.tolist()) & set(hb0.tolist())) and not (set(hb1.tolist()) & set(t[t >= 0].tolist()))
    r.remove(0)                                         # its pages and its hot blocks return
    assert r.free_blocks() == 7 + 2
