"""Property tests (Hypothesis) on the CPU: random shapes, tie-heavy keys and
random operation sequences, each checked against a definition written out in
the test rather than against the code under test.

* top-k ("8 agents x 250K context on two 3090s ...", *What shipped*: the top
  2048 by a deterministic select, unioned with 64 sinks and the last 1024
  tokens; "3.14M Context on 3x 3090 ...", *Why*: pooled blocks expand to
  their 4 tokens once the context exceeds 4 * block_topk + 3): the oracle's
  selection equals a brute-force sort by (key descending, index ascending);
* int4 sketch scores: the oracle's integer score equals a numpy dot of the
  unpacked two's-complement codes with the int8 query;
* the residency manager ("vLLM's Hybrid HiSparse ...", *Three residency
  states, one block pool*): under any sequence of adds, appends, copies,
  reclaims and removals, blocks are conserved and owned once, the newest page
  stays resident, and only pages with a host copy become placeholders.
"""
import numpy as np
import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

import skvtest as T  # noqa: E402

SETTINGS = settings(max_examples=60, deadline=None)


def brute_topk(keys, T_len, k, S, W, ratio):
    """The selection rule, written out: dense when short, else the k best
    candidates by (key desc, index asc) -- tokens in [S, T-W) or complete
    blocks -- in ascending order, with sinks / tail / the incomplete block."""
    if ratio == 1:
        if T_len <= S + W + k:
            return list(range(T_len))
        cand = sorted(range(S, T_len - W), key=lambda t: (-int(keys[t]), t))[:k]
        return list(range(S)) + sorted(cand) + list(range(T_len - W, T_len))
    if T_len <= ratio * k + ratio - 1:
        return list(range(T_len))
    nb = T_len // ratio
    blocks = sorted(sorted(range(nb), key=lambda b: (-int(keys[b]), b))[:k])
    out = [ratio * b + u for b in blocks for u in range(ratio)]
    return out + list(range(nb * ratio, T_len))


@SETTINGS
@given(st.data())
def test_oracle_topk_equals_brute_force(orc, data):
    ratio = data.draw(st.sampled_from([1, 4]))
    k = data.draw(st.integers(1, 24))
    S, W = (0, 0) if ratio > 1 else (data.draw(st.integers(0, 6)), data.draw(st.integers(0, 9)))
    B = data.draw(st.integers(1, 3))
    lengths = np.array([data.draw(st.integers(0, 200)) for _ in range(B)], np.int32)
    n_cap = max(1, int(lengths.max()) // ratio + 1)
    alphabet = data.draw(st.sampled_from([2, 5, 2 ** 32]))
    seed = data.draw(st.integers(0, 2 ** 31 - 1))
    rng = np.random.default_rng(seed)
    keys = rng.integers(0, alphabet, (B, n_cap), dtype=np.uint64).astype(np.uint32)
    idx, cnt = orc.topk_select(keys, lengths, k, S=S, W=W, ratio=ratio)
    for b in range(B):
        want = brute_topk(keys[b], int(lengths[b]), k, S, W, ratio)
        assert int(cnt[b]) == len(want)
        assert idx[b, :cnt[b]].tolist() == want


@SETTINGS
@given(st.integers(1, 3), st.sampled_from([128, 256, 512]), st.integers(1, 90), st.integers(0, 2 ** 31 - 1))
def test_oracle_int4_scores_equal_integer_dots(orc, B, width, n, seed):
    rng = np.random.default_rng(seed)
    q8 = rng.integers(-127, 128, (B, width), dtype=np.int64).astype(np.int8)
    sk = rng.integers(0, 256, (B, n, width // 2), dtype=np.int64).astype(np.uint8)
    L = np.full((B,), n, np.int32)
    sc = orc.index_score(orc.SKETCH_INT4, q8, sk, L)
    codes = T.unpack_int4(sk).astype(np.int64)                       # [B][n][width]
    want = np.einsum("bnw,bw->bn", codes, q8.astype(np.int64))
    np.testing.assert_array_equal(sc["iscore"][:, :n], want)
    # the order key orders like the signed score
    assert np.array_equal(np.argsort(sc["okey"][0, :n], kind="stable"), np.argsort(want[0], kind="stable"))


@SETTINGS
@given(st.lists(st.tuples(st.sampled_from(["append", "copy", "reclaim", "remove", "add"]),
                          st.integers(0, 3), st.integers(1, 40)), min_size=1, max_size=80),
       st.integers(1, 3))
def test_residency_invariants(ops, tail_pages):
    import sparse_kv_long_gb300 as skv
    from sparse_kv_long_gb300 import SkvError, _build
    _build.build()
    page, nb, R, max_pages = 4, 24, 4, 64
    r = skv.Residency(n_blocks=nb, page=page, max_requests=R, max_pages=max_pages, tail_pages=tail_pages)
    live = [False] * R
    n_tok = [0] * R
    tail_res = [False] * R     # after a successful append the newest page must stay resident
    copied = [set() for _ in range(R)]
    for op, b, n in ops:
        before = r.block_table()
        try:
            if op == "add" and not live[b]:
                r.add(b, n, host_prefix=bool(n % 2))
                live[b], n_tok[b], copied[b], tail_res[b] = True, n, set(), False
            elif op == "append" and live[b]:
                r.append(b, n)
                n_tok[b] += n
                tail_res[b] = True
            elif op == "copy" and live[b]:
                p = r.pending(b)
                r.mark_copied(b, p)
                copied[b] |= set(p.tolist())
                r.mark_filled(b, r.fills(b))
            elif op == "reclaim":
                r.reclaim(n)
            elif op == "remove" and live[b]:
                r.remove(b)
                live[b], n_tok[b], tail_res[b] = False, 0, False
        except SkvError:
            if op == "append":      # the pool ran dry part-way: the token count is no longer known here
                return
        t = r.block_table()
        used = t[t >= 0]
        assert len(set(used.tolist())) == used.size              # a block has one owner
        assert used.size + r.free_blocks() == nb                 # and none is lost
        for q in range(R):
            if not live[q]:
                assert (t[q] == -1).all()
                continue
            if op != "remove":
                for p in np.nonzero((before[q] >= 0) & (t[q] < 0))[0]:
                    assert p in copied[q]                        # only pages with a host copy are given up
            if tail_res[q]:
                assert t[q, (n_tok[q] - 1) // page] >= 0         # the newest page stays resident
            assert (t[q, -(-n_tok[q] // page):] == -1).all()     # nothing past the last token
