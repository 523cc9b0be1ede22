"""One workspace, zero-filled once, serving selections of different batch
sizes in turn.

The top-k and the fused score + select keep each request's scratch (digit
histograms, tickets, barrier counters, per-chunk records) at a fixed stride
whatever the batch size, and every call returns the words that must start at
zero to zero.  So a workspace sized for the largest batch serves any smaller
or larger call up to that size, in any order: here B = 4, then 8, then 3 on
one buffer, each selection bit-exact against the oracle.
"""
import numpy as np
import pytest
import torch

import skvtest as T

pytestmark = pytest.mark.gpu

B_MAX = 8


@pytest.fixture(scope="module")
def skv():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from sparse_kv_long_gb300 import _build
    _build.build()
    import sparse_kv_long_gb300 as m
    return m


def _check(got_idx, got_cnt, ref_idx, ref_cnt):
    assert np.array_equal(got_cnt, ref_cnt)
    for b in range(len(ref_cnt)):
        assert np.array_equal(got_idx[b, :got_cnt[b]], ref_idx[b, :ref_cnt[b]])


def test_topk_workspace_serves_growing_and_shrinking_batches(skv, orc):
    rng = np.random.default_rng(515)
    k, S, W = 700, 16, 64
    ws = torch.zeros((skv.topk_workspace_size(B_MAX),), dtype=torch.uint8, device="cuda")
    for B in (4, 8, 3):
        L = rng.integers(900, 60_000, B).astype(np.int32)
        n_cap = int(L.max())
        okey = rng.integers(0, 2 ** 32, (B, n_cap), dtype=np.uint64).astype(np.uint32)
        okey[:, ::53] = okey[:, 7:8]  # exact ties among large keys
        idx = torch.full((B, S + k + W), -7, dtype=torch.int32, device="cuda")
        cnt = torch.zeros((B,), dtype=torch.int32, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        skv.topk_select(T.dev(okey.view(np.int32)), T.dev(L), k, idx, cnt, ws, S=S, W=W, status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        ri, rc = orc.topk_select(okey, L, k, S=S, W=W)
        _check(T.host(idx), T.host(cnt), ri, rc)


@pytest.mark.parametrize("mode", ["int4", "pooled"])
def test_score_select_workspace_serves_growing_and_shrinking_batches(skv, orc, mode):
    rng = np.random.default_rng(616 if mode == "int4" else 617)
    ws = torch.zeros((skv.score_select_workspace_size(B_MAX),), dtype=torch.uint8, device="cuda")
    for B in (4, 8, 3):
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        if mode == "int4":
            k, S, W, width = 512, 64, 256, 256
            L = rng.integers(1000, 40_000, B).astype(np.int32)
            n_cap = int(L.max())
            q8 = rng.integers(-127, 128, (B, width)).astype(np.int8)
            sk = rng.integers(0, 256, (B, n_cap, width // 2)).astype(np.uint8)
            idx = torch.full((B, S + k + W), -7, dtype=torch.int32, device="cuda")
            cnt = torch.zeros((B,), dtype=torch.int32, device="cuda")
            skv.score_select(skv.SKETCH_INT4, T.dev(q8), T.dev(sk), T.dev(L), k, idx, cnt, ws, S=S, W=W,
                             status=st)
            ref = orc.index_score(orc.SKETCH_INT4, q8, sk, L, S=S, W=W)
            ri, rc = orc.topk_select(ref["okey"], L, k, S=S, W=W)
            torch.cuda.synchronize()
            assert int(st.item()) == 0
            _check(T.host(idx), T.host(cnt), ri, rc)
        else:
            # Integer-valued bf16 keys and query: every fp32 dot is exact, so
            # the selection is unique and compared bit for bit.
            k, ratio = 128, 4
            nb = rng.integers(600, 9000, B)
            L = (nb * ratio + rng.integers(0, ratio, B)).astype(np.int32)
            n_cap = int(nb.max()) + 1  # room for the incomplete last block
            qi = rng.integers(-3, 4, (B, 128)).astype(np.float32)
            pk = rng.integers(-3, 4, (B, n_cap, 128)).astype(np.float32)
            q_bits = (qi.view(np.uint32) >> 16).astype(np.uint16)
            p_bits = (pk.view(np.uint32) >> 16).astype(np.uint16)
            idx = torch.full((B, ratio * k + ratio - 1), -7, dtype=torch.int32, device="cuda")
            cnt = torch.zeros((B,), dtype=torch.int32, device="cuda")
            skv.score_select(skv.POOLED_BF16, T.bf16_dev(q_bits), T.bf16_dev(p_bits), T.dev(L), k, idx, cnt, ws,
                             ratio=ratio, status=st)
            ref = orc.index_score(orc.POOLED_BF16, q_bits, p_bits, L, ratio=ratio)
            ri, rc = orc.topk_select(ref["okey"], L, k, ratio=ratio)
            torch.cuda.synchronize()
            assert int(st.item()) == 0
            _check(T.host(idx), T.host(cnt), ri, rc)


# Layout of one request's score + select scratch (words): barrier counters
# [0, 2), the range word and the launch counter [2, 4), two 8,192-bin
# histograms, the 256-bin final histogram, then 512 per-CTA records of 260
# words whose high 16 bits carry the launch's tag (launch counter mod 65,535,
# plus one).
_REQ_WORDS = 4 + 2 * 8192 + 256 + 512 * 260
_EPOCH, _FIN, _FIN_WORDS, _SLOTS = 3, 4 + 2 * 8192 + 256, 260, 512


def test_score_select_launch_counter_wrap(skv, orc):
    """Across the wrap of the records' tag: the launch counter is preset to
    the last launch of a tag cycle and every record slot holds a stale record
    carrying the next cycle's first tag.  The launch at the end of the cycle
    clears the request's records, so the next launch (whose tag equals the
    stale one) reads only its own; both selections equal the oracle's."""
    rng = np.random.default_rng(77)
    B, Tn, k, S, W, width = 4, 30_000, 500, 16, 64, 256
    q8 = rng.integers(-127, 128, (B, width), dtype=np.int8)
    sk = rng.integers(0, 256, (B, Tn, width // 2), dtype=np.uint8)
    L = np.full((B,), Tn, np.int32)
    sc = orc.index_score(orc.SKETCH_INT4, q8, sk, L, S=S, W=W)
    ridx, rcnt = orc.topk_select(sc["okey"], L, k, S=S, W=W)
    ws = torch.zeros((skv.score_select_workspace_size(B),), dtype=torch.uint8, device="cuda")
    w32 = ws.view(torch.int32)
    assert w32.numel() >= B * _REQ_WORDS
    for b in range(B):
        base = b * _REQ_WORDS
        w32[base + _EPOCH] = 65533                    # the next launch has the cycle's last tag
        stale = (1 << 16) | 0x1234                    # the first tag of the next cycle, a bogus count
        w32[base + _FIN: base + _FIN + _SLOTS * _FIN_WORDS] = stale
    idx = torch.zeros((B, S + k + W), dtype=torch.int32, device="cuda")
    cnt = torch.zeros((B,), dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    q8d, skd, Ld = T.dev(q8), T.dev(sk), T.dev(L)
    for launch in range(3):
        idx.zero_()
        cnt.zero_()
        skv.score_select(skv.SKETCH_INT4, q8d, skd, Ld, k, idx, cnt, ws, S=S, W=W, status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0, (launch, int(st.item()))
        _check(T.host(idx), T.host(cnt), ridx, rcnt)
    assert int(w32[_EPOCH].item()) == 65536
