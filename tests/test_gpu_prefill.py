"""Chunked sparse prefill against the oracle.

"3.14M Context on 3x 3090 ...", *The Downside to Keep in Mind*: every token of
a prefill chunk picks its own top blocks from the pooled indexer (causally:
query at position p sees the blocks complete within its first p + 1 tokens),
and the attention runs with the loops swapped -- the history staged into a
small working buffer chunk by chunk, partial softmax states merged.  The
swap changes only the order of the work, so each query's output must equal
the plain sparse attention over its own selected rows:

* scores: every order key decodes to the oracle's fp32 dot within the fp32
  rounding bound of a 128-term sum;
* selection (scores + skv_topk_select): counts equal, block sets differ only
  where the oracle's score is within 1e-3 relative of the k-th, the
  incomplete last block and the dense fallback as in decode;
* attention: every output within 2e-3 of the fp64 oracle on the same rows,
  for several working-buffer sizes (one chunk, ragged chunks, chunks smaller
  than a query's run of picks), K/V in device or registered host memory.
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


def okey_to_f32(k: np.ndarray) -> np.ndarray:
    """Inverse of the fp32 order-key map (positive: sign bit set; negative: inverted)."""
    k = k.astype(np.uint32)
    u = np.where(k & 0x80000000, k & 0x7FFFFFFF, ~k).astype(np.uint32)
    return u.view(np.float32)


def _pooled_case(seed, nq, n_blocks):
    rng = np.random.default_rng(seed)
    q = wl.to_bf16_bits(rng.standard_normal((nq, 128)).astype(np.float32))
    P = wl.to_bf16_bits(rng.standard_normal((n_blocks, 128)).astype(np.float32))
    return q, P


@pytest.mark.parametrize("nq,n_blocks", [(1, 1), (150, 1000), (64, 2100), (70, 4096 + 3)])
def test_prefill_scores_match_oracle_dots(skv, orc, nq, n_blocks):
    q, P = _pooled_case(11 + nq, nq, n_blocks)
    stride = n_blocks + (n_blocks & 1)
    keys = torch.zeros((nq, stride), dtype=torch.int32, device="cuda")
    keys.fill_(-1)                                   # sentinel 0xFFFFFFFF beyond n_blocks
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    skv.prefill_index_scores(T.bf16_dev(q), T.bf16_dev(P), keys, n_blocks=n_blocks, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    got_k = T.host(keys).view(np.uint32)
    assert (got_k[:, n_blocks:] == 0xFFFFFFFF).all()
    got = okey_to_f32(got_k[:, :n_blocks]).astype(np.float64)
    qf, Pf = wl.bf16_bits_to_f32(q).astype(np.float64), wl.bf16_bits_to_f32(P).astype(np.float64)
    exact = qf @ Pf.T
    # fp32 accumulation of exact bf16 products: a few units of 128 * 2^-24 of
    # sum |q_x k_x| (tensor-core accumulation need not round to nearest)
    bound = 8 * 128 * 2.0 ** -24 * (np.abs(qf) @ np.abs(Pf).T) + 1e-30
    assert np.all(np.abs(got - exact) <= bound)
    # the oracle's own fp32 dots (fixed order) lie in the same band
    sc = orc.index_score(orc.POOLED_BF16, q[:1], P[None], np.array([4 * n_blocks], np.int32), ratio=4)
    assert np.all(np.abs(sc["fscore"][0, :n_blocks] - exact[0]) <= bound[0])


def _select_gpu(skv, keys, L, k, max_rows):
    nq = keys.shape[0]
    idx = torch.zeros((nq, max_rows), dtype=torch.int32, device="cuda")
    cnt = torch.zeros((nq,), dtype=torch.int32, device="cuda")
    ws = torch.zeros((skv.topk_workspace_size(nq),), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    skv.topk_select(keys.view(torch.int32), T.dev(L), k, idx, cnt, ws, ratio=4, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return idx, cnt


def test_prefill_selection_causal(skv, orc):
    """Queries at positions spread over [0, 9000): early ones fall back to
    dense, the rest select 64 of their complete blocks plus the incomplete
    block's tokens; sets within the 1e-3 band of the oracle's k-th score."""
    k, nq, n_tok = 64, 96, 9000
    rng = np.random.default_rng(5)
    pos = np.sort(rng.choice(n_tok, size=nq, replace=False)).astype(np.int32)
    pos[:3] = [0, 4 * k + 2, 4 * k + 3]             # dense, dense at the edge, first sparse
    pos.sort()
    L = pos + 1
    n_blocks = n_tok // 4
    q, P = _pooled_case(7, nq, n_blocks)
    keys = torch.zeros((nq, n_blocks), dtype=torch.int32, device="cuda")
    skv.prefill_index_scores(T.bf16_dev(q), T.bf16_dev(P), keys)
    max_rows = 4 * k + 3
    idx, cnt = _select_gpu(skv, keys, L, k, max_rows)
    gidx, gcnt = T.host(idx), T.host(cnt)
    for i in range(nq):
        Li = int(L[i])
        sc = orc.index_score(orc.POOLED_BF16, q[i:i + 1], P[None], np.array([Li], np.int32), ratio=4)
        ridx, rcnt = orc.topk_select(sc["okey"], np.array([Li], np.int32), k, ratio=4, max_rows=max_rows)
        assert gcnt[i] == rcnt[0], i
        n = int(gcnt[i])
        if Li <= 4 * k + 3:                         # dense
            np.testing.assert_array_equal(gidx[i, :n], np.arange(Li))
            continue
        nb = Li // 4
        kth = np.sort(sc["fscore"][0, :nb])[::-1][k - 1]
        gb, rb = set((gidx[i, :4 * k:4] // 4).tolist()), set((ridx[0, :4 * k:4] // 4).tolist())
        for blk in gb ^ rb:
            assert abs(sc["fscore"][0, blk] - kth) <= 1e-3 * abs(kth), (i, blk)
        np.testing.assert_array_equal(gidx[i, 4 * k:n], np.arange(4 * nb, Li))
        assert np.all(np.diff(gidx[i, :n]) > 0)


def _attend_case(seed, nq, Hq, Hkv, d, n_tok, max_rows):
    rng = np.random.default_rng(seed)
    K = wl.to_bf16_bits(rng.standard_normal((n_tok, Hkv, d)).astype(np.float32))
    V = wl.to_bf16_bits(rng.standard_normal((n_tok, Hkv, d)).astype(np.float32))
    q = wl.to_bf16_bits(rng.standard_normal((nq, Hq, d)).astype(np.float32))
    idx = np.zeros((nq, max_rows), np.int32)
    cnt = np.zeros((nq,), np.int32)
    for i in range(nq):
        if i == 1:
            continue                                 # a query with no rows
        n = int(rng.integers(1, max_rows + 1)) if i != 2 else max_rows
        hi = n_tok if i != 3 else min(n_tok, 2 * max_rows)   # one query clustered at the start
        rows = np.sort(rng.choice(hi, size=min(n, hi), replace=False)).astype(np.int32)
        idx[i, :rows.size] = rows
        cnt[i] = rows.size
    return K, V, q, idx, cnt


@pytest.mark.parametrize("chunk", [1000, 4096, 8192, 37])
@pytest.mark.parametrize("where", ["device", "host"])
@pytest.mark.parametrize("Hq,Hkv", [(16, 2), (6, 1), (16, 1)], ids=["G8", "G6", "G16"])
def test_prefill_attend_loop_swapped(skv, orc, chunk, where, Hq, Hkv):
    """G <= 8 runs the tensor-core chunk kernel (G = 6 with padded heads),
    G = 16 the CUDA-core one."""
    nq, d, n_tok, max_rows = 29, 256, 5000, 700
    K, V, q, idx, cnt = _attend_case(3 + chunk, nq, Hq, Hkv, d, n_tok, max_rows)
    scale = 1 / math.sqrt(d)
    kst = torch.zeros((chunk, Hkv, d), dtype=torch.bfloat16, device="cuda")
    vst = torch.zeros_like(kst)
    state = torch.zeros((nq, Hq, d + 4), dtype=torch.float32, device="cuda")
    out = torch.full((nq, Hq, d), 7.0, dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    mm = None
    if where == "device":
        ks, vs = T.bf16_dev(K), T.bf16_dev(V)
        srcs = (ks, vs)
    else:
        mm = mmap.mmap(-1, K.nbytes + V.nbytes)
        harr = np.frombuffer(mm, dtype=np.uint8, count=K.nbytes + V.nbytes)
        harr[:K.nbytes] = K.view(np.uint8).reshape(-1)
        harr[K.nbytes:] = V.view(np.uint8).reshape(-1)
        skv.host_register(harr.ctypes.data, harr.nbytes)
        srcs = (harr.ctypes.data, harr.ctypes.data + K.nbytes)
    try:
        skv.prefill_attend(T.bf16_dev(q), srcs[0], srcs[1], n_tok, kst, vst, T.dev(idx), T.dev(cnt), scale,
                           state, out, Hkv, status=st)
        torch.cuda.synchronize()
    finally:
        if mm is not None:
            skv.host_unregister(harr.ctypes.data)
            del harr
            mm.close()
    assert int(st.item()) == 0
    ref = orc.attend(orc.KV_BF16, q, K.reshape(n_tok, -1), V.reshape(n_tok, -1), idx, cnt, scale, Hkv, d, d)
    got = T.host(out)
    assert np.all(got[1] == 0.0)                     # no rows: zeros
    err = np.max(np.abs(got - ref))
    assert err < 2e-3, err


def test_prefill_attend_flags_rows_past_the_history(skv):
    """A pick at or past n_tokens sets SKV_DEV_RANGE and is left out; the other
    rows still count (and nothing outside the staged chunks is read)."""
    nq, Hq, Hkv, d, n_tok = 2, 8, 1, 256, 300
    rng = np.random.default_rng(9)
    K = torch.from_numpy(rng.standard_normal((n_tok, Hkv, d)).astype(np.float32)).to(torch.bfloat16).cuda()
    V = torch.ones_like(K)
    q = torch.zeros((nq, Hq, d), dtype=torch.bfloat16, device="cuda")
    idx = torch.tensor([[5, 17, 299, 300], [0, 1, 2, 3]], dtype=torch.int32, device="cuda")
    cnt = torch.tensor([4, 4], dtype=torch.int32, device="cuda")
    kst = torch.zeros((128, Hkv, d), dtype=torch.bfloat16, device="cuda")
    vst = torch.zeros_like(kst)
    state = torch.zeros((nq, Hq, d + 4), dtype=torch.float32, device="cuda")
    out = torch.zeros((nq, Hq, d), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    skv.prefill_attend(q, K, V, n_tok, kst, vst, idx, cnt, 0.0625, state, out, Hkv, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & skv.DEV_RANGE
    # q = 0: uniform weights over the valid rows, V = 1 -> outputs of 1
    np.testing.assert_allclose(T.host(out), 1.0, atol=1e-6)
