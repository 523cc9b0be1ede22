"""Pins for the CPU oracle: each test fixes part of the oracle against something
other than the oracle itself -- a library routine, a closed form, a brute-force
enumeration, a hand-worked example, or a number printed on the pages.

Page titles cited:
  [P1] 8 agents x 250K context on two 3090s: sparse KV decode with a rank-64
       key sketch and a host-RAM tier
  [P2] vLLM's Hybrid HiSparse Triples Concurrent Requests on Million-Token Contexts
  [P3] You can offload most of Qwen3.8-Flash-Next's KV cache to RAM ...
  [P4] 3.14M Context on 3x 3090: The Power of an Architecture That Puts KV Cache in Host RAM
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_numbers.json")


def golden():
    with open(GOLDEN) as f:
        return json.load(f)


# ---------------------------------------------------------------------------
# Number formats (library routines: numpy float16, torch bfloat16 / float8)
# ---------------------------------------------------------------------------

def test_f16_decode_all_codes(orc):
    codes = np.arange(65536, dtype=np.uint16)
    ref = codes.view(np.float16).astype(np.float64)
    got = orc.f16_to_f64(codes)
    fin = np.isfinite(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(np.isinf(got), np.isinf(ref))


def test_f32_to_f16_rounding(orc):
    rng = np.random.default_rng(0)
    vals = np.concatenate([
        rng.standard_normal(2000).astype(np.float32) * 10,
        rng.standard_normal(500).astype(np.float32) * 1e-5,      # subnormal range
        np.array([65504, 65519.99, 65520, 70000, -65520, 2.0 ** -24, 2.0 ** -25,
                  3 * 2.0 ** -26, 1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11, 0.0, -0.0,
                  6.1e-5, 1e-8], np.float32),
    ])
    with np.errstate(over="ignore"):                             # 65520 and beyond round to inf
        ref = vals.astype(np.float16).view(np.uint16)
    got = orc.f32_to_f16(vals)
    assert np.array_equal(got, ref)


def test_bf16_roundtrip(orc):
    rng = np.random.default_rng(1)
    vals = np.concatenate([rng.standard_normal(3000).astype(np.float32) * 3,
                           np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -0.0, 3e38, 1e-40],
                                    np.float32)])
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(orc.f32_to_bf16(vals), ref)
    back = torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16).float().numpy()
    assert np.array_equal(orc.bf16_to_f32(ref), back)


def test_fp8_e4m3_all_codes(orc):
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = orc.fp8_e4m3_to_f64(codes)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    fin = ~np.isnan(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.nanmax(got) == 448.0  # OCP E4M3 largest finite value


def test_order_keys_preserve_order(orc):
    rng = np.random.default_rng(2)
    ints = np.sort(np.concatenate([rng.integers(-2**31, 2**31 - 1, 500), [-2**31, -1, 0, 1, 2**31 - 1]]))
    k = orc.order_key_i32(ints.astype(np.int32))
    assert np.all(np.diff(k.astype(np.int64)) >= 0)
    fl = np.sort(np.concatenate([rng.standard_normal(500) * 1e3, [-np.inf, np.inf, 1e-45, -1e-45]]).astype(np.float32))
    kf = orc.order_key_f32(fl)
    assert np.all(np.diff(kf.astype(np.int64)) >= 0)
    assert orc.order_key_f32(np.float32(-0.0))[0] == orc.order_key_f32(np.float32(0.0))[0]


# ---------------------------------------------------------------------------
# a1 sketch projection
# ---------------------------------------------------------------------------

def test_sketch_identity_basis_is_exact(orc):
    """With P = I (r = d) the sketch of a key is the key itself."""
    rng = np.random.default_rng(3)
    d = 64
    keys = wl.to_bf16_bits(rng.standard_normal((5, 2, d)).astype(np.float32))
    out = orc.sketch_project(keys, np.eye(d, dtype=np.float32))
    assert np.array_equal(out["s"], wl.bf16_bits_to_f32(keys))


def test_sketch_matches_library_matmul(orc):
    rng = np.random.default_rng(4)
    n, Hkv, d, r = 7, 3, 256, 64
    keys = wl.to_bf16_bits(rng.standard_normal((n, Hkv, d)).astype(np.float32))
    P = wl.orthonormal_basis(d, r, 5)
    s = orc.sketch_project(keys, P)["s"]
    kf = wl.bf16_bits_to_f32(keys).astype(np.float64)
    ref = np.einsum("thi,ij->thj", kf, P.astype(np.float64))
    bound = d * 2.0 ** -23 * np.einsum("thi,ij->thj", np.abs(kf), np.abs(P.astype(np.float64)))
    assert np.all(np.abs(s - ref) <= bound)


def test_sketch_int4_codes_hand_worked(orc):
    """Hand-worked codes: round half to even, clamp to [-8, 7], two's-complement
    nibbles, dim 2b in the low nibble ([P1] 'What shipped': the sketch is int4)."""
    d = r = 16
    vals = np.array([0.5, 1.5, 2.5, -0.5, -1.5, -2.5, 7.5, -8.5,
                     100.0, -100.0, 3.25, -3.75, 0.0, 6.5, -7.5, 1.0], np.float32)
    expected_codes = [0, 2, 2, 0, -2, -2, 7, -8, 7, -8, 3, -4, 0, 6, -8, 1]
    keys = wl.to_bf16_bits(vals.reshape(1, 1, d))
    assert np.array_equal(wl.bf16_bits_to_f32(keys).ravel(), vals)  # all exact in bf16
    out = orc.sketch_project(keys, np.eye(d, dtype=np.float32), c=np.ones((1, r), np.float32))
    expected_bytes = [((expected_codes[2 * b] & 15) | ((expected_codes[2 * b + 1] & 15) << 4))
                      for b in range(d // 2)]
    assert list(out["q4"][0]) == expected_bytes


def test_sketch_int4_roundtrip_within_half_step(orc):
    rng = np.random.default_rng(6)
    n, Hkv, d, r = 50, 2, 256, 64
    P = wl.orthonormal_basis(d, r, 7)
    keys = wl.to_bf16_bits(rng.standard_normal((n, Hkv, d)).astype(np.float32))
    c = np.full((Hkv, r), 0.6, np.float32)
    out = orc.sketch_project(keys, P, c)
    q4 = out["q4"].reshape(n, Hkv, r // 2)
    lo = (q4 & 15).astype(np.int64)
    hi = (q4 >> 4).astype(np.int64)
    codes = np.stack([lo, hi], axis=-1).reshape(n, Hkv, r)
    codes = np.where(codes >= 8, codes - 16, codes)
    s = out["s"]
    inside = np.abs(s / 0.6) <= 7.49
    assert np.all(np.abs(codes * 0.6 - s)[inside] <= 0.3 + 1e-6)
    assert np.all(codes[s / 0.6 > 7.5] == 7) and np.all(codes[s / 0.6 < -8.5] == -8)


# ---------------------------------------------------------------------------
# a2 sketch query
# ---------------------------------------------------------------------------

def test_sketch_query_group_sum_closed_form(orc):
    """P = I, c = 1: the folded query of KV head h is the sum of its group's
    query heads (contiguous groups, kv_head = g / G)."""
    rng = np.random.default_rng(8)
    B, Hq, Hkv, d = 2, 6, 2, 32
    q = wl.to_bf16_bits(rng.standard_normal((B, Hq, d)).astype(np.float32))
    out = orc.sketch_query(q, Hkv, np.eye(d, dtype=np.float32), c=np.ones((Hkv, d), np.float32))
    qf = wl.bf16_bits_to_f32(q).astype(np.float64)
    ref = qf.reshape(B, Hkv, Hq // Hkv, d).sum(axis=2).reshape(B, Hkv * d)
    assert np.allclose(out["qp"], ref, rtol=1e-6, atol=1e-6)


def test_sketch_query_int8_hand_worked(orc):
    """sigma = max|qp| / 127; q8 = rint(qp / sigma), half to even."""
    d = 8
    vals = np.array([127.0, 63.5, 62.5, -0.5, 2.5, -127.0, 1.5, 0.0], np.float32)
    q = wl.to_bf16_bits(vals.reshape(1, 1, d))
    out = orc.sketch_query(q, 1, np.eye(d, dtype=np.float32), c=np.ones((1, d), np.float32))
    assert out["sigma"][0] == np.float32(1.0)
    assert list(out["q8"][0]) == [127, 64, 62, 0, 2, -127, 2, 0]


def test_sketch_query_scale_folding(orc):
    """Multiplying c by 2 doubles qp and leaves q8 unchanged (sigma doubles)."""
    rng = np.random.default_rng(9)
    d, r, Hkv, Hq = 256, 64, 4, 8
    P = wl.orthonormal_basis(d, r, 10)
    q = wl.to_bf16_bits(rng.standard_normal((1, Hq, d)).astype(np.float32))
    c = rng.uniform(0.1, 1.0, (Hkv, r)).astype(np.float32)
    a = orc.sketch_query(q, Hkv, P, c)
    b = orc.sketch_query(q, Hkv, P, 2 * c)
    assert np.array_equal(2 * a["qp"], b["qp"])
    assert np.array_equal(a["q8"], b["q8"])


# ---------------------------------------------------------------------------
# a2' pooled keys
# ---------------------------------------------------------------------------

def test_pool_keys_is_bf16_mean(orc):
    """Mean of 4 bf16 tokens, rounded to bf16 (library rounding)."""
    rng = np.random.default_rng(11)
    x = wl.to_bf16_bits(rng.standard_normal((4 * 37, 128)).astype(np.float32))
    got = orc.pool_keys(x, 4)
    xf = wl.bf16_bits_to_f32(x).astype(np.float64).reshape(37, 4, 128)
    ref = wl.to_bf16_bits(xf.mean(axis=1).astype(np.float32))
    assert np.array_equal(got, ref)


def test_pool_keys_constant_block(orc):
    rng = np.random.default_rng(12)
    one = wl.to_bf16_bits(rng.standard_normal((1, 128)).astype(np.float32))
    x = np.repeat(one, 4, axis=0)
    assert np.array_equal(orc.pool_keys(x, 4), one)


# ---------------------------------------------------------------------------
# a3 index scores
# ---------------------------------------------------------------------------

def test_int4_score_equals_integer_dot_of_construction(orc):
    """Keys built on the integer grid (k = n * c, P = I) and a query whose
    scale sigma is exactly 1: the int4 score is the textbook integer dot product
    of the constructed integer vectors, summed over KV heads and group heads."""
    rng = np.random.default_rng(13)
    B, Hkv, G, d = 2, 2, 2, 16
    Hq = Hkv * G
    T = 40
    n = rng.integers(-8, 8, (B, T, Hkv, d))
    m = rng.integers(-31, 32, (B, Hq, d))
    m[:, 0, 0] = 63
    m[:, 1, 0] = 64  # group sum at (h=0, j=0) = 127 -> sigma = 1 exactly
    keys = wl.to_bf16_bits(n.astype(np.float32))
    q = wl.to_bf16_bits(m.astype(np.float32))
    P = np.eye(d, dtype=np.float32)
    c = np.ones((Hkv, d), np.float32)
    sk = orc.sketch_project(keys.reshape(B * T, Hkv, d), P, c)["q4"].reshape(B, T, Hkv * d // 2)
    qq = orc.sketch_query(q, Hkv, P, c)
    assert np.all(qq["sigma"] == 1.0)
    lengths = np.full((B,), T, np.int32)
    res = orc.index_score(orc.SKETCH_INT4, qq["q8"], sk, lengths)
    msum = m.reshape(B, Hkv, G, d).sum(axis=2)
    ref = np.einsum("bhj,bthj->bt", msum, n)
    assert np.array_equal(res["iscore"], ref.astype(np.int32))


def test_f32_score_identity_basis_is_exact_attention_score(orc):
    """r = d, P = I: the sketch score of token t is sum_h sum_{g in G(h)} q_g . k_{t,h}
    (the exact dot products of 'exact top-k attention')."""
    rng = np.random.default_rng(14)
    B, Hkv, G, d, T = 1, 2, 3, 64, 50
    Hq = Hkv * G
    keys = wl.to_bf16_bits(rng.standard_normal((B, T, Hkv, d)).astype(np.float32))
    q = wl.to_bf16_bits(rng.standard_normal((B, Hq, d)).astype(np.float32))
    P = np.eye(d, dtype=np.float32)
    s = orc.sketch_project(keys.reshape(B * T, Hkv, d), P)["s"].reshape(B, T, Hkv * d)
    qp = orc.sketch_query(q, Hkv, P, None, int8=False)["qp"]
    res = orc.index_score(orc.SKETCH_F32, qp, s, np.array([T], np.int32))
    kf = wl.bf16_bits_to_f32(keys).astype(np.float64)
    qf = wl.bf16_bits_to_f32(q).astype(np.float64)
    ref = np.zeros((B, T))
    for g in range(Hq):
        ref += np.einsum("d,btd->bt", qf[0, g], kf[:, :, g // G, :])
    assert np.allclose(res["fscore"], ref, rtol=1e-5, atol=1e-4)


def test_pooled_score_matches_library_dot(orc):
    rng = np.random.default_rng(15)
    B, nb, D = 2, 33, 128
    pooled = wl.to_bf16_bits(rng.standard_normal((B, nb, D)).astype(np.float32))
    qi = wl.to_bf16_bits(rng.standard_normal((B, D)).astype(np.float32))
    lengths = np.array([4 * nb, 4 * nb - 5], np.int32)
    res = orc.index_score(orc.POOLED_BF16, qi, pooled, lengths, ratio=4)
    ref = np.einsum("bd,bnd->bn", wl.bf16_bits_to_f32(qi).astype(np.float64),
                    wl.bf16_bits_to_f32(pooled).astype(np.float64))
    assert np.allclose(res["fscore"][0], ref[0], rtol=1e-5, atol=1e-4)
    nb1 = (4 * nb - 5) // 4  # only complete blocks are candidates
    assert np.allclose(res["fscore"][1, :nb1], ref[1, :nb1], rtol=1e-5, atol=1e-4)
    assert np.all(res["okey"][1, nb1:] == 0)


def test_sketch_candidates_exclude_sinks_and_tail(orc):
    rng = np.random.default_rng(16)
    T, S, W = 100, 8, 16
    q8 = rng.integers(-127, 128, (1, 32)).astype(np.int8)
    sk = rng.integers(0, 256, (1, T, 16)).astype(np.uint8)
    res = orc.index_score(orc.SKETCH_INT4, q8, sk, np.array([T], np.int32), S=S, W=W)
    assert np.all(res["okey"][0, :S] == 0) and np.all(res["okey"][0, T - W:] == 0)
    assert np.all(res["okey"][0, S:T - W] != 0)


# ---------------------------------------------------------------------------
# a4 selection: brute force and exhaustive ties
# ---------------------------------------------------------------------------

def brute_topk(keys, k):
    """Rank each candidate by counting who beats it (key larger, or equal key
    and lower index); the k with rank < k are selected."""
    n = len(keys)
    sel = []
    for i in range(n):
        beat = sum(1 for j in range(n) if keys[j] > keys[i] or (keys[j] == keys[i] and j < i))
        if beat < k:
            sel.append(i)
    return sel


def test_topk_exhaustive_ties(orc):
    for n in range(1, 7):
        for keys in itertools.product([5, 6, 7], repeat=n):
            for k in range(1, n):
                okey = np.array([keys], np.uint32)
                idx, cnt = orc.topk_select(okey, np.array([n], np.int32), k, max_rows=k)
                assert cnt[0] == k
                assert list(idx[0, :k]) == brute_topk(list(keys), k)


def test_topk_random_vs_brute(orc):
    rng = np.random.default_rng(17)
    for trial in range(30):
        T = int(rng.integers(20, 90))
        S, W, k = int(rng.integers(0, 5)), int(rng.integers(0, 7)), int(rng.integers(1, 9))
        if T <= S + W + k:
            continue
        okey = rng.integers(0, 12, (1, T)).astype(np.uint32)
        idx, cnt = orc.topk_select(okey, np.array([T], np.int32), k, S=S, W=W)
        picks = [S + i for i in brute_topk(list(okey[0, S:T - W]), k)]
        expect = list(range(S)) + picks + list(range(T - W, T))
        assert cnt[0] == S + k + W
        assert list(idx[0, :cnt[0]]) == expect


def test_topk_dense_fallback_boundary(orc):
    S, W, k = 4, 8, 5
    for T, dense in [(S + W + k, True), (S + W + k + 1, False), (1, True), (S, True)]:
        okey = np.arange(T, dtype=np.uint32)[None, :]
        idx, cnt = orc.topk_select(okey, np.array([T], np.int32), k, S=S, W=W)
        if dense:
            assert cnt[0] == T and list(idx[0, :T]) == list(range(T))
        else:
            assert cnt[0] == S + k + W


def test_pooled_threshold_from_page(orc):
    """[P4] 'Why': sparse once the context exceeds 4 * block_topk + 3 = 2051."""
    g = golden()["sparse_threshold_tokens"]
    kb, ratio = g["block_topk"], g["ratio"]
    assert ratio * kb + 3 == g["value"]
    for T, dense in [(g["value"], True), (g["value"] + 1, False)]:
        okey = np.zeros((1, (T + 3) // 4), np.uint32) + 7
        idx, cnt = orc.topk_select(okey, np.array([T], np.int32), kb, ratio=ratio)
        if dense:
            assert cnt[0] == T
        else:
            assert cnt[0] == ratio * kb + T % ratio


def test_pooled_block_expansion(orc):
    T, kb = 4 * 10 + 3, 3
    okey = np.zeros((1, 11), np.uint32)
    okey[0, [2, 7, 9]] = [9, 8, 9]
    okey[0, 5] = 8  # tie with block 7: lower index wins
    idx, cnt = orc.topk_select(okey, np.array([T], np.int32), kb, ratio=4)
    exp = [8, 9, 10, 11, 20, 21, 22, 23, 36, 37, 38, 39, 40, 41, 42]
    assert cnt[0] == len(exp) and list(idx[0, :cnt[0]]) == exp


def test_planted_recall_tiny(orc):
    """Every planted token of the tiny workload is selected (the pages report
    31/32 on real documents, [P1] 'Measured results')."""
    w = wl.TINY
    x = wl.tiny_inputs(w)
    B, T = w.B, w.T
    s = orc.sketch_project(x["K"].reshape(B * T, w.Hkv, w.d), x["basis"])["s"].reshape(B, T, w.Hkv * w.r)
    qp = orc.sketch_query(x["q"], w.Hkv, x["basis"], None, int8=False)["qp"]
    res = orc.index_score(orc.SKETCH_F32, qp, s, x["lengths"], S=w.S, W=w.W)
    idx, cnt = orc.topk_select(res["okey"], x["lengths"], w.k, S=w.S, W=w.W)
    sel = set(idx[0, :cnt[0]].tolist())
    assert all(int(t) in sel for t in x["planted"][0])


# ---------------------------------------------------------------------------
# a6 attention
# ---------------------------------------------------------------------------

def dense_attention_ref(q, K, V, scale, G):
    """Textbook softmax attention with grouped KV heads (library softmax)."""
    from scipy.special import softmax
    B, Hq, d = q.shape
    out = np.zeros((B, Hq, V.shape[-1]))
    for b in range(B):
        for g in range(Hq):
            logits = scale * K[b, :, g // G, :] @ q[b, g]
            out[b, g] = softmax(logits) @ V[b, :, g // G, :]
    return out


def test_sparse_equals_dense_when_all_rows_selected(orc):
    rng = np.random.default_rng(18)
    B, T, Hq, Hkv, d = 2, 37, 6, 2, 32
    q = wl.to_bf16_bits(rng.standard_normal((B, Hq, d)).astype(np.float32))
    K = wl.to_bf16_bits(rng.standard_normal((B, T, Hkv, d)).astype(np.float32))
    V = wl.to_bf16_bits(rng.standard_normal((B, T, Hkv, d)).astype(np.float32))
    rows = np.tile(np.arange(T, dtype=np.int32), (B, 1))
    rows[1] = rows[1][::-1]  # order of the rows does not matter
    count = np.full((B,), T, np.int32)
    got = orc.attend(orc.KV_BF16, q, K.reshape(B * T, Hkv * d), V.reshape(B * T, Hkv * d), rows,
                     count, 1 / math.sqrt(d), Hkv, d, d, req_row_stride=T)
    ref = dense_attention_ref(wl.bf16_bits_to_f32(q).astype(np.float64),
                              wl.bf16_bits_to_f32(K).astype(np.float64),
                              wl.bf16_bits_to_f32(V).astype(np.float64), 1 / math.sqrt(d), Hq // Hkv)
    assert np.max(np.abs(got - ref)) < 1e-12


def test_single_row_attention_returns_value(orc):
    rng = np.random.default_rng(19)
    Hq, Hkv, d = 4, 2, 16
    q = wl.to_bf16_bits(rng.standard_normal((1, Hq, d)).astype(np.float32))
    K = wl.to_bf16_bits(rng.standard_normal((10, Hkv * d)).astype(np.float32))
    V = wl.to_bf16_bits(rng.standard_normal((10, Hkv * d)).astype(np.float32))
    got = orc.attend(orc.KV_BF16, q, K, V, np.array([[7]], np.int32), np.array([1], np.int32), 0.1, Hkv, d, d)
    vf = wl.bf16_bits_to_f32(V).reshape(10, Hkv, d)
    for g in range(Hq):
        assert np.array_equal(got[0, g], vf[7, g // 2].astype(np.float64))


def test_int8_attention_equals_dequantised_dense(orc):
    rng = np.random.default_rng(20)
    B, T, Hq, Hkv, d = 1, 29, 4, 2, 32
    q = wl.to_bf16_bits(rng.standard_normal((B, Hq, d)).astype(np.float32))
    k8 = rng.integers(-127, 128, (B * T, Hkv, d)).astype(np.int8)
    v8 = rng.integers(-127, 128, (B * T, Hkv, d)).astype(np.int8)
    ks = (rng.uniform(0.001, 0.05, (B * T, Hkv)).astype(np.float16)).view(np.uint16)
    vs = (rng.uniform(0.001, 0.05, (B * T, Hkv)).astype(np.float16)).view(np.uint16)
    rows = np.arange(T, dtype=np.int32)[None, :]
    got = orc.attend(orc.KV_INT8, q, k8.reshape(B * T, -1), v8.reshape(B * T, -1), rows,
                     np.array([T], np.int32), 0.2, Hkv, d, d, k_scale=ks, v_scale=vs)
    Kf = (k8.astype(np.float64) * ks.view(np.float16).astype(np.float64)[..., None]).reshape(B, T, Hkv, d)
    Vf = (v8.astype(np.float64) * vs.view(np.float16).astype(np.float64)[..., None]).reshape(B, T, Hkv, d)
    ref = dense_attention_ref(wl.bf16_bits_to_f32(q).astype(np.float64), Kf, Vf, 0.2, Hq // Hkv)
    assert np.max(np.abs(got - ref)) < 1e-12


def test_fp8_latent_attention(orc):
    """Latent rows: K is the full row (512 + 64), V the first 512 dims, scaled
    by the row scale; decoded values from the OCP E4M3 definition (library)."""
    rng = np.random.default_rng(21)
    T, Hq, d, dv = 9, 3, 576, 512
    q = wl.to_bf16_bits(rng.standard_normal((1, Hq, d)).astype(np.float32))
    lat = rng.integers(0, 256, (T, d)).astype(np.uint8)
    lat[(lat & 0x7f) == 0x7f] = 0x11  # no NaN codes
    rs = rng.uniform(0.5, 2.0, T).astype(np.float32)
    got = orc.attend(orc.KV_FP8, q, lat, lat, np.arange(T, dtype=np.int32)[None], np.array([T], np.int32),
                     1 / math.sqrt(d), 1, d, dv, row_scale=rs, k_pitch=d, v_pitch=d)
    dec = torch.from_numpy(lat).view(torch.float8_e4m3fn).to(torch.float64).numpy() * rs[:, None].astype(np.float64)
    ref = dense_attention_ref(wl.bf16_bits_to_f32(q).astype(np.float64), dec[None, :, None, :],
                              dec[None, :, None, :dv], 1 / math.sqrt(d), Hq)
    assert np.max(np.abs(got - ref)) < 1e-12


# ---------------------------------------------------------------------------
# Row encodings
# ---------------------------------------------------------------------------

def test_int8_rows_hand_worked_and_bound(orc):
    vals = np.zeros((1, 8), np.float32)
    vals[0, :4] = [12.7, -6.35, 0.05, 0.15]
    q, s = orc.quant_int8_rows(wl.to_bf16_bits(vals))
    xf = wl.bf16_bits_to_f32(wl.to_bf16_bits(vals)).astype(np.float64)
    sf = np.float64(np.uint16(s[0]).view(np.float16))
    assert sf == np.float64(np.float16(np.float32(np.abs(xf).max()) / np.float32(127)))
    assert np.all(np.abs(q[0] * sf - xf[0]) <= sf / 2 + 1e-12)
    rng = np.random.default_rng(22)
    x = wl.to_bf16_bits(rng.standard_normal((300, 256)).astype(np.float32))
    q, s = orc.quant_int8_rows(x)
    sf = s.view(np.float16).astype(np.float64)[:, None]
    err = np.abs(q * sf - wl.bf16_bits_to_f32(x))
    assert np.all(err <= sf / 2 * (1 + 1e-3) + 1e-12)
    assert np.all(np.abs(q).max(axis=1) >= 126)
    q0, s0 = orc.quant_int8_rows(np.zeros((1, 16), np.uint16))
    assert s0[0] == 0 and np.all(q0 == 0)


def test_int4_row_bytes_match_page(orc):
    """[P1] 'What shipped': 272 B per token-head (K and V, 64-dim groups, fp16 scales)."""
    g = golden()["int4_token_head_bytes"]
    assert 2 * orc.int4_row_bytes(256) == g["value"]
    agent = 250_000 * 16 * 4 * g["value"]
    ga = golden()["int4_agent_gb"]
    assert abs(agent / 1e9 - ga["value"]) <= ga["tolerance_rel"] * ga["value"]


def test_int4_rows_roundtrip(orc):
    rng = np.random.default_rng(23)
    x = wl.to_bf16_bits(rng.standard_normal((40, 256)).astype(np.float32))
    enc = orc.quant_int4_rows(x)
    assert enc.shape == (40, 136)
    xf = wl.bf16_bits_to_f32(x)
    for t in range(40):
        sc = enc[t, 128:136].view(np.uint16).view(np.float16).astype(np.float64)
        codes = np.stack([enc[t, :128] & 15, enc[t, :128] >> 4], -1).reshape(256).astype(np.int64)
        codes = np.where(codes >= 8, codes - 16, codes)
        deq = codes * np.repeat(sc, 64)
        assert np.all(np.abs(deq - xf[t]) <= np.repeat(sc, 64) * 0.5 * (1 + 1e-3) + 1e-12)


def test_int4_to_int8_against_fp64(orc):
    rng = np.random.default_rng(24)
    x = wl.to_bf16_bits(rng.standard_normal((30, 256)).astype(np.float32))
    enc = orc.quant_int4_rows(x)
    for t in range(30):
        q8, s8 = orc.int4_to_int8_row(enc[t], 256)
        sc = enc[t, 128:136].view(np.uint16).view(np.float16).astype(np.float64)
        codes = np.stack([enc[t, :128] & 15, enc[t, :128] >> 4], -1).reshape(256).astype(np.int64)
        codes = np.where(codes >= 8, codes - 16, codes)
        deq = codes * np.repeat(sc, 64)
        s8_ref = np.float16(np.float32(np.abs(deq).max()) / np.float32(127))
        assert np.uint16(s8) == s8_ref.view(np.uint16)
        ratio = deq / np.float64(s8_ref)
        ref = np.clip(np.round(ratio), -127, 127)  # numpy rounds half to even
        tie = np.abs(np.abs(ratio - np.trunc(ratio)) - 0.5) < 1e-6
        assert np.all((q8 == ref) | tie)


# ---------------------------------------------------------------------------
# Resolvers: hand-worked examples and invariants
# ---------------------------------------------------------------------------

def test_clock_hand_worked(orc):
    """Hs = 3.  Step 0: picks {1,2} fill slots 0,1.  Step 1: picks {2,5,6}: 2 is a
    hit (slot 1, used this step); 5 takes empty slot 2; 6 sweeps: slot 0 has
    ref 1 -> cleared, slot 1 in use -> skipped, slot 2 in use -> skipped, slot 0
    ref 0 -> taken (token 1 loses it).  Hand ends after slot 0 -> 1."""
    st = orc.ClockState(3, 10)
    slot, miss, m = st.step([1, 2], 0)
    assert list(slot) == [0, 1] and list(miss) == [True, True] and m == 2
    slot, miss, m = st.step([2, 5, 6], 1)
    assert list(slot) == [1, 2, 0] and list(miss) == [False, True, True] and m == 2
    assert st.hand[0] == 1
    assert st.token_slot[1] == -1 and st.token_slot[6] == 0 and st.token_slot[5] == 2
    assert list(st.ref) == [1, 1, 1]


def test_clock_invariants_random(orc):
    rng = np.random.default_rng(25)
    Hs, n_tok, k = 40, 400, 25
    st = orc.ClockState(Hs, n_tok)
    hits = misses = 0
    for step in range(60):
        picks = np.sort(rng.choice(n_tok if step % 2 else 80, size=k, replace=False)).astype(np.int32)
        slot, miss, m = st.step(picks, step)
        hits += int((~miss).sum())
        misses += m
        assert len(set(slot.tolist())) == k  # distinct slots
        for s in range(Hs):  # token_slot / slot_token form a bijection
            t = st.slot_token[s]
            if t >= 0:
                assert st.token_slot[t] == s
        assert (st.token_slot >= 0).sum() == (st.slot_token >= 0).sum() <= Hs
    assert hits + misses == 60 * k


def test_clock_capacity_covers_all_tokens(orc):
    st = orc.ClockState(64, 64)
    rng = np.random.default_rng(26)
    st.step(np.arange(64, dtype=np.int32)[:32], 0)
    st.step(np.arange(64, dtype=np.int32)[32:], 1)
    for step in range(2, 20):
        picks = np.sort(rng.choice(64, 20, replace=False)).astype(np.int32)
        _, _, m = st.step(picks, step)
        assert m == 0


def _int4_vector(codes, scale_bits=0x3C00):
    """One int4 vector in the host-row encoding: codes of dims 2i (low nibble)
    and 2i+1 (high nibble) in byte i, two's complement, then one fp16 scale
    per 64-dim group (all groups get `scale_bits`; 0x3C00 is 1.0)."""
    codes = np.asarray(codes, np.int64)
    nib = (codes & 15).astype(np.uint8)
    body = (nib[0::2] | (nib[1::2] << 4)).astype(np.uint8)
    scales = np.full((codes.size // 64,), scale_bits, np.uint16).view(np.uint8)
    return np.concatenate([body, scales])


def test_clock_resolve_hand_worked(orc):
    """The CLOCK resolve composed with the host tier, worked by hand.
    S = 2 sinks, W = 3 tail tokens, Hs = 3 hot slots, Hkv = 2 heads, D = 64.
    HBM rows of the request: sink t -> t; tail t -> S + t mod W (the ring);
    pick -> S + W + slot.  Host row of token t: for head h, the K vector then
    the V vector, 34 bytes each (32 of codes, one fp16 group scale).
    Vector (t, h, kv) holds code c on even dims and -c on odd dims, scale 1,
    c = (4t + 2h + kv) mod 15 - 7, so every (head, K/V) of a token differs.
    Requantised to int8: s8 = fp16(|c| / 127) and the codes are
    +-127 * sign(c) (|c| / s8 lies within half a step of 127).
      step 0, T = 10, picks {3, 5}: both miss, take empty slots 0, 1.
      step 1, T = 11, picks {5, 6}: 5 hits slot 1; 6 takes empty slot 2.
      step 2, T = 12, picks {2, 4}: the hand clears the ref bits of slots 0,
        1, 2, then takes slot 0 (token 3 out) for 2 and slot 1 (token 5 out)
        for 4.
      step 3, T = 12, picks {3, 6}: 6 hits slot 2 (used this step, skipped by
        the hand); 3 clears slot 0, slot 1 and takes slot 0 (token 2 out)."""
    S, W, Hs, Hkv, D = 2, 3, 3, 2, 64
    rb = orc.int4_row_bytes(D)
    assert rb == 34
    n_tok = 12

    def code(t, h, kv):
        return (4 * t + 2 * h + kv) % 15 - 7

    host = np.zeros((n_tok, Hkv, 2, rb), np.uint8)
    for t in range(n_tok):
        for h in range(Hkv):
            for kv in range(2):
                c = code(t, h, kv)
                host[t, h, kv] = _int4_vector(np.tile([c, -c], D // 2))

    def expect_int8(c):
        s8 = np.float16(np.float32(abs(c)) / np.float32(127))
        if c:
            assert 126.5 < abs(c) / float(s8) < 127.5
        q = np.tile(np.array([127, -127], np.int64) * int(np.sign(c)), D // 2).astype(np.int8)
        return q, int(s8.view(np.uint16))

    n_rows = S + W + Hs
    k8 = np.full((n_rows, Hkv, D), 0x11, np.int8)
    v8 = np.full((n_rows, Hkv, D), 0x22, np.int8)
    ks = np.full((n_rows, Hkv), 0x1111, np.uint16)
    vs = np.full((n_rows, Hkv), 0x2222, np.uint16)
    st = orc.ClockState(Hs, n_tok)
    steps = [  # T, selection, expected rows, expected misses, slot -> token after the step
        (10, [0, 1, 3, 5, 7, 8, 9], [0, 1, 5, 6, 3, 4, 2], 2, [3, 5, -1]),
        (11, [0, 1, 5, 6, 8, 9, 10], [0, 1, 6, 7, 4, 2, 3], 1, [3, 5, 6]),
        (12, [0, 1, 2, 4, 9, 10, 11], [0, 1, 5, 6, 2, 3, 4], 2, [2, 4, 6]),
        (12, [0, 1, 3, 6, 9, 10, 11], [0, 1, 5, 7, 2, 3, 4], 1, [3, 4, 6]),
    ]
    for step, (T, sel, want_rows, want_m, want_slots) in enumerate(steps):
        rows, m = st.resolve(T, S, W, np.array(sel, np.int32), step, host, k8, v8, ks, vs, Hkv, D)
        assert list(rows) == want_rows, step
        assert m == want_m, step
        assert list(st.slot_token) == want_slots, step
        for slot, t in enumerate(want_slots):
            if t < 0:
                continue
            r = S + W + slot
            for h in range(Hkv):
                qk, sk = expect_int8(code(t, h, 0))
                qv, sv = expect_int8(code(t, h, 1))
                assert np.array_equal(k8[r, h], qk) and ks[r, h] == sk, (step, slot, h)
                assert np.array_equal(v8[r, h], qv) and vs[r, h] == sv, (step, slot, h)
        # sink and tail rows are HBM-resident: never written by the resolve
        assert np.all(k8[:S + W] == 0x11) and np.all(v8[:S + W] == 0x22)
        assert np.all(ks[:S + W] == 0x1111) and np.all(vs[:S + W] == 0x2222)
    assert list(st.ref) == [1, 0, 1] and int(st.hand[0]) == 1
    assert list(st.token_slot[[2, 3, 4, 5, 6]]) == [-1, 0, 1, -1, 2]


def test_lru_hand_worked_with_leased_hot_rows(orc):
    """The LRU resolve with the hot buffer made of rows leased from the pool:
    hot slot s is pool row hot_rows[s] (here 40, 17, 33), never hot_base + s.
    Pages of 2 tokens; page 2 (tokens 4, 5) is resident at pool page 9 (rows
    18, 19), the rest host-only.  Host row of token t: 4 bytes, all t + 100.
      step 1, picks {0, 3, 5}: 5 resident -> row 19; 0, 3 miss -> slots 0, 1.
      step 2, picks {3, 6, 7}: 3 hits slot 1 -> row 17; 6 takes slot 2 (empty);
        7 needs an untouched slot: slot 0 (stamp 1) -> row 40, token 0 out.
      step 3, picks {0, 4, 7}: 4 resident -> row 18; 7 hits slot 0 -> row 40
        (stamp 3); 0 misses: the untouched slots, by (stamp, slot), are slot 1
        (stamp 2) and slot 2 (stamp 2) -> slot 1, token 3 out -> row 17."""
    st = orc.LruState(3, 8)
    bt = np.array([-1, -1, 9, -1], np.int32)
    hot_rows = np.array([40, 17, 33], np.int32)
    host = np.repeat((np.arange(8) + 100).astype(np.uint8)[:, None], 4, axis=1)
    pool = np.zeros((64, 4), np.uint8)
    rows, m = st.resolve([0, 3, 5], 2, bt, 1000, 1, host, pool, 4, hot_rows=hot_rows)
    assert list(rows) == [40, 17, 19] and m == 2
    assert np.all(pool[40] == 100) and np.all(pool[17] == 103)
    rows, m = st.resolve([3, 6, 7], 2, bt, 1000, 2, host, pool, 4, hot_rows=hot_rows)
    assert list(rows) == [17, 33, 40] and m == 2
    assert np.all(pool[33] == 106) and np.all(pool[40] == 107) and st.token_slot[0] == -1
    rows, m = st.resolve([0, 4, 7], 2, bt, 1000, 3, host, pool, 4, hot_rows=hot_rows)
    assert list(rows) == [17, 18, 40] and m == 1
    assert np.all(pool[17] == 100) and st.token_slot[3] == -1
    assert list(st.slot_token) == [7, 0, 6] and list(st.stamp) == [3, 3, 2]
    # nothing outside the leased rows was written
    touched = {17, 33, 40}
    assert all(np.all(pool[r] == 0) for r in range(64) if r not in touched)


def test_lru_hand_worked(orc):
    """Pages of 2 tokens, 3 pages; page 0 host-only, pages 1,2 resident at pool
    pages 5,6.  2 hot slots at pool rows 100,101.  Host row of token t is the
    byte t.  Step 1 selects tokens 0,1,4: 4 is resident (row 6*2+0 = 12), 0 and 1
    miss and take slots 0 and 1.  Step 2 selects 1 only: hit (stamp 2).  Step 3
    selects 0: hit.  Step 4 selects 5 (resident) and token 0,1 again: both hits.
    Step 5 with 3 slots-worth of misses is refused (only 2 slots)."""
    st = orc.LruState(2, 6)
    bt = np.array([-1, 5, 6], np.int32)
    host = np.arange(6, dtype=np.uint8).reshape(6, 1)
    pool = np.zeros((200, 1), np.uint8)
    rows, m = st.resolve([0, 1, 4], 2, bt, 100, 1, host, pool, 1)
    assert list(rows) == [100, 101, 12] and m == 2
    assert pool[100, 0] == 0 and pool[101, 0] == 1
    rows, m = st.resolve([1], 2, bt, 100, 2, host, pool, 1)
    assert list(rows) == [101] and m == 0 and list(st.stamp) == [1, 2]
    rows, m = st.resolve([0, 1, 5], 2, bt, 100, 3, host, pool, 1)
    assert list(rows) == [100, 101, 13] and m == 0


def test_lru_evicts_least_recent_then_lowest_slot(orc):
    st = orc.LruState(3, 10)
    bt = np.full((10,), -1, np.int32)  # page size 1, everything host-only
    host = np.arange(10, dtype=np.uint8).reshape(10, 1)
    pool = np.zeros((10, 1), np.uint8)
    st.resolve([0, 1, 2], 1, bt, 0, 1, host, pool, 1)   # slots 0,1,2 <- 0,1,2 (stamp 1)
    st.resolve([1], 1, bt, 0, 2, host, pool, 1)         # slot 1 stamp 2
    rows, m = st.resolve([3, 4], 1, bt, 0, 3, host, pool, 1)
    assert m == 2 and list(rows) == [0, 2]              # (1,0) then (1,2) are oldest
    assert st.token_slot[0] == -1 and st.token_slot[2] == -1


def test_lru_all_resident_is_identity(orc):
    st = orc.LruState(4, 16)
    bt = np.array([0, 1, 2, 3], np.int32)
    rows, m = st.resolve(list(range(16)), 4, bt, 100, 1, np.zeros((16, 1), np.uint8),
                         np.zeros((200, 1), np.uint8), 1)
    assert m == 0 and list(rows) == list(range(16))


def test_lru_no_residency_misses_are_first_touches(orc):
    rng = np.random.default_rng(27)
    n_tok = 50
    st = orc.LruState(n_tok, n_tok)
    bt = np.full((n_tok,), -1, np.int32)
    seen = set()
    total = 0
    for step in range(1, 15):
        idx = np.sort(rng.choice(n_tok, 12, replace=False))
        _, m = st.resolve(idx.tolist(), 1, bt, 0, step, np.zeros((n_tok, 1), np.uint8),
                          np.zeros((n_tok, 1), np.uint8), 1)
        new = set(idx.tolist()) - seen
        seen |= new
        assert m == len(new)
        total += m
    assert total == len(seen)


# ---------------------------------------------------------------------------
# Byte arithmetic printed on the pages
# ---------------------------------------------------------------------------

def test_page_byte_arithmetic():
    g = golden()
    assert 2048 * 256 * 2 * 2 * 2 == g["sparse_read_per_layer_mib"]["value"] * 2 ** 20
    assert 12 * g["sparse_read_per_layer_mib"]["value"] == g["sparse_read_per_step_mib"]["value"]
    assert 2 * 256 * 2 * 2 == g["dense_row_bytes_per_token_layer"]["value"]
    assert 2 + (128 // 4) * 2 == g["vram_per_token_layer_bytes"]["value"]
    assert 2 ** 18 * 128 * 2 == g["pooled_scan_mib_per_layer"]["value"] * 2 ** 20
    sp = g["split_kib_per_token"]
    assert 12 * (128 // 4) * 2 / 1024 == sp["vram"]
    assert 12 * (2048 + 128 * 2) / 1024 == sp["host"]
    assert sp["vram"] + sp["host"] == sp["total"]
    sk = g["sketch_agent_gb"]
    assert abs(250_000 * 16 * (4 * 64 // 2 + 4) / 1e9 - sk["value"]) <= sk["tolerance_rel"] * sk["value"]
    assert abs(2048 / 250_000 - g["selected_fraction"]["value"]) < 5e-4
