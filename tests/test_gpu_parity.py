"""Parity of the CUDA path (through the C ABI) with the CPU oracle, on seeded
inputs sized to span several tiles and a ragged tail.

Bars: bit-exact for integer work (int4 scores, selections, int8 encodings,
pooled keys); sketch codes exact except +-1 at rounding ties; fp32/bf16
scores: selections may differ only within 1e-3 relative of the k-th score;
attention within 2e-3 max abs error of the fp64 oracle on the same rows.
"""
import math

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


def status_word():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def check_status(st):
    torch.cuda.synchronize()
    assert int(st.item()) == 0, f"device status {int(st.item())}"


# ---------------------------------------------------------------------------
# a1 / a2 / encodings
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("n,Hkv", [(1, 4), (333, 4), (77, 2)])
def test_sketch_project_int4_and_f32(skv, orc, n, Hkv):
    rng = np.random.default_rng(100 + n)
    d, r = 256, 64
    U = wl.orthonormal_basis(d, r, 5)
    keys = wl.to_bf16_bits(wl.lowrank_rows(rng, n * Hkv, U).reshape(n, Hkv, d))
    c = wl.sketch_step(Hkv, r, d)
    ref = orc.sketch_project(keys, U, c)
    out4 = torch.zeros((n, Hkv * r // 2), dtype=torch.uint8, device="cuda")
    skv.sketch_project(T.bf16_dev(keys), T.dev(U), T.dev(c), out4)
    out32 = torch.zeros((n, Hkv * r), dtype=torch.float32, device="cuda")
    skv.sketch_project(T.bf16_dev(keys), T.dev(U), None, out32)
    torch.cuda.synchronize()
    got = T.unpack_int4(T.host(out4)).reshape(n, Hkv, r)
    want = T.unpack_int4(ref["q4"]).reshape(n, Hkv, r)
    T.assert_codes_match_except_ties(got, want, ref["x"])
    s = T.host(out32).reshape(n, Hkv, r)
    kf = wl.bf16_bits_to_f32(keys).astype(np.float64)
    bound = d * 2.0 ** -23 * np.einsum("thi,ij->thj", np.abs(kf), np.abs(U.astype(np.float64)))
    assert np.all(np.abs(s - ref["s"]) <= 2 * bound)


def test_sketch_project_append_rows(skv, orc):
    rng = np.random.default_rng(7)
    Hkv, d, r, n_cap = 4, 256, 64, 50
    U = wl.orthonormal_basis(d, r, 6)
    keys = wl.to_bf16_bits(rng.standard_normal((3, Hkv, d)).astype(np.float32))
    c = wl.sketch_step(Hkv, r, d)
    rows = np.array([49, 0, 17], np.int64)
    out = torch.full((n_cap, Hkv * r // 2), 0x5A, dtype=torch.uint8, device="cuda")
    skv.sketch_project(T.bf16_dev(keys), T.dev(U), T.dev(c), out, out_rows=T.dev(rows))
    torch.cuda.synchronize()
    o = T.host(out)
    ref = orc.sketch_project(keys, U, c)
    for i, row in enumerate(rows):
        T.assert_codes_match_except_ties(T.unpack_int4(o[row]), T.unpack_int4(ref["q4"][i]), ref["x"][i].ravel())
    untouched = np.setdiff1d(np.arange(n_cap), rows)
    assert np.all(o[untouched] == 0x5A)


@pytest.mark.parametrize("B,Hq,Hkv", [(1, 8, 2), (8, 24, 4), (3, 16, 2)])
def test_sketch_query(skv, orc, B, Hq, Hkv):
    rng = np.random.default_rng(200 + B)
    d, r = 256, 64
    U = wl.orthonormal_basis(d, r, 9)
    q = wl.to_bf16_bits(wl.lowrank_rows(rng, B * Hq, U).reshape(B, Hq, d))
    c = wl.sketch_step(Hkv, r, d)
    ref = orc.sketch_query(q, Hkv, U, c)
    q8 = torch.zeros((B, Hkv * r), dtype=torch.int8, device="cuda")
    sig = torch.zeros((B,), dtype=torch.float32, device="cuda")
    skv.sketch_query(T.bf16_dev(q), Hkv, T.dev(U), T.dev(c), q8, sig)
    qf = torch.zeros((B, Hkv * r), dtype=torch.float32, device="cuda")
    skv.sketch_query(T.bf16_dev(q), Hkv, T.dev(U), None, qf)
    torch.cuda.synchronize()
    assert np.allclose(T.host(sig), ref["sigma"], rtol=1e-5)
    T.assert_codes_match_except_ties(T.host(q8), ref["q8"], ref["x"])
    ref32 = orc.sketch_query(q, Hkv, U, None, int8=False)["qp"]
    assert np.allclose(T.host(qf), ref32, rtol=1e-4, atol=1e-4)


@pytest.mark.parametrize("n,Hkv,d", [(1, 1, 256), (301, 4, 256), (40, 2, 128)])
def test_quantize_int8_rows_bit_exact(skv, orc, n, Hkv, d):
    rng = np.random.default_rng(300 + n)
    x = rng.standard_normal((n, Hkv, d)).astype(np.float32) * rng.uniform(0.01, 10, (n, Hkv, 1)).astype(np.float32)
    x[0, 0] = 0.0  # an all-zero row
    xb = wl.to_bf16_bits(x)
    qr, sr = orc.quant_int8_rows(xb)
    q = torch.zeros((n, Hkv, d), dtype=torch.int8, device="cuda")
    s = torch.zeros((n, Hkv), dtype=torch.float16, device="cuda")
    skv.quantize_int8_rows(T.bf16_dev(xb), q, s)
    torch.cuda.synchronize()
    assert np.array_equal(T.host(q), qr)
    assert np.array_equal(T.host(s), sr)


@pytest.mark.parametrize("B,n_tok", [(1, 4), (2, 4 * 1000 + 3), (3, 4 * 517)])
def test_pool_keys_bit_exact(skv, orc, B, n_tok):
    rng = np.random.default_rng(400 + n_tok)
    D = 128
    t_cap = ((n_tok + 3) // 4) * 4 + 8
    x = wl.to_bf16_bits(rng.standard_normal((B, t_cap, D)).astype(np.float32))
    nb = n_tok // 4
    pooled = torch.zeros((B, t_cap // 4, D), dtype=torch.bfloat16, device="cuda")
    skv.pool_keys(T.bf16_dev(x), pooled, 0, nb)
    torch.cuda.synchronize()
    got = T.host(pooled)
    for b in range(B):
        assert np.array_equal(got[b, :nb], orc.pool_keys(x[b, :4 * nb], 4))
    assert np.all(got[:, nb:] == 0)


# ---------------------------------------------------------------------------
# a3 scores
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("lengths,width", [([5000], 256), ([1, 3000, 20000, 7], 256), ([4096, 999], 128),
                                           ([2500], 512)])
def test_index_score_int4_bit_exact(skv, orc, lengths, width):
    rng = np.random.default_rng(500 + sum(lengths))
    B, n_cap, S, W = len(lengths), max(lengths) + 5, 64, 100
    q8 = rng.integers(-127, 128, (B, width)).astype(np.int8)
    sk = rng.integers(0, 256, (B, n_cap, width // 2)).astype(np.uint8)
    L = np.array(lengths, np.int32)
    ref = orc.index_score(orc.SKETCH_INT4, q8, sk, L, S=S, W=W)
    okeys = torch.zeros((B, n_cap), dtype=torch.int32, device="cuda")
    raw = torch.zeros((B, n_cap), dtype=torch.int32, device="cuda")
    st = status_word()
    skv.index_score(skv.SKETCH_INT4, T.dev(q8), T.dev(sk), T.dev(L), okeys, S=S, W=W, raw=raw, status=st)
    check_status(st)
    got_k = T.host(okeys).view(np.uint32)
    got_s = T.host(raw)
    for b in range(B):
        lo, hi = S, max(S, lengths[b] - W)
        assert np.array_equal(got_k[b, lo:hi], ref["okey"][b, lo:hi])
        assert np.array_equal(got_s[b, lo:hi], ref["iscore"][b, lo:hi])
        assert np.all(got_k[b, :lo] == 0) and np.all(got_k[b, hi:] == 0)


def test_index_score_f32_and_pooled(skv, orc):
    rng = np.random.default_rng(600)
    B, n_cap, width = 2, 3001, 128
    qp = rng.standard_normal((B, width)).astype(np.float32)
    s = rng.standard_normal((B, n_cap, width)).astype(np.float32)
    L = np.array([3001, 1777], np.int32)
    ref = orc.index_score(orc.SKETCH_F32, qp, s, L, S=8, W=16)
    okeys = torch.zeros((B, n_cap), dtype=torch.int32, device="cuda")
    raw = torch.zeros((B, n_cap), dtype=torch.float32, device="cuda")
    st = status_word()
    skv.index_score(skv.SKETCH_F32, T.dev(qp), T.dev(s), T.dev(L), okeys, S=8, W=16, raw=raw, status=st)
    check_status(st)
    for b in range(B):
        lo, hi = 8, L[b] - 16
        assert np.allclose(T.host(raw)[b, lo:hi], ref["dscore"][b, lo:hi], rtol=1e-5, atol=1e-4)
    nb_cap = 2049
    qi = wl.to_bf16_bits(rng.standard_normal((B, 128)).astype(np.float32))
    pk = wl.to_bf16_bits(rng.standard_normal((B, nb_cap, 128)).astype(np.float32))
    L2 = np.array([4 * nb_cap, 4 * 1000 + 2], np.int32)
    ref2 = orc.index_score(orc.POOLED_BF16, qi, pk, L2, ratio=4)
    okeys2 = torch.zeros((B, nb_cap), dtype=torch.int32, device="cuda")
    raw2 = torch.zeros((B, nb_cap), dtype=torch.float32, device="cuda")
    skv.index_score(skv.POOLED_BF16, T.bf16_dev(qi), T.bf16_dev(pk), T.dev(L2), okeys2, ratio=4, raw=raw2,
                    status=st)
    check_status(st)
    for b in range(B):
        nb = L2[b] // 4
        assert np.allclose(T.host(raw2)[b, :nb], ref2["dscore"][b, :nb], rtol=1e-5, atol=1e-4)
        assert np.all(T.host(okeys2)[b, nb:] == 0)


def test_index_score_nan_is_reported(skv):
    qp = torch.full((1, 128), float("nan"), device="cuda")
    s = torch.ones((1, 40, 128), device="cuda")
    L = torch.tensor([40], dtype=torch.int32, device="cuda")
    okeys = torch.zeros((1, 40), dtype=torch.int32, device="cuda")
    st = status_word()
    skv.index_score(skv.SKETCH_F32, qp, s, L, okeys, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & skv.DEV_NAN


# ---------------------------------------------------------------------------
# a4 selection
# ---------------------------------------------------------------------------

def run_topk(skv, okey, L, k, S=0, W=0, ratio=1):
    B, n_cap = okey.shape
    max_rows = (S + k + W) if ratio == 1 else ratio * k + ratio - 1
    idx = torch.full((B, max_rows), -7, dtype=torch.int32, device="cuda")
    cnt = torch.zeros((B,), dtype=torch.int32, device="cuda")
    ws = torch.zeros((skv.topk_workspace_size(B),), dtype=torch.uint8, device="cuda")
    st = status_word()
    skv.topk_select(T.dev(okey.view(np.int32)), T.dev(L), k, idx, cnt, ws, S=S, W=W, ratio=ratio, status=st)
    check_status(st)
    # histograms and tickets (the parts that must start at zero) are left
    # zero-filled: per request, a block of 3 x 2048 bins and 3 tickets at the
    # start of a fixed 6280-word stride
    blocks = ws.view(torch.int32).view(B, -1)
    assert int(blocks[:, :3 * 2048 + 3].count_nonzero().item()) == 0
    return T.host(idx), T.host(cnt)


@pytest.mark.parametrize("case", [
    dict(lengths=[250_000], k=2048, S=64, W=1024, alphabet=None),
    dict(lengths=[9000, 3136, 3137, 20, 40000], k=2048, S=64, W=1024, alphabet=None),
    dict(lengths=[5000, 7000], k=512, S=64, W=256, alphabet=3),     # massive ties
    dict(lengths=[6000], k=100, S=0, W=0, alphabet=1),               # all keys equal
    dict(lengths=[3000, 4000], k=1, S=5, W=5, alphabet=50),
    dict(lengths=[70000, 1234], k=777, S=3, W=9, alphabet=None),
])
def test_topk_bit_exact(skv, orc, case):
    rng = np.random.default_rng(700 + case["k"] + len(case["lengths"]))
    L = np.array(case["lengths"], np.int32)
    n_cap = int(L.max())
    if case["alphabet"] is None:
        okey = rng.integers(0, 2 ** 32, (len(L), n_cap), dtype=np.uint64).astype(np.uint32)
        okey[:, ::97] = okey[:, 5:6]  # some exact ties among large keys
    else:
        okey = (0x80000000 + rng.integers(0, case["alphabet"], (len(L), n_cap))).astype(np.uint32)
    k, S, W = case["k"], case["S"], case["W"]
    gi, gc = run_topk(skv, okey, L, k, S, W)
    ri, rc = orc.topk_select(okey, L, k, S=S, W=W)
    assert np.array_equal(gc, rc)
    for b in range(len(L)):
        assert np.array_equal(gi[b, :gc[b]], ri[b, :rc[b]])


def test_topk_many_requests_bit_exact(skv, orc):
    """More requests than SMs (one CTA each): ragged lengths, dense and sparse
    requests side by side, heavy ties, sinks and tail."""
    rng = np.random.default_rng(901)
    B, k, S, W = 600, 300, 4, 16
    L = rng.integers(100, 20000, B).astype(np.int32)
    L[:5] = [S + W + k, S + W + k + 1, 1, 0, 19999]
    n_cap = int(L.max())
    okey = (0x80000000 + rng.integers(0, 40, (B, n_cap))).astype(np.uint32)   # few distinct keys
    okey[::2] = rng.integers(0, 2 ** 32, (B // 2, n_cap), dtype=np.uint64).astype(np.uint32)
    gi, gc = run_topk(skv, okey, L, k, S, W)
    ri, rc = orc.topk_select(okey, L, k, S=S, W=W)
    assert np.array_equal(gc, rc)
    for b in range(B):
        assert np.array_equal(gi[b, :gc[b]], ri[b, :rc[b]]), b


def test_topk_many_requests_filter_and_fallbacks(skv, orc):
    """One CTA per request (more requests than twice the SMs): the threshold
    filter for ordinary keys, and the radix passes for the two ways the
    filter gives up -- too many candidates (every key equal) and too few
    (the sampled positions hold the largest keys, so the threshold lands
    above the k-th key)."""
    rng = np.random.default_rng(905)
    B, k, n = 400, 2000, 10_000
    L = np.full(B, n, np.int32)
    okey = rng.integers(0, 2 ** 32, (B, n), dtype=np.uint64).astype(np.uint32)
    okey[1::3] = 0x80000000                                        # all equal
    samp = (np.arange(4096, dtype=np.int64) * n) // 4096           # the filter's sample positions
    low = rng.integers(0, 2 ** 20, (B, n), dtype=np.uint64).astype(np.uint32)
    high = (0xF0000000 + rng.integers(0, 2 ** 20, (B, 4096), dtype=np.uint64)).astype(np.uint32)
    for b in range(2, B, 3):
        okey[b] = low[b]
        okey[b, samp] = high[b]
    gi, gc = run_topk(skv, okey, L, k)
    ri, rc = orc.topk_select(okey, L, k)
    assert np.array_equal(gc, rc)
    for b in range(B):
        assert np.array_equal(gi[b, :gc[b]], ri[b, :rc[b]]), b


@pytest.mark.parametrize("lengths", [[2051], [2052, 2055, 4 * 262_144], [9, 2048 * 4 + 3]])
def test_topk_pooled_bit_exact(skv, orc, lengths):
    rng = np.random.default_rng(800 + len(lengths))
    L = np.array(lengths, np.int32)
    n_cap = int(L.max()) // 4 + 1
    okey = rng.integers(0x7fff0000, 0x80010000, (len(L), n_cap), dtype=np.uint64).astype(np.uint32)
    gi, gc = run_topk(skv, okey, L, 512, ratio=4)
    ri, rc = orc.topk_select(okey, L, 512, ratio=4)
    assert np.array_equal(gc, rc)
    for b in range(len(L)):
        assert np.array_equal(gi[b, :gc[b]], ri[b, :rc[b]])


def test_topk_pooled_many_requests_bit_exact(skv, orc):
    """Block selection with expansion, one CTA per request, ragged lengths
    (dense fallback, incomplete last blocks)."""
    rng = np.random.default_rng(906)
    B = 350
    L = rng.integers(1000, 60_000, B).astype(np.int32)
    L[:3] = [4 * 512 + 3, 4 * 512 + 4, 4 * 512 + 7]
    n_cap = int(L.max()) // 4 + 1
    okey = rng.integers(0x7fff0000, 0x80010000, (B, n_cap), dtype=np.uint64).astype(np.uint32)
    gi, gc = run_topk(skv, okey, L, 512, ratio=4)
    ri, rc = orc.topk_select(okey, L, 512, ratio=4)
    assert np.array_equal(gc, rc)
    for b in range(B):
        assert np.array_equal(gi[b, :gc[b]], ri[b, :rc[b]]), b


# ---------------------------------------------------------------------------
# a6 attention
# ---------------------------------------------------------------------------

def attention_case(rng, B, Hq, Hkv, n_rows_pool, counts, max_rows, kind, shuffle=True):
    d = 256
    q = wl.to_bf16_bits(rng.standard_normal((B, Hq, d)).astype(np.float32))
    K = rng.standard_normal((n_rows_pool, Hkv, d)).astype(np.float32)
    V = rng.standard_normal((n_rows_pool, Hkv, d)).astype(np.float32)
    rows = np.full((B, max_rows), -1, np.int32)
    per_req = n_rows_pool // B
    for b in range(B):
        sel = rng.choice(per_req, size=counts[b], replace=False)
        rows[b, :counts[b]] = np.sort(sel) if not shuffle else sel
    return q, K, V, rows, per_req


@pytest.mark.parametrize("kind", ["bf16", "int8"])
@pytest.mark.parametrize("B,Hq,Hkv,counts,max_rows", [
    (1, 8, 2, [832], 832),
    (3, 24, 4, [3136, 17, 1], 3136),
    (2, 16, 2, [2048, 2051], 2051),
    (2, 32, 2, [500, 0], 600),       # 16 query heads per KV head, an empty request
    (1, 4, 4, [33], 40),             # one query head per KV head
])
def test_attention_matches_oracle(skv, orc, kind, B, Hq, Hkv, counts, max_rows):
    rng = np.random.default_rng(900 + Hq + sum(counts))
    d = 256
    pool_rows = B * 4000
    q, K, V, rows, per_req = attention_case(rng, B, Hq, Hkv, pool_rows, counts, max_rows, kind)
    cnt = np.array(counts, np.int32)
    scale = 1 / math.sqrt(d)
    out = torch.zeros((B, Hq, d), dtype=torch.float32, device="cuda")
    ws = torch.zeros((skv.attend_workspace_size(B, Hq, Hkv, d, max_rows),), dtype=torch.uint8, device="cuda")
    st = status_word()
    if kind == "bf16":
        Kb, Vb = wl.to_bf16_bits(K), wl.to_bf16_bits(V)
        skv.sparse_attend_decode(skv.KV_BF16, T.bf16_dev(q), T.bf16_dev(Kb), T.bf16_dev(Vb), T.dev(rows),
                                 T.dev(cnt), scale, out, ws, Hkv, req_row_stride=per_req, status=st)
        ref = orc.attend(orc.KV_BF16, q, Kb.reshape(pool_rows, -1), Vb.reshape(pool_rows, -1), rows, cnt,
                         scale, Hkv, d, d, req_row_stride=per_req)
    else:
        k8, ks = orc.quant_int8_rows(wl.to_bf16_bits(K))
        v8, vs = orc.quant_int8_rows(wl.to_bf16_bits(V))
        skv.sparse_attend_decode(skv.KV_INT8, T.bf16_dev(q), T.dev(k8), T.dev(v8), T.dev(rows), T.dev(cnt),
                                 scale, out, ws, Hkv, k_scale=T.f16_dev(ks), v_scale=T.f16_dev(vs),
                                 req_row_stride=per_req, status=st)
        ref = orc.attend(orc.KV_INT8, q, k8.reshape(pool_rows, -1), v8.reshape(pool_rows, -1), rows, cnt,
                         scale, Hkv, d, d, k_scale=ks, v_scale=vs, req_row_stride=per_req)
    check_status(st)
    got = T.host(out)
    err = np.max(np.abs(got - ref))
    assert err < ATOL, err
    assert int(ws.count_nonzero().item()) <= ws.numel()  # partials may remain; tickets are reset
    tickets = ws[:256].view(torch.int32)
    assert int(tickets.count_nonzero().item()) == 0


def test_attention_out_of_range_rows_are_flagged(skv):
    B, Hq, Hkv, d = 1, 8, 2, 256
    q = torch.randn((B, Hq, d), device="cuda").to(torch.bfloat16)
    K = torch.randn((100, Hkv, d), device="cuda").to(torch.bfloat16)
    rows = torch.tensor([[3, 150, 7, -2]], dtype=torch.int32, device="cuda")
    cnt = torch.tensor([4], dtype=torch.int32, device="cuda")
    out = torch.zeros((B, Hq, d), device="cuda")
    ws = torch.zeros((skv.attend_workspace_size(B, Hq, Hkv, d, 4),), dtype=torch.uint8, device="cuda")
    st = status_word()
    skv.sparse_attend_decode(skv.KV_BF16, q, K, K, rows, cnt, 0.0625, out, ws, Hkv, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & skv.DEV_RANGE
    assert torch.isfinite(out).all()


def test_attention_is_deterministic(skv):
    torch.manual_seed(0)
    B, Hq, Hkv, d, n = 2, 24, 4, 256, 3136
    q = torch.randn((B, Hq, d), device="cuda").to(torch.bfloat16)
    K = torch.randint(-127, 128, (B * 5000, Hkv, d), device="cuda", dtype=torch.int8)
    ks = torch.rand((B * 5000, Hkv), device="cuda").to(torch.float16) * 0.02
    rows = torch.stack([torch.randperm(5000, device="cuda")[:n] for _ in range(B)]).to(torch.int32)
    cnt = torch.full((B,), n, dtype=torch.int32, device="cuda")
    ws = torch.zeros((skv.attend_workspace_size(B, Hq, Hkv, d, n),), dtype=torch.uint8, device="cuda")
    outs = []
    for _ in range(3):
        out = torch.zeros((B, Hq, d), device="cuda")
        skv.sparse_attend_decode(skv.KV_INT8, q, K, K, rows, cnt, 0.0625, out, ws, Hkv, k_scale=ks, v_scale=ks,
                                 req_row_stride=5000)
        outs.append(out)
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2])


# ---------------------------------------------------------------------------
# a3 + a4 fused (one cooperative launch)
# ---------------------------------------------------------------------------

def run_fused(skv, mode, query, keys, L, k, S=0, W=0, ratio=1, want_keys=True):
    B, n_cap = keys.shape[0], keys.shape[1]
    max_rows = (S + k + W) if ratio == 1 else ratio * k + ratio - 1
    idx = torch.full((B, max_rows), -7, dtype=torch.int32, device="cuda")
    cnt = torch.zeros((B,), dtype=torch.int32, device="cuda")
    okeys = torch.zeros((B, n_cap), dtype=torch.int32, device="cuda") if want_keys else None
    ws = torch.zeros((skv.score_select_workspace_size(B),), dtype=torch.uint8, device="cuda")
    st = status_word()
    for _ in range(2):  # the workspace must be reusable without clearing
        skv.score_select(mode, query, keys, T.dev(L), k, idx, cnt, ws, S=S, W=W, ratio=ratio, order_keys=okeys,
                         status=st)
    check_status(st)
    return T.host(idx), T.host(cnt), (T.host(okeys).view(np.uint32) if want_keys else None)


@pytest.mark.parametrize("lengths,width,k,S,W", [
    ([250_000, 250_000], 256, 2048, 64, 1024),
    ([9000, 3136, 3137, 20, 40000, 70001, 5000, 1], 256, 2048, 64, 1024),
    ([4096, 999], 128, 512, 64, 256),
    ([2500, 7000, 12000], 512, 100, 8, 16),
])
def test_score_select_int4_bit_exact(skv, orc, lengths, width, k, S, W):
    rng = np.random.default_rng(1000 + sum(lengths))
    B, n_cap = len(lengths), max(lengths)
    q8 = rng.integers(-127, 128, (B, width)).astype(np.int8)
    sk = rng.integers(0, 256, (B, n_cap, width // 2)).astype(np.uint8)
    L = np.array(lengths, np.int32)
    ref = orc.index_score(orc.SKETCH_INT4, q8, sk, L, S=S, W=W)
    ri, rc = orc.topk_select(ref["okey"], L, k, S=S, W=W)
    gi, gc, gk = run_fused(skv, skv.SKETCH_INT4, T.dev(q8), T.dev(sk), L, k, S, W)
    assert np.array_equal(gc, rc)
    for b in range(B):
        assert np.array_equal(gi[b, :gc[b]], ri[b, :rc[b]])
        if lengths[b] > S + W + k:
            assert np.array_equal(gk[b, S:lengths[b] - W], ref["okey"][b, S:lengths[b] - W])


@pytest.mark.parametrize("k,S,W", [(512, 64, 256), (7, 0, 0), (1, 4, 4)])
def test_score_select_and_topk_edge_lengths(skv, orc, k, S, W):
    """The lengths around every boundary at once (1, 3-5, 63-65 tokens, the
    dense threshold S + W + k and its neighbours, 2051/2052, 8192), the fused
    launch and the standalone selection both bit-exact against the oracle."""
    rng = np.random.default_rng(1200 + k)
    edge = S + W + k
    lengths = sorted({1, 3, 4, 5, 63, 64, 65, 831, 832, 833, 2051, 2052, 8192, edge - 1, edge, edge + 1})
    lengths = [t for t in lengths if t >= 1]
    B, n_cap, width = len(lengths), max(lengths), 256
    q8 = rng.integers(-127, 128, (B, width)).astype(np.int8)
    sk = rng.integers(0, 256, (B, n_cap, width // 2)).astype(np.uint8)
    L = np.array(lengths, np.int32)
    ref = orc.index_score(orc.SKETCH_INT4, q8, sk, L, S=S, W=W)
    ri, rc = orc.topk_select(ref["okey"], L, k, S=S, W=W)
    gi, gc, _ = run_fused(skv, skv.SKETCH_INT4, T.dev(q8), T.dev(sk), L, k, S, W, want_keys=False)
    ti, tc = run_topk(skv, ref["okey"], L, k, S, W)
    assert np.array_equal(gc, rc) and np.array_equal(tc, rc)
    for b in range(B):
        assert np.array_equal(gi[b, :gc[b]], ri[b, :rc[b]]), lengths[b]
        assert np.array_equal(ti[b, :tc[b]], ri[b, :rc[b]]), lengths[b]


@pytest.mark.parametrize("distinct", [1, 2, 5])
def test_score_select_ties(skv, orc, distinct):
    """All rows drawn from a few distinct sketches: massive exact ties, incl. the
    case where every candidate has the same key."""
    rng = np.random.default_rng(77 + distinct)
    B, n_cap, width, k, S, W = 3, 30000, 256, 2048, 64, 1024
    q8 = rng.integers(-127, 128, (B, width)).astype(np.int8)
    proto = rng.integers(0, 256, (distinct, width // 2)).astype(np.uint8)
    sk = proto[rng.integers(0, distinct, (B, n_cap))]
    L = np.array([30000, 29000, 5000], np.int32)
    ref = orc.index_score(orc.SKETCH_INT4, q8, sk, L, S=S, W=W)
    ri, rc = orc.topk_select(ref["okey"], L, k, S=S, W=W)
    gi, gc, _ = run_fused(skv, skv.SKETCH_INT4, T.dev(q8), T.dev(sk), L, k, S, W, want_keys=False)
    assert np.array_equal(gc, rc)
    for b in range(B):
        assert np.array_equal(gi[b, :gc[b]], ri[b, :rc[b]])


def test_score_select_concentrated_top_keys(skv, orc):
    """Request 0 has its highest scores packed into one contiguous region, so
    one chunk holds far more of the top k than any per-chunk candidate list;
    request 1 is plain random.  Both must match the oracle bit for bit."""
    rng = np.random.default_rng(2718)
    B, n_cap, width, k, S, W = 2, 120_000, 256, 2048, 64, 1024
    q8 = rng.integers(-127, 128, (B, width)).astype(np.int8)
    sk = rng.integers(0, 256, (B, n_cap, width // 2)).astype(np.uint8)
    # high-scoring rows: each two's-complement code near +7 where the query is
    # positive and near -8 where it is negative (dim 2b in the low nibble,
    # 2b+1 in the high one), jittered by one step so the keys differ
    lo = (q8[0, 0::2] > 0).astype(np.int64)
    hi = (q8[0, 1::2] > 0).astype(np.int64)
    r0, nr = 50_000, 3000
    jl = rng.integers(0, 2, (nr, width // 2))
    jh = rng.integers(0, 2, (nr, width // 2))
    nib_lo = np.where(lo > 0, 7 - jl, 8 + jl)
    nib_hi = np.where(hi > 0, 7 - jh, 8 + jh)
    sk[0, r0:r0 + nr] = (nib_lo | (nib_hi << 4)).astype(np.uint8)
    L = np.array([n_cap, 100_000], np.int32)
    ref = orc.index_score(orc.SKETCH_INT4, q8, sk, L, S=S, W=W)
    ri, rc = orc.topk_select(ref["okey"], L, k, S=S, W=W)
    picks = ri[0, S:S + k]
    assert ((picks >= r0) & (picks < r0 + nr)).all()  # the construction did concentrate the picks
    gi, gc, _ = run_fused(skv, skv.SKETCH_INT4, T.dev(q8), T.dev(sk), L, k, S, W, want_keys=False)
    assert np.array_equal(gc, rc)
    for b in range(B):
        assert np.array_equal(gi[b, :gc[b]], ri[b, :rc[b]])


def test_score_select_float_modes_match_two_calls(skv, orc):
    rng = np.random.default_rng(4321)
    # pooled bf16, ratio 4
    B, nb_cap = 3, 70000
    qi = wl.to_bf16_bits(rng.standard_normal((B, 128)).astype(np.float32))
    pk = wl.to_bf16_bits(rng.standard_normal((B, nb_cap, 128)).astype(np.float32))
    L = np.array([4 * nb_cap, 4 * 30000 + 3, 2051], np.int32)
    gi, gc, gk = run_fused(skv, skv.POOLED_BF16, T.bf16_dev(qi), T.bf16_dev(pk), L, 512, ratio=4)
    okeys = torch.zeros((B, nb_cap), dtype=torch.int32, device="cuda")
    skv.index_score(skv.POOLED_BF16, T.bf16_dev(qi), T.bf16_dev(pk), T.dev(L), okeys, ratio=4)
    si, sc = run_topk(skv, T.host(okeys).view(np.uint32), L, 512, ratio=4)
    assert np.array_equal(gc, sc)
    for b in range(B):
        assert np.array_equal(gi[b, :gc[b]], si[b, :sc[b]])
    # against the oracle: selections differ only within 1e-3 of the k-th score
    ref = orc.index_score(orc.POOLED_BF16, qi, pk, L, ratio=4)
    ri, rc = orc.topk_select(ref["okey"], L, 512, ratio=4)
    for b in range(2):
        nb = L[b] // 4
        kth = np.sort(ref["fscore"][b, :nb])[::-1][511]
        gblk = set((gi[b, :4 * 512:4] // 4).tolist())
        rblk = set((ri[b, :4 * 512:4] // 4).tolist())
        for blk in gblk ^ rblk:
            assert abs(ref["fscore"][b, blk] - kth) <= 1e-3 * abs(kth)
    # fp32 sketch
    B, n_cap, width = 2, 20000, 128
    qp = rng.standard_normal((B, width)).astype(np.float32)
    s = rng.standard_normal((B, n_cap, width)).astype(np.float32)
    L = np.array([20000, 9000], np.int32)
    gi, gc, _ = run_fused(skv, skv.SKETCH_F32, T.dev(qp), T.dev(s), L, 512, 64, 256, want_keys=False)
    okeys = torch.zeros((B, n_cap), dtype=torch.int32, device="cuda")
    skv.index_score(skv.SKETCH_F32, T.dev(qp), T.dev(s), T.dev(L), okeys, S=64, W=256)
    si, sc = run_topk(skv, T.host(okeys).view(np.uint32), L, 512, S=64, W=256)
    assert np.array_equal(gc, sc)
    for b in range(B):
        assert np.array_equal(gi[b, :gc[b]], si[b, :sc[b]])


# ---------------------------------------------------------------------------
# fused per-layer preparation (a1 append + int8 append + a2)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("B,Hq,Hkv", [(8, 24, 4), (3, 16, 2), (1, 8, 8)])
def test_decode_prepare_matches_oracle(skv, orc, B, Hq, Hkv):
    rng = np.random.default_rng(3000 + B * Hq)
    d, r, rows = 256, 64, 50
    U = wl.orthonormal_basis(d, r, 11)
    c = wl.sketch_step(Hkv, r, d)
    q = wl.to_bf16_bits(wl.lowrank_rows(rng, B * Hq, U).reshape(B, Hq, d))
    nk = wl.to_bf16_bits(wl.lowrank_rows(rng, B * Hkv, U).reshape(B, Hkv, d))
    nv = wl.to_bf16_bits(rng.standard_normal((B, Hkv, d)).astype(np.float32))
    new_rows = rng.choice(rows, size=B, replace=False).astype(np.int64)
    sketch = torch.full((rows, Hkv * r // 2), 0x77, dtype=torch.uint8, device="cuda")
    k8 = torch.zeros((rows, Hkv, d), dtype=torch.int8, device="cuda")
    v8 = torch.zeros((rows, Hkv, d), dtype=torch.int8, device="cuda")
    ks = torch.zeros((rows, Hkv), dtype=torch.float16, device="cuda")
    vs = torch.zeros((rows, Hkv), dtype=torch.float16, device="cuda")
    q8 = torch.zeros((B, Hkv * r), dtype=torch.int8, device="cuda")
    sig = torch.zeros((B,), dtype=torch.float32, device="cuda")
    ws = torch.zeros((skv.decode_prepare_workspace_size(B, Hkv),), dtype=torch.uint8, device="cuda")
    for _ in range(2):  # tickets must return to zero
        skv.decode_prepare(T.bf16_dev(q), T.bf16_dev(nk), T.bf16_dev(nv), T.dev(U), T.dev(c), T.dev(new_rows), sketch,
                           k8, ks, v8, vs, q8, ws, sigma=sig)
    torch.cuda.synchronize()
    ref_sk = orc.sketch_project(nk, U, c)
    ref_q = orc.sketch_query(q, Hkv, U, c)
    rk8, rks = orc.quant_int8_rows(nk)
    rv8, rvs = orc.quant_int8_rows(nv)
    s_host, k8h, v8h, ksh, vsh = T.host(sketch), T.host(k8), T.host(v8), T.host(ks), T.host(vs)
    for i in range(B):
        row = new_rows[i]
        T.assert_codes_match_except_ties(T.unpack_int4(s_host[row]), T.unpack_int4(ref_sk["q4"][i]),
                                         ref_sk["x"][i].ravel())
        assert np.array_equal(k8h[row], rk8[i]) and np.array_equal(v8h[row], rv8[i])
        assert np.array_equal(ksh[row], rks[i]) and np.array_equal(vsh[row], rvs[i])
    untouched = np.setdiff1d(np.arange(rows), new_rows)
    assert np.all(s_host[untouched] == 0x77)
    assert np.allclose(T.host(sig), ref_q["sigma"], rtol=1e-5)
    T.assert_codes_match_except_ties(T.host(q8), ref_q["q8"], ref_q["x"])


def test_score_select_pooled_ratio1_raw_indexer_keys(skv, orc):
    """Raw 128-dim bf16 indexer keys, one per token (ratio 1, no sinks/tail):
    the fused select against the oracle within 1e-3 of the k-th score, and
    identical to the two-call path."""
    rng = np.random.default_rng(777)
    B, n_cap, k = 3, 50000, 2048
    qi = wl.to_bf16_bits(rng.standard_normal((B, 128)).astype(np.float32))
    keys = wl.to_bf16_bits(rng.standard_normal((B, n_cap, 128)).astype(np.float32))
    L = np.array([50000, 20001, 2048], np.int32)
    gi, gc, _ = run_fused(skv, skv.POOLED_BF16, T.bf16_dev(qi), T.bf16_dev(keys), L, k, ratio=1)
    okeys = torch.zeros((B, n_cap), dtype=torch.int32, device="cuda")
    skv.index_score(skv.POOLED_BF16, T.bf16_dev(qi), T.bf16_dev(keys), T.dev(L), okeys, ratio=1)
    si, sc = run_topk(skv, T.host(okeys).view(np.uint32), L, k, ratio=1)
    assert np.array_equal(gc, sc)
    for b in range(B):
        assert np.array_equal(gi[b, :gc[b]], si[b, :sc[b]])
    ref = orc.index_score(orc.POOLED_BF16, qi, keys, L, ratio=1)
    ri, rc = orc.topk_select(ref["okey"], L, k, ratio=1)
    assert np.array_equal(gc, rc)
    np.testing.assert_array_equal(gi[2, :gc[2]], np.arange(2048))        # T <= k: dense
    for b in range(2):
        kth = np.sort(ref["fscore"][b, :L[b]])[::-1][k - 1]
        for t in set(gi[b, :gc[b]].tolist()) ^ set(ri[b, :rc[b]].tolist()):
            assert abs(ref["fscore"][b, t] - kth) <= 1e-3 * abs(kth)


@pytest.mark.parametrize("lengths,Hq,Hkv", [([9000, 5000, 3136, 3137], 24, 4), ([40000, 2000], 16, 2)])
def test_decode_select_equals_prepare_then_select(skv, orc, lengths, Hq, Hkv):
    """The one-launch prepare + select gives the same bits as decode_prepare
    followed by score_select: folded query, appended sketch and int8 rows,
    selection; and the selection equals the oracle's on those bytes."""
    B, d, r, k, S, W = len(lengths), 256, 64, 2048, 64, 1024
    x = wl.sketch_inputs_cpu(B, lengths, Hq, Hkv, d, r, seed=71 + B)
    Tcap = int(max(lengths))
    L = x["lengths"]
    sk0 = orc.sketch_project(x["K"].reshape(B * Tcap, Hkv, d), x["basis"], x["c"])["q4"].reshape(B, Tcap, -1)
    k80, ks0 = orc.quant_int8_rows(x["K"].reshape(B * Tcap, Hkv, d))
    v80, vs0 = orc.quant_int8_rows(x["V"].reshape(B * Tcap, Hkv, d))
    rng = np.random.default_rng(5)
    nk = wl.to_bf16_bits(wl.lowrank_rows(rng, B * Hkv, x["basis"]).reshape(B, Hkv, d))
    nv = wl.to_bf16_bits(rng.standard_normal((B, Hkv, d)).astype(np.float32))
    new_rows = (np.arange(B) * Tcap + (L - 1)).astype(np.int64)
    U, c = T.dev(x["basis"]), T.dev(x["c"])
    max_rows = S + k + W

    def state():
        return (T.dev(sk0.copy()), T.dev(k80), T.f16_dev(ks0), T.dev(v80), T.f16_dev(vs0))

    # two launches
    skA, k8A, ksA, v8A, vsA = state()
    q8A = torch.zeros((B, Hkv * r), dtype=torch.int8, device="cuda")
    pws = torch.zeros((skv.decode_prepare_workspace_size(B, Hkv),), dtype=torch.uint8, device="cuda")
    skv.decode_prepare(T.bf16_dev(x["q"]), T.bf16_dev(nk), T.bf16_dev(nv), U, c, T.dev(new_rows),
                       skA.view(B * Tcap, -1), k8A.view(B * Tcap, Hkv, d), ksA, v8A.view(B * Tcap, Hkv, d), vsA, q8A,
                       pws)
    idxA = torch.zeros((B, max_rows), dtype=torch.int32, device="cuda")
    cntA = torch.zeros((B,), dtype=torch.int32, device="cuda")
    tws = torch.zeros((skv.score_select_workspace_size(B),), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    skv.score_select(skv.SKETCH_INT4, q8A, skA, T.dev(L), k, idxA, cntA, tws, S=S, W=W, status=st)
    # one launch
    skB, k8B, ksB, v8B, vsB = state()
    q8B = torch.zeros((B, Hkv * r), dtype=torch.int8, device="cuda")
    idxB = torch.full((B, max_rows), -3, dtype=torch.int32, device="cuda")
    cntB = torch.zeros((B,), dtype=torch.int32, device="cuda")
    for _ in range(2):  # the workspace is reusable without clearing
        skv.decode_select(T.bf16_dev(x["q"]), T.bf16_dev(nk), T.bf16_dev(nv), U, c, T.dev(new_rows), skB,
                          k8B.view(B * Tcap, Hkv, d), ksB, v8B.view(B * Tcap, Hkv, d), vsB, T.dev(L), k, idxB, cntB,
                          tws, S=S, W=W, q8_out=q8B, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for a_, b_ in ((q8A, q8B), (skA, skB), (k8A, k8B), (ksA, ksB), (v8A, v8B), (vsA, vsB), (cntA, cntB)):
        np.testing.assert_array_equal(T.host(a_), T.host(b_))
    gi, gc = T.host(idxB), T.host(cntB)
    ai = T.host(idxA)
    for b in range(B):
        np.testing.assert_array_equal(gi[b, :gc[b]], ai[b, :gc[b]])
    sc = orc.index_score(orc.SKETCH_INT4, T.host(q8B), T.host(skB), L, S=S, W=W)
    ri, rc = orc.topk_select(sc["okey"], L, k, S=S, W=W)
    np.testing.assert_array_equal(gc, rc)
    for b in range(B):
        np.testing.assert_array_equal(gi[b, :gc[b]], ri[b, :rc[b]])
