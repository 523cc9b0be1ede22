"""Parity of the latent-row (MLA) attention on the tensor cores with the
fp64 oracle: 128 absorbed heads over fp8 e4m3 rows of 576 values (V = the
first 512), ragged counts, optional per-row scales, one and several row
splits.  Bar: max abs error 2e-3 on the same selected rows."""
import math

import numpy as np
import pytest
import torch

import skvtest as T
import workloads as wl

pytestmark = pytest.mark.gpu

ATOL = 2e-3
H, D, DV = 128, 576, 512


@pytest.fixture(scope="module")
def skv():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from sparse_kv_long_gb300 import _build
    _build.build()
    import sparse_kv_long_gb300 as m
    return m


def run_mla(skv, q, pool, rows, count, scale, row_scale=None, req_row_stride=0):
    B = q.shape[0]
    max_rows = rows.shape[1]
    out = torch.full((B, H, DV), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.zeros((max(16, skv.mla_workspace_size(B, max_rows)),), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    skv.sparse_attend_mla(T.bf16_dev(q), T.dev(pool), T.dev(rows), T.dev(count), scale, out, ws,
                          row_scale=None if row_scale is None else T.dev(row_scale), req_row_stride=req_row_stride,
                          status=st)
    torch.cuda.synchronize()
    return T.host(out), int(st.item())


@pytest.mark.parametrize("B,counts,max_rows,scaled", [
    (1, [2048], 2048, False),
    (3, [2048, 1000, 63], 2048, True),
    (32, [2048] * 30 + [1, 700], 2048, False),
    (2, [130, 0], 192, True),
])
def test_mla_matches_oracle(skv, orc, B, counts, max_rows, scaled):
    n_pool = 6000
    x = wl.mla_inputs_cpu(B, n_pool, seed=17 + B)
    rng = np.random.default_rng(99 + B)
    rows = np.full((B, max_rows), -1, np.int32)
    for b, c in enumerate(counts):
        rows[b, :c] = np.sort(rng.choice(n_pool, size=c, replace=False))
    count = np.array(counts, np.int32)
    rs = rng.uniform(0.5, 2.0, n_pool).astype(np.float32) if scaled else None
    scale = 1.0 / math.sqrt(D)
    got, st = run_mla(skv, x["q"], x["pool"], rows, count, scale, rs)
    assert st == 0
    ref = orc.attend(orc.KV_FP8, x["q"], x["pool"], x["pool"], rows, count, scale, 1, D, DV, row_scale=rs,
                     k_pitch=D, v_pitch=D)
    err = np.max(np.abs(got - ref))
    assert np.isfinite(got).all()
    assert err < ATOL, err
    for b, c in enumerate(counts):
        if c == 0:
            assert (got[b] == 0).all()


def test_mla_many_requests_take_two_split_clusters(skv, orc):
    """40 requests of up to 256 rows on 152 SMs: one CTA pair per request
    would fit in a wave, but a request of more than one 64-row chunk is never
    run as a single split; it takes two splits merged inside a 4-CTA cluster,
    and the 40 clusters run in more than one wave."""
    B, max_rows, n_pool = 40, 256, 6000
    counts = [256] * 36 + [65, 130, 0, 200]
    x = wl.mla_inputs_cpu(B, n_pool, seed=40)
    rng = np.random.default_rng(4040)
    rows = np.full((B, max_rows), -1, np.int32)
    for b, c in enumerate(counts):
        rows[b, :c] = np.sort(rng.choice(n_pool, size=c, replace=False))
    count = np.array(counts, np.int32)
    scale = 1.0 / math.sqrt(D)
    assert skv.mla_workspace_size(B, max_rows) <= 16  # two splits: merged in the cluster, no partials
    got, st = run_mla(skv, x["q"], x["pool"], rows, count, scale)
    assert st == 0
    ref = orc.attend(orc.KV_FP8, x["q"], x["pool"], x["pool"], rows, count, scale, 1, D, DV, k_pitch=D, v_pitch=D)
    assert np.isfinite(got).all()
    assert np.max(np.abs(got - ref)) < ATOL
    assert (got[38] == 0).all()


def test_mla_single_row_gives_v(skv, orc):
    x = wl.mla_inputs_cpu(1, 64, seed=5)
    rows = np.array([[37]], np.int32)
    got, st = run_mla(skv, x["q"], x["pool"], rows, np.array([1], np.int32), 0.1)
    assert st == 0
    v = orc.fp8_e4m3_to_f64(x["pool"][37, :DV])
    assert np.max(np.abs(got[0] - v[None, :])) < 1e-6


def test_mla_request_row_stride_and_range(skv, orc):
    B, per = 2, 500
    x = wl.mla_inputs_cpu(B, B * per, seed=8)
    rng = np.random.default_rng(1)
    rows = np.stack([np.sort(rng.choice(per, 300, replace=False)) for _ in range(B)]).astype(np.int32)
    count = np.array([300, 300], np.int32)
    got, st = run_mla(skv, x["q"], x["pool"], rows, count, 0.05, req_row_stride=per)
    assert st == 0
    ref = orc.attend(orc.KV_FP8, x["q"], x["pool"], x["pool"], rows, count, 0.05, 1, D, DV, k_pitch=D, v_pitch=D,
                     req_row_stride=per)
    assert np.max(np.abs(got - ref)) < ATOL
    bad = rows.copy()
    bad[1, 7] = per + 10 ** 6                   # outside the pool: skipped and flagged
    got2, st2 = run_mla(skv, x["q"], x["pool"], bad, count, 0.05, req_row_stride=per)
    assert st2 & 2
    np.testing.assert_array_equal(got2[0], got[0])


def test_mla_is_deterministic(skv):
    B = 4
    x = wl.mla_inputs_cpu(B, 4096, seed=3)
    rng = np.random.default_rng(2)
    rows = np.stack([np.sort(rng.choice(4096, 2048, replace=False)) for _ in range(B)]).astype(np.int32)
    count = np.full((B,), 2048, np.int32)
    a, _ = run_mla(skv, x["q"], x["pool"], rows, count, 1 / 24)
    b, _ = run_mla(skv, x["q"], x["pool"], rows, count, 1 / 24)
    assert np.array_equal(a, b)
