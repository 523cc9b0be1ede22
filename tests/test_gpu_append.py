"""The append (write) path of a decode step, exercised token by token.

Each decode step appends the current token to the cache before the layer
scores it: its raw indexer key (and, once 4 tokens complete a block, the
block's pooled key: "3.14M Context on 3x 3090 ...", *No Need to Rewrite the
Kernel*), its int4 K/V rows in the host tier ("8 agents x 250K context on
two 3090s ...", *What shipped*: the main KV lives in host RAM), and its
int8 rows and sketch codes in HBM (covered by the prepare tests).  These
tests append step by step and check the cache against the oracle's encoding
of the whole sequence, and that nothing else was written.
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


def test_pooled_keys_appended_block_by_block(skv, orc):
    """Two requests decode 41 and 38 tokens past a pooled prefix; every
    completed block is pooled by a one-block call at the step that completes
    it.  The pooled array equals the oracle's pooling of the final raw keys
    on every complete block, and is untouched (zero) beyond."""
    B, D, cap = 2, 128, 1200
    rng = np.random.default_rng(41)
    raw = wl.to_bf16_bits(rng.standard_normal((B, cap, D)).astype(np.float32))
    t0 = [1001, 1030]                         # tokens present before decoding
    steps = [41, 38]
    keys = torch.zeros((B, cap, D), dtype=torch.bfloat16, device="cuda")
    pooled = torch.zeros((B, cap // 4, D), dtype=torch.bfloat16, device="cuda")
    for b in range(B):
        keys[b, :t0[b]] = T.bf16_dev(raw[b, :t0[b]])
    # the prefix: every complete block at once (one call per request length)
    for b in range(B):
        one = keys[b:b + 1]
        skv.pool_keys(one, pooled[b:b + 1], 0, t0[b] // 4)
    for s in range(max(steps)):
        for b in range(B):
            if s >= steps[b]:
                continue
            t = t0[b] + s                      # the token appended at this step
            keys[b, t] = T.bf16_dev(raw[b, t])
            if (t + 1) % 4 == 0:               # it completes block t // 4
                skv.pool_keys(keys[b:b + 1], pooled[b:b + 1], t // 4, 1)
    torch.cuda.synchronize()
    got = T.host(pooled)
    for b in range(B):
        n = t0[b] + steps[b]
        nb = n // 4
        np.testing.assert_array_equal(got[b, :nb], orc.pool_keys(raw[b, :4 * nb], 4))
        assert (got[b, nb:] == 0).all()


def test_int4_host_rows_appended_in_place(skv, orc):
    """The host tier ([T][Hkv][K|V][136 B] per request) gets each new token's
    K and V int4 rows written zero-copy at its own position, through the
    registered alias, over several steps; the rows equal the oracle's
    encoding and every other byte keeps its fill."""
    B, cap, Hkv, d = 3, 300, 4, 256
    rb = orc.int4_row_bytes(d)
    tok_bytes = Hkv * 2 * rb
    rng = np.random.default_rng(43)
    nbytes = B * cap * tok_bytes
    mm = mmap.mmap(-1, nbytes)
    harr = np.frombuffer(mm, dtype=np.uint8, count=nbytes)
    harr[:] = 0x5C
    alias = skv.host_register(harr.ctypes.data, nbytes)
    try:
        pos = [17, 250, 299 - 5]               # first appended position per request
        written = np.zeros((B, cap), bool)
        Ks, Vs = {}, {}
        for s in range(6):
            k = wl.to_bf16_bits(rng.standard_normal((B, Hkv, d)).astype(np.float32) * 3)
            v = wl.to_bf16_bits(rng.standard_normal((B, Hkv, d)).astype(np.float32))
            rows = torch.tensor([b * cap + pos[b] + s for b in range(B)], dtype=torch.int64, device="cuda")
            skv.quantize_int4_rows(T.bf16_dev(k), None, tok_bytes, 2 * rb, out_rows=rows, out_ptr=alias)
            skv.quantize_int4_rows(T.bf16_dev(v), None, tok_bytes, 2 * rb, out_rows=rows, out_ptr=alias + rb)
            for b in range(B):
                written[b, pos[b] + s] = True
                Ks[(b, pos[b] + s)], Vs[(b, pos[b] + s)] = k[b], v[b]
        torch.cuda.synchronize()
        tier = harr.reshape(B, cap, Hkv, 2, rb)
        for (b, t), kb in Ks.items():
            np.testing.assert_array_equal(tier[b, t, :, 0], orc.quant_int4_rows(kb[None])[0])
            np.testing.assert_array_equal(tier[b, t, :, 1], orc.quant_int4_rows(Vs[(b, t)][None])[0])
        assert (tier[~written] == 0x5C).all()
    finally:
        torch.cuda.synchronize()
        skv.host_unregister(harr.ctypes.data)
