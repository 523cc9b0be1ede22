"""CPU oracle for sparse long-context decode -- TEST INFRASTRUCTURE ONLY.

A thin numpy/ctypes wrapper around ``skv_oracle.c``: a plain, slow,
obviously-correct restatement of the method (key sketch, sketch query, pooled
keys, indexer scores, deterministic top-k with sinks/tail union and dense
fallback, int8/int4 row encodings, CLOCK and LRU resolvers, fp64 attention).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never does, and shares
no code with it.

Every function cites the page passage it follows in the C source.  Parity
status of each function is recorded with its pins in ``tests/test_oracle_*``;
real-model quality (KL divergence, recall on documents) is "parity unpinned"
and out of scope.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "skv_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libskv_oracle.so")
_lock = threading.Lock()
_lib = None

SKETCH_INT4, SKETCH_F32, POOLED_BF16 = 0, 1, 2
KV_BF16, KV_INT8, KV_FP8 = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile skv_oracle.c into libskv_oracle.so (gcc, no fused multiply-add)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-fopenmp", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            i32, i64, f32, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_double
            sig = {
                "orc_version": ([], i32),
                "orc_max_threads": ([], i32),
                "orc_set_threads": ([i32], None),
                "orc_bf16_to_f32": ([ctypes.c_uint16], f32),
                "orc_f16_to_f64": ([ctypes.c_uint16], f64),
                "orc_f32_to_f16": ([f32], ctypes.c_uint16),
                "orc_f32_to_bf16": ([f32], ctypes.c_uint16),
                "orc_fp8_e4m3_to_f64": ([ctypes.c_uint8], f64),
                "orc_order_key_i32": ([ctypes.c_int32], ctypes.c_uint32),
                "orc_order_key_f32": ([f32], ctypes.c_uint32),
                "orc_sketch_project": ([P, i64, i32, i32, i32, P, P, P, P, P], None),
                "orc_sketch_query": ([P, i32, i32, i32, i32, i32, P, P, P, P, P, P], None),
                "orc_pool_keys": ([P, i64, i32, i32, P], None),
                "orc_index_score": ([i32, i32, i32, P, P, i64, P, i32, i32, i32, P, P, P, P], i64),
                "orc_topk_select": ([i32, P, i64, P, i32, i32, i32, i32, P, i32, P], i32),
                "orc_quant_int8_rows": ([P, i64, i32, P, P], None),
                "orc_int4_row_bytes": ([i32], i32),
                "orc_quant_int4_rows": ([P, i64, i32, P], None),
                "orc_int4_to_int8_row": ([P, i32, P, P], None),
                "orc_attend": ([i32, i32, i32, i32, i32, i32, P, P, P, P, P, P, i64, i64, i64,
                                P, i32, P, f64, P], None),
                "orc_clock_step": ([i32, P, P, P, P, P, ctypes.c_int32, P, i32, P, P], i32),
                "orc_resolve_clock": ([i64, i32, i32, i32, i32, i32, P, i32, ctypes.c_int32,
                                       P, P, P, P, P, P, P, P, P, P, P], i32),
                "orc_resolve_lru": ([P, i32, i32, P, i64, P, i32, i64, P, P, P, P, P, i64, P], i32),
            }
            for name, (args, res) in sig.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = res
            _lib = lib
    return _lib


def _p(a):
    """Pointer of a C-contiguous numpy array (or NULL for None)."""
    if a is None:
        return None
    assert isinstance(a, np.ndarray) and a.flags["C_CONTIGUOUS"], "need a C-contiguous array"
    return a.ctypes.data


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def set_threads(n: int) -> None:
    _load().orc_set_threads(int(n))


def max_threads() -> int:
    return int(_load().orc_max_threads())


# ---- number formats -------------------------------------------------------

def bf16_to_f32(bits):
    lib = _load()
    return np.array([lib.orc_bf16_to_f32(int(b)) for b in np.ravel(bits)], np.float32)


def f16_to_f64(bits):
    lib = _load()
    return np.array([lib.orc_f16_to_f64(int(b)) for b in np.ravel(bits)], np.float64)


def f32_to_f16(x):
    lib = _load()
    return np.array([lib.orc_f32_to_f16(float(v)) for v in np.ravel(np.asarray(x, np.float32))], np.uint16)


def f32_to_bf16(x):
    lib = _load()
    return np.array([lib.orc_f32_to_bf16(float(v)) for v in np.ravel(np.asarray(x, np.float32))], np.uint16)


def fp8_e4m3_to_f64(codes):
    lib = _load()
    return np.array([lib.orc_fp8_e4m3_to_f64(int(c)) for c in np.ravel(codes)], np.float64)


def order_key_i32(s):
    lib = _load()
    return np.array([lib.orc_order_key_i32(int(v)) for v in np.ravel(s)], np.uint32)


def order_key_f32(s):
    lib = _load()
    return np.array([lib.orc_order_key_f32(float(v)) for v in np.ravel(np.asarray(s, np.float32))], np.uint32)


# ---- a1 / a2 / a2' --------------------------------------------------------

def sketch_project(keys_bf16, basis, c=None):
    """keys: uint16 bf16 bits [n][Hkv][d]; basis fp32 [d][r]; c fp32 [Hkv][r] or None.

    Returns dict(s=fp32 [n][Hkv][r], q4=uint8 [n][Hkv*r/2] (if c), x=fp32 ratio s/c).
    """
    lib = _load()
    keys = _c(keys_bf16, np.uint16)
    n, Hkv, d = keys.shape
    basis = _c(basis, np.float32)
    r = basis.shape[1]
    s = np.zeros((n, Hkv, r), np.float32)
    out = {"s": s}
    q4 = x = cc = None
    if c is not None:
        cc = _c(c, np.float32)
        q4 = np.zeros((n, Hkv * r // 2), np.uint8)
        x = np.zeros((n, Hkv, r), np.float32)
        out.update(q4=q4, x=x)
    lib.orc_sketch_project(_p(keys), n, Hkv, d, r, _p(basis), _p(cc), _p(q4), _p(s), _p(x))
    return out


def sketch_query(q_bf16, Hkv, basis, c=None, int8=True):
    """q: uint16 bf16 bits [B][Hq][d].  Returns dict(qp, q8, sigma, x)."""
    lib = _load()
    q = _c(q_bf16, np.uint16)
    B, Hq, d = q.shape
    basis = _c(basis, np.float32)
    r = basis.shape[1]
    qp = np.zeros((B, Hkv * r), np.float32)
    q8 = np.zeros((B, Hkv * r), np.int8) if int8 else None
    sigma = np.zeros((B,), np.float32) if int8 else None
    x = np.zeros((B, Hkv * r), np.float32) if int8 else None
    cc = None if c is None else _c(c, np.float32)
    lib.orc_sketch_query(_p(q), B, Hq, Hkv, d, r, _p(basis), _p(cc), _p(qp), _p(q8), _p(sigma), _p(x))
    return {"qp": qp, "q8": q8, "sigma": sigma, "x": x}


def pool_keys(keys_bf16, ratio=4):
    """keys: uint16 bf16 bits [n_tok][D] (n_tok multiple of ratio) -> [n_tok/ratio][D]."""
    lib = _load()
    keys = _c(keys_bf16, np.uint16)
    n_tok, D = keys.shape
    nb = n_tok // ratio
    out = np.zeros((nb, D), np.uint16)
    lib.orc_pool_keys(_p(keys), nb, D, ratio, _p(out))
    return out


# ---- a3 / a4 --------------------------------------------------------------

def index_score(mode, query, keys, lengths, S=0, W=0, ratio=1):
    """query [B][width] (int8 | fp32 | bf16 bits), keys [B][n_cap][...].

    Returns dict(okey=uint32 [B][n_cap], iscore/fscore, dscore, nan=count).
    Non-candidate entries are 0.
    """
    lib = _load()
    if mode == SKETCH_INT4:
        query = _c(query, np.int8)
        keys = _c(keys, np.uint8)
        width = query.shape[1]
    elif mode == SKETCH_F32:
        query = _c(query, np.float32)
        keys = _c(keys, np.float32)
        width = query.shape[1]
    else:
        query = _c(query, np.uint16)
        keys = _c(keys, np.uint16)
        width = query.shape[1]
    B, n_cap = keys.shape[0], keys.shape[1]
    lengths = _c(lengths, np.int32)
    okey = np.zeros((B, n_cap), np.uint32)
    dscore = np.zeros((B, n_cap), np.float64)
    iscore = np.zeros((B, n_cap), np.int32) if mode == SKETCH_INT4 else None
    fscore = np.zeros((B, n_cap), np.float32) if mode != SKETCH_INT4 else None
    nan = lib.orc_index_score(mode, B, width, _p(query), _p(keys), n_cap, _p(lengths), ratio, S, W,
                              _p(iscore), _p(fscore), _p(dscore), _p(okey))
    return {"okey": okey, "iscore": iscore, "fscore": fscore, "dscore": dscore, "nan": int(nan)}


def topk_select(okey, lengths, k, S=0, W=0, ratio=1, max_rows=None):
    lib = _load()
    okey = _c(okey, np.uint32)
    B, n_cap = okey.shape
    lengths = _c(lengths, np.int32)
    if max_rows is None:
        max_rows = (S + k + W) if ratio <= 1 else (ratio * k + ratio - 1)
    idx = np.full((B, max_rows), -1, np.int32)
    count = np.zeros((B,), np.int32)
    rc = lib.orc_topk_select(B, _p(okey), n_cap, _p(lengths), k, S, W, ratio, _p(idx), max_rows, _p(count))
    if rc != 0:
        raise ValueError("selection does not fit max_rows")
    return idx, count


# ---- row encodings --------------------------------------------------------

def quant_int8_rows(x_bf16):
    lib = _load()
    x = _c(x_bf16, np.uint16)
    shape = x.shape
    D = shape[-1]
    n = int(np.prod(shape[:-1]))
    q = np.zeros(shape, np.int8)
    s = np.zeros(shape[:-1], np.uint16)
    lib.orc_quant_int8_rows(_p(x), n, D, _p(q), _p(s))
    return q, s


def int4_row_bytes(D):
    return int(_load().orc_int4_row_bytes(D))


def quant_int4_rows(x_bf16):
    lib = _load()
    x = _c(x_bf16, np.uint16)
    shape = x.shape
    D = shape[-1]
    n = int(np.prod(shape[:-1]))
    out = np.zeros(shape[:-1] + (int4_row_bytes(D),), np.uint8)
    lib.orc_quant_int4_rows(_p(x), n, D, _p(out))
    return out


def int4_to_int8_row(enc, D):
    lib = _load()
    enc = _c(enc, np.uint8)
    q8 = np.zeros((D,), np.int8)
    s8 = np.zeros((1,), np.uint16)
    lib.orc_int4_to_int8_row(_p(enc), D, _p(q8), _p(s8))
    return q8, int(s8[0])


# ---- a6 -------------------------------------------------------------------

def attend(kind, q_bf16, k_pool, v_pool, rows, count, softmax_scale, Hkv, d, dv,
           k_scale=None, v_scale=None, row_scale=None, req_row_stride=0,
           k_pitch=None, v_pitch=None):
    """fp64 attention over selected rows.  Pools are 2-D [n_rows][pitch] arrays
    (or anything reshaped to that); returns float64 [B][Hq][dv]."""
    lib = _load()
    q = _c(q_bf16, np.uint16)
    B, Hq, _ = q.shape
    kdt = {KV_BF16: np.uint16, KV_INT8: np.int8, KV_FP8: np.uint8}[kind]
    kp = _c(k_pool, kdt)
    vp = _c(v_pool, kdt)
    if k_pitch is None:
        k_pitch = Hkv * d
    if v_pitch is None:
        v_pitch = Hkv * dv
    rows = _c(rows, np.int32)
    count = _c(count, np.int32)
    ks = None if k_scale is None else _c(k_scale, np.uint16)
    vs = None if v_scale is None else _c(v_scale, np.uint16)
    rs = None if row_scale is None else _c(row_scale, np.float32)
    out = np.zeros((B, Hq, dv), np.float64)
    lib.orc_attend(kind, B, Hq, Hkv, d, dv, _p(q), _p(kp), _p(vp), _p(ks), _p(vs), _p(rs),
                   int(k_pitch), int(v_pitch), int(req_row_stride), _p(rows), rows.shape[1],
                   _p(count), float(softmax_scale), _p(out))
    return out


# ---- a5 -------------------------------------------------------------------

class ClockState:
    """One request's windowed-CLOCK hot-buffer state (see orc_clock_step)."""

    def __init__(self, Hs, n_tok):
        self.Hs = Hs
        self.slot_token = np.full((Hs,), -1, np.int32)
        self.ref = np.zeros((Hs,), np.uint8)
        self.use_step = np.full((Hs,), -1, np.int32)
        self.token_slot = np.full((n_tok,), -1, np.int32)
        self.hand = np.zeros((1,), np.int32)

    def step(self, picks, step):
        lib = _load()
        picks = _c(picks, np.int32)
        n = picks.shape[0]
        slot = np.zeros((n,), np.int32)
        miss = np.zeros((n,), np.int32)
        m = lib.orc_clock_step(self.Hs, _p(self.slot_token), _p(self.ref), _p(self.use_step),
                               _p(self.token_slot), _p(self.hand), int(step), _p(picks), n,
                               _p(slot), _p(miss))
        if m < 0:
            raise ValueError("CLOCK sweep could not place every miss")
        return slot, miss.astype(bool), int(m)

    def resolve(self, T, S, W, idx, step, host_rows, k8, v8, k_s, v_s, Hkv, D):
        lib = _load()
        idx = _c(idx, np.int32)
        rows = np.zeros((idx.shape[0],), np.int32)
        m = lib.orc_resolve_clock(int(T), S, W, Hkv, D, self.Hs, _p(idx), idx.shape[0], int(step),
                                  _p(self.slot_token), _p(self.ref), _p(self.use_step),
                                  _p(self.token_slot), _p(self.hand), _p(host_rows), _p(k8), _p(v8),
                                  _p(k_s), _p(v_s), _p(rows))
        if m < 0:
            raise ValueError("CLOCK resolve failed")
        return rows, int(m)


class LruState:
    """One request's hot-buffer LRU state (see orc_resolve_lru)."""

    def __init__(self, n_slots, n_tok):
        self.n_slots = n_slots
        self.stamp = np.full((n_slots,), -1, np.int64)
        self.slot_token = np.full((n_slots,), -1, np.int32)
        self.token_slot = np.full((n_tok,), -1, np.int32)

    def resolve(self, idx, page, block_table, hot_base, step, host, pool, row_bytes, hot_rows=None):
        """hot_rows: int32 [n_slots] pool row of each hot slot (leased blocks), or None for hot_base + s."""
        lib = _load()
        idx = _c(idx, np.int32)
        bt = _c(block_table, np.int32)
        hr = None if hot_rows is None else _c(hot_rows, np.int32)
        rows = np.zeros((idx.shape[0],), np.int32)
        m = lib.orc_resolve_lru(_p(idx), idx.shape[0], page, _p(bt), int(hot_base), _p(hr), self.n_slots,
                                int(step), _p(self.stamp), _p(self.slot_token), _p(self.token_slot),
                                _p(host), _p(pool), int(row_bytes), _p(rows))
        if m < 0:
            raise ValueError("LRU resolve: not enough untouched slots")
        return rows, int(m)
