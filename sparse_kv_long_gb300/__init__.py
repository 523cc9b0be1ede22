"""Python binding of libsparsekv.so (sparse long-context decode on GB300).

Argument marshalling only: every function passes tensor pointers, sizes and
the current CUDA stream to the C ABI declared in ``include/sparsekv.h`` and
raises ``SkvError`` on a non-zero status.  All computation runs in the CUDA
kernels of the library; there is no fallback.  If the library has not been
built, the first call raises.

bf16 tensors are passed as torch.bfloat16; fp16 scales as torch.float16.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsparsekv.so")

SKETCH_INT4, SKETCH_F32, POOLED_BF16 = 0, 1, 2
KV_BF16, KV_INT8 = 0, 1
RESIDENT, HOST_CLOCK = 0, 1
DEV_NAN, DEV_RANGE, DEV_TIMEOUT, DEV_COUNT = 1, 2, 4, 8

_lock = threading.Lock()
_lib = None


class LayerStep(ctypes.Structure):
    """The C struct skv_layer_step (include/sparsekv.h), field for field."""
    _fields_ = [
        ("B", ctypes.c_int), ("Hq", ctypes.c_int), ("Hkv", ctypes.c_int), ("d", ctypes.c_int), ("r", ctypes.c_int),
        ("n_cap", ctypes.c_int64), ("k", ctypes.c_int), ("S", ctypes.c_int), ("W", ctypes.c_int),
        ("softmax_scale", ctypes.c_float), ("policy", ctypes.c_int), ("Hs", ctypes.c_int),
        ("basis", ctypes.c_void_p), ("c", ctypes.c_void_p),
        ("sketch", ctypes.c_void_p), ("k8", ctypes.c_void_p), ("v8", ctypes.c_void_p),
        ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p), ("host_rows", ctypes.c_void_p),
        ("step", ctypes.c_void_p), ("slot_token", ctypes.c_void_p), ("ref", ctypes.c_void_p),
        ("use_step", ctypes.c_void_p), ("token_slot", ctypes.c_void_p), ("hand", ctypes.c_void_p),
        ("q", ctypes.c_void_p), ("new_k", ctypes.c_void_p), ("new_v", ctypes.c_void_p), ("lengths", ctypes.c_void_p),
        ("idx", ctypes.c_void_p), ("count", ctypes.c_void_p), ("n_miss", ctypes.c_void_p), ("q8_out", ctypes.c_void_p),
        ("out", ctypes.c_void_p),
    ]


class SkvError(RuntimeError):
    def __init__(self, name, status):
        msg = _load().skv_status_string(status).decode()
        super().__init__(f"{name} failed: status {status} ({msg})")
        self.status = status


def _load():
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                                   "(nvcc, sm_103a); there is no CPU fallback")
            lib = ctypes.CDLL(LIB_PATH)
            P, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
            sig = {
                "skv_version": ([], i32),
                "skv_status_string": ([i32], ctypes.c_char_p),
                "skv_device_sm_count": ([], i32),
                "skv_sketch_project": ([P, i64, i32, i32, i32, P, P, P, P, P], i32),
                "skv_sketch_query": ([P, i32, i32, i32, i32, i32, P, P, P, P, P], i32),
                "skv_pool_keys": ([P, i32, i64, i32, i32, i64, i64, P, P], i32),
                "skv_decode_prepare_workspace_size": ([i32, i32, i32], sz),
                "skv_decode_prepare": ([P, P, P, i32, i32, i32, i32, i32, P, P, P, P, P, P, P, P, P, P, P, sz, P],
                                       i32),
                "skv_index_score": ([i32, i32, i32, P, P, i64, P, i32, i32, i32, P, P, P, P], i32),
                "skv_topk_workspace_size": ([i32], sz),
                "skv_topk_select": ([i32, P, i64, P, i32, i32, i32, i32, P, i32, P, P, sz, P, P], i32),
                "skv_score_select_workspace_size": ([i32], sz),
                "skv_score_select": ([i32, i32, i32, P, P, i64, P, i32, i32, i32, i32, P, i32, P, P, P, sz, P, P],
                                     i32),
                "skv_decode_select": ([i32, i32, i32, i32, i32, P, P, P, P, P, P, P, P, P, P, P, i64, P, i32, i32,
                                       i32, P, i32, P, P, P, sz, P, P], i32),
                "skv_quantize_int8_rows": ([P, i64, i32, i32, P, P, P, P], i32),
                "skv_decode_layer_step_workspace_size": ([ctypes.POINTER(LayerStep)], sz),
                "skv_decode_layer_step": ([ctypes.POINTER(LayerStep), P, sz, P, P], i32),
                "skv_attend_workspace_size": ([i32, i32, i32, i32, i32], sz),
                "skv_sparse_attend_decode": ([i32, i32, i32, i32, i32, P, P, P, P, P, i64, i64, P, i32, P,
                                              f32, P, P, sz, P, P], i32),
                "skv_mla_workspace_size": ([i32, i32], sz),
                "skv_sparse_attend_mla": ([i32, i32, i32, i32, P, P, P, i64, i64, P, i32, P, f32, P, P, sz, P, P],
                                          i32),
                "skv_resolve_workspace_size": ([i32, i32], sz),
                "skv_resolve_rows_clock": ([i32, i64, P, i32, i32, i32, i32, i32, P, i32, P, P, P, P, P, P, P, P,
                                            P, P, P, P, i64, P, P, P, sz, P, P], i32),
                "skv_resolve_rows_lru": ([i32, i64, P, i32, P, i64, i64, i64, i32, P, P, P, P, P, P, P, i64, i64,
                                          P, i32, P, P, P, P, sz, P, P], i32),
                "skv_resolve_rows_lru_leased": ([i32, i64, P, i32, P, i64, P, i32, P, P, P, P, P, P, P, i64, i64,
                                                 P, i32, P, P, P, P, sz, P, P], i32),
                "skv_residency_lease_hot": ([P, i32, i32, P], i32),
                "skv_quantize_int4_rows": ([P, i64, i32, i32, P, P, i64, i64, P], i32),
                "skv_stream_read": ([P, sz, P, i32, P], i32),
                "skv_gather_read": ([P, P, i32, i64, P, P], i32),
                "skv_prefill_index_scores": ([i32, P, P, i64, P, i64, P, P], i32),
                "skv_prefill_attend": ([i32, i32, i32, i32, P, P, P, i64, P, P, i64, P, i32, P, f32, P, P, P, P],
                                       i32),
                "skv_residency_create": ([i32, i32, i32, i64, i32, ctypes.POINTER(ctypes.c_void_p)], i32),
                "skv_residency_destroy": ([P], None),
                "skv_residency_add": ([P, i32, i64, i32], i32),
                "skv_residency_remove": ([P, i32], i32),
                "skv_residency_append": ([P, i32, i64], i32),
                "skv_residency_pending": ([P, i32, P, i32, ctypes.POINTER(i32)], i32),
                "skv_residency_mark_copied": ([P, i32, P, i32], i32),
                "skv_residency_fills": ([P, i32, P, i32, ctypes.POINTER(i32)], i32),
                "skv_residency_mark_filled": ([P, i32, P, i32], i32),
                "skv_residency_reclaim": ([P, i32, P, ctypes.POINTER(i32)], i32),
                "skv_residency_block_table": ([P, P], i32),
                "skv_residency_state": ([P, i32], i32),
                "skv_residency_free_blocks": ([P], i32),
                "skv_materialize_pages": ([i32, P, i32, i32, P, i64, P, i64, i64, P, i64, P, P], i32),
                "skv_fill_pages": ([i32, P, i32, i32, P, i64, P, i64, i64, P, i64, P, P], i32),
                "skv_host_register": ([P, sz, ctypes.POINTER(ctypes.c_void_p)], i32),
                "skv_host_unregister": ([P], i32),
            }
            for name, (args, res) in sig.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = res
            _lib = lib
    return _lib


def lib():
    """The loaded ctypes library (raises if it was not built)."""
    return _load()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(name, status):
    if status != 0:
        raise SkvError(name, status)


def version() -> int:
    return int(_load().skv_version())


def sm_count() -> int:
    return int(_load().skv_device_sm_count())


# ---- a1 / a2 / a2' ----------------------------------------------------------

def sketch_project(keys, basis, c, out, out_rows=None, stream=None):
    """keys bf16 [n][Hkv][d]; basis fp32 [d][r]; c fp32 [Hkv][r] or None; out u8/fp32."""
    n, Hkv, d = keys.shape
    r = basis.shape[1]
    _check("skv_sketch_project", _load().skv_sketch_project(
        _ptr(keys), n, Hkv, d, r, _ptr(basis), _ptr(c), _ptr(out_rows), _ptr(out), _stream(stream)))
    return out


def sketch_query(q, Hkv, basis, c, out, sigma=None, stream=None):
    """q bf16 [B][Hq][d] -> out int8 (c given) or fp32 (c None) [B][Hkv*r]."""
    B, Hq, d = q.shape
    r = basis.shape[1]
    _check("skv_sketch_query", _load().skv_sketch_query(
        _ptr(q), B, Hq, Hkv, d, r, _ptr(basis), _ptr(c), _ptr(out), _ptr(sigma), _stream(stream)))
    return out


def decode_prepare_workspace_size(B, Hkv, r=64) -> int:
    return int(_load().skv_decode_prepare_workspace_size(B, Hkv, r))


def decode_prepare(q, new_k, new_v, basis, c, new_rows, sketch, k8, k_scale, v8, v_scale, q8, workspace,
                   sigma=None, stream=None):
    """Append the current token (sketch + int8 K/V rows at new_rows) and fold the query into q8."""
    B, Hq, d = q.shape
    Hkv = new_k.shape[1]
    r = basis.shape[1]
    _check("skv_decode_prepare", _load().skv_decode_prepare(
        _ptr(q), _ptr(new_k), _ptr(new_v), B, Hq, Hkv, d, r, _ptr(basis), _ptr(c), _ptr(new_rows), _ptr(sketch),
        _ptr(k8), _ptr(k_scale), _ptr(v8), _ptr(v_scale), _ptr(q8), _ptr(sigma), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))
    return q8


def layer_step_args(*, q, new_k, new_v, lengths, basis, c, sketch, k8, k_scale, v8, v_scale, idx, count, out, k, S,
                    W, softmax_scale, policy=RESIDENT, Hs=0, host_rows=None, step=None, slot_token=None, ref=None,
                    use_step=None, token_slot=None, hand=None, n_miss=None, q8_out=None) -> LayerStep:
    """Fills the skv_layer_step struct from tensors (host_rows: a device
    alias, as an int address or anything with data_ptr())."""
    B, Hq, d = q.shape
    Hkv, r = new_k.shape[1], basis.shape[1]
    n_cap = sketch.shape[1]

    def addr(t):
        if t is None:
            return None
        return int(t) if isinstance(t, int) else t.data_ptr()

    return LayerStep(B, Hq, Hkv, d, r, n_cap, k, S, W, float(softmax_scale), policy, Hs, addr(basis), addr(c),
                     addr(sketch), addr(k8), addr(v8), addr(k_scale), addr(v_scale), addr(host_rows), addr(step),
                     addr(slot_token), addr(ref), addr(use_step), addr(token_slot), addr(hand), addr(q), addr(new_k),
                     addr(new_v), addr(lengths), addr(idx), addr(count), addr(n_miss), addr(q8_out), addr(out))


def decode_layer_step_workspace_size(args: LayerStep) -> int:
    return int(_load().skv_decode_layer_step_workspace_size(ctypes.byref(args)))


def decode_layer_step(args: LayerStep, workspace, status=None, stream=None):
    """One decode step of one layer, every step of the path chained on one
    stream (append, fold, score + select, resolve, attend)."""
    _check("skv_decode_layer_step", _load().skv_decode_layer_step(
        ctypes.byref(args), _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(status),
        _stream(stream)))
    return args


def pool_keys(keys, pooled, first_block, n_blocks, ratio=4, stream=None):
    """keys bf16 [B][t_cap][D] -> pooled bf16 [B][t_cap/4][D] for the given blocks."""
    B, t_cap, D = keys.shape
    _check("skv_pool_keys", _load().skv_pool_keys(
        _ptr(keys), B, t_cap, D, ratio, int(first_block), int(n_blocks), _ptr(pooled), _stream(stream)))
    return pooled


# ---- a3 / a4 ----------------------------------------------------------------

def index_score(mode, query, keys, lengths, order_keys, S=0, W=0, ratio=1, raw=None, status=None,
                stream=None):
    B, width = query.shape[0], query.shape[1]
    n_cap = keys.shape[1]
    _check("skv_index_score", _load().skv_index_score(
        mode, B, width, _ptr(query), _ptr(keys), n_cap, _ptr(lengths), ratio, S, W, _ptr(order_keys),
        _ptr(raw), _ptr(status), _stream(stream)))
    return order_keys


def topk_workspace_size(B) -> int:
    return int(_load().skv_topk_workspace_size(B))


def topk_select(order_keys, lengths, k, idx, count, workspace, S=0, W=0, ratio=1, status=None,
                stream=None):
    B, n_cap = order_keys.shape
    _check("skv_topk_select", _load().skv_topk_select(
        B, _ptr(order_keys), n_cap, _ptr(lengths), k, S, W, ratio, _ptr(idx), idx.shape[1], _ptr(count),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(status), _stream(stream)))
    return idx, count


def score_select_workspace_size(B) -> int:
    return int(_load().skv_score_select_workspace_size(B))


def score_select(mode, query, keys, lengths, k, idx, count, workspace, S=0, W=0, ratio=1, order_keys=None,
                 status=None, stream=None):
    """Fused a3 + a4: scores every candidate and selects as topk_select does."""
    B, width = query.shape[0], query.shape[1]
    n_cap = keys.shape[1]
    _check("skv_score_select", _load().skv_score_select(
        mode, B, width, _ptr(query), _ptr(keys), n_cap, _ptr(lengths), ratio, k, S, W, _ptr(idx), idx.shape[1],
        _ptr(count), _ptr(order_keys), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _ptr(status), _stream(stream)))
    return idx, count


def decode_select(q, new_k, new_v, basis, c, new_rows, sketch, k8, k_scale, v8, v_scale, lengths, k, idx, count,
                  workspace, S=0, W=1, q8_out=None, status=None, stream=None):
    """decode_prepare + score_select(SKETCH_INT4) in one launch.  sketch uint8 [B][n_cap][Hkv*r/2]
    (also the append target); k8/v8 [B*n_cap][Hkv][d]; new_rows int64 [B] flat rows."""
    B, Hq, d = q.shape
    Hkv = new_k.shape[1]
    r = basis.shape[1]
    n_cap = sketch.shape[1]
    _check("skv_decode_select", _load().skv_decode_select(
        B, Hq, Hkv, d, r, _ptr(q), _ptr(new_k), _ptr(new_v), _ptr(basis), _ptr(c), _ptr(new_rows), _ptr(sketch),
        _ptr(k8), _ptr(k_scale), _ptr(v8), _ptr(v_scale), n_cap, _ptr(lengths), k, S, W, _ptr(idx), idx.shape[1],
        _ptr(count), _ptr(q8_out), _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(status),
        _stream(stream)))
    return idx, count


# ---- row encodings ------------------------------------------------------------

def quantize_int8_rows(x, q, scale, out_rows=None, stream=None):
    """x bf16 [n][Hkv][d] -> q int8 [rows][Hkv][d], scale fp16 [rows][Hkv]."""
    n, Hkv, d = x.shape
    _check("skv_quantize_int8_rows", _load().skv_quantize_int8_rows(
        _ptr(x), n, Hkv, d, _ptr(out_rows), _ptr(q), _ptr(scale), _stream(stream)))
    return q, scale


def quantize_int4_rows(x, out, token_pitch, head_pitch, out_rows=None, out_ptr=None, stream=None):
    """x bf16 [n][Hkv][d] -> int4 vectors at out + orow*token_pitch + h*head_pitch.

    `out` is a uint8 tensor, or None with `out_ptr` a device alias (int)."""
    n, Hkv, d = x.shape
    ptr = ctypes.c_void_p(out_ptr) if out is None else _ptr(out)
    _check("skv_quantize_int4_rows", _load().skv_quantize_int4_rows(
        _ptr(x), n, Hkv, d, _ptr(out_rows), ptr, int(token_pitch), int(head_pitch), _stream(stream)))
    return out


# ---- a5 -------------------------------------------------------------------------

def _addr(t):
    """A tensor's data pointer, or an int address (a host alias or a registered host pointer)."""
    return ctypes.c_void_p(t if isinstance(t, int) else t.data_ptr())


def resolve_workspace_size(B, max_rows) -> int:
    return int(_load().skv_resolve_workspace_size(B, max_rows))


def _resolve_ws(workspace, B, max_rows):
    if workspace is None:
        workspace = torch.empty((resolve_workspace_size(B, max_rows),), dtype=torch.uint8, device="cuda")
    return workspace


def resolve_rows_clock(lengths, idx, count, step, S, W, Hs, slot_token, ref, use_step, token_slot, hand,
                       host_rows, k8, v8, k_scale, v_scale, req_row_stride, rows_out, n_miss, workspace=None,
                       status=None, stream=None):
    """Windowed CLOCK resolve (see skv_resolve_rows_clock).  step: int32 device tensor [2] (advanced by
    the call); host_rows: uint8 tensor or an int alias."""
    B, max_rows = idx.shape
    t_cap = token_slot.shape[1]
    Hkv, d = k8.shape[-2], k8.shape[-1]
    workspace = _resolve_ws(workspace, B, max_rows)
    _check("skv_resolve_rows_clock", _load().skv_resolve_rows_clock(
        B, t_cap, _ptr(lengths), S, W, Hkv, d, Hs, _ptr(idx), max_rows, _ptr(count), _ptr(step),
        _ptr(slot_token), _ptr(ref), _ptr(use_step), _ptr(token_slot), _ptr(hand), _addr(host_rows),
        _ptr(k8), _ptr(v8), _ptr(k_scale), _ptr(v_scale), int(req_row_stride), _ptr(rows_out), _ptr(n_miss),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(status), _stream(stream)))
    return rows_out, n_miss


def resolve_rows_lru(lengths, idx, count, step, page, block_table, hot_base, hot_stride, stamp, slot_token,
                     token_slot, order, host, pool, rows_out, n_miss, workspace=None, status=None, stream=None,
                     hot_blocks=None):
    """Block table + LRU hot buffer resolve (see skv_resolve_rows_lru).  step: int32 device tensor [2]
    (advanced by the call); host: uint8 tensor or int alias.  hot_blocks: int32 device tensor
    [B][ceil(n_slots / page)] of leased blocks (skv_resolve_rows_lru_leased; hot_base, hot_stride unused)."""
    B, max_rows = idx.shape
    t_cap = token_slot.shape[1]
    n_slots = stamp.shape[1]
    n_pool_rows, row_bytes = pool.shape
    workspace = _resolve_ws(workspace, B, max_rows)
    if hot_blocks is not None:
        _check("skv_resolve_rows_lru_leased", _load().skv_resolve_rows_lru_leased(
            B, t_cap, _ptr(lengths), page, _ptr(block_table), block_table.shape[1], _ptr(hot_blocks), n_slots,
            _ptr(step), _ptr(stamp), _ptr(slot_token), _ptr(token_slot), _ptr(order), _addr(host), _ptr(pool),
            row_bytes, n_pool_rows, _ptr(idx), max_rows, _ptr(count), _ptr(rows_out), _ptr(n_miss),
            _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(status), _stream(stream)))
        return rows_out, n_miss
    _check("skv_resolve_rows_lru", _load().skv_resolve_rows_lru(
        B, t_cap, _ptr(lengths), page, _ptr(block_table), block_table.shape[1], int(hot_base), int(hot_stride),
        n_slots, _ptr(step), _ptr(stamp), _ptr(slot_token), _ptr(token_slot), _ptr(order), _addr(host), _ptr(pool),
        row_bytes,
        n_pool_rows, _ptr(idx), max_rows, _ptr(count), _ptr(rows_out), _ptr(n_miss), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(status), _stream(stream)))
    return rows_out, n_miss


def gather_read(base, rows, row_bytes, sink, stream=None):
    """Read rows[i] * row_bytes from base (tensor or int address), one warp per row; XOR into sink."""
    _check("skv_gather_read", _load().skv_gather_read(_addr(base), _ptr(rows), rows.numel(), int(row_bytes),
                                                      _ptr(sink), _stream(stream)))


def stream_read(src, nbytes, sink, grid=0, stream=None):
    """Read nbytes at src (tensor or int address) with 16-byte loads; XOR into sink (int64 tensor)."""
    _check("skv_stream_read", _load().skv_stream_read(_addr(src), int(nbytes), _ptr(sink), int(grid),
                                                      _stream(stream)))


# ---- a6 -------------------------------------------------------------------------

def attend_workspace_size(B, Hq, Hkv, d, max_rows) -> int:
    return int(_load().skv_attend_workspace_size(B, Hq, Hkv, d, max_rows))


def sparse_attend_decode(kv_kind, q, k_pool, v_pool, rows, count, softmax_scale, out, workspace,
                         Hkv, k_scale=None, v_scale=None, req_row_stride=0, n_pool_rows=None,
                         status=None, stream=None):
    """q bf16 [B][Hq][d]; pools [n_rows][Hkv][d] (bf16 or int8); rows int32 [B][max_rows]."""
    B, Hq, d = q.shape
    if n_pool_rows is None:
        n_pool_rows = k_pool.shape[0]
    _check("skv_sparse_attend_decode", _load().skv_sparse_attend_decode(
        kv_kind, B, Hq, Hkv, d, _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(k_scale), _ptr(v_scale),
        int(req_row_stride), int(n_pool_rows), _ptr(rows), rows.shape[1], _ptr(count), float(softmax_scale),
        _ptr(out), _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(status),
        _stream(stream)))
    return out


def mla_workspace_size(B, max_rows) -> int:
    return int(_load().skv_mla_workspace_size(B, max_rows))


def sparse_attend_mla(q, kv_pool, rows, count, softmax_scale, out, workspace, row_scale=None, req_row_stride=0,
                      n_pool_rows=None, status=None, stream=None):
    """q bf16 [B][128][576]; kv_pool uint8 (fp8 e4m3) [n_rows][576]; rows int32 [B][max_rows] -> out fp32."""
    B, Hq, d = q.shape
    dv = out.shape[2]
    if n_pool_rows is None:
        n_pool_rows = kv_pool.shape[0]
    _check("skv_sparse_attend_mla", _load().skv_sparse_attend_mla(
        B, Hq, d, dv, _ptr(q), _ptr(kv_pool), _ptr(row_scale), int(req_row_stride), int(n_pool_rows), _ptr(rows),
        rows.shape[1], _ptr(count), float(softmax_scale), _ptr(out), _ptr(workspace),
        0 if workspace is None else workspace.numel() * workspace.element_size(), _ptr(status), _stream(stream)))
    return out


# ---- chunked sparse prefill -------------------------------------------------------

def prefill_index_scores(q_idx, pooled, order_keys, n_blocks=None, status=None, stream=None):
    """q_idx bf16 [nq][128], pooled bf16 [n_blocks][128] -> order_keys u32 [nq][stride]."""
    nq = q_idx.shape[0]
    if n_blocks is None:
        n_blocks = pooled.shape[0]
    _check("skv_prefill_index_scores", _load().skv_prefill_index_scores(
        nq, _ptr(q_idx), _ptr(pooled), int(n_blocks), _ptr(order_keys), order_keys.shape[1], _ptr(status),
        _stream(stream)))
    return order_keys


def prefill_attend(q, k_src, v_src, n_tokens, k_stage, v_stage, idx, count, softmax_scale, state, out, Hkv,
                   status=None, stream=None):
    """q bf16 [nq][Hq][d]; k_src / v_src: a tensor or an int address (a registered
    HOST pointer, or device memory) of bf16 [n_tokens][Hkv][d]; stages bf16
    [chunk][Hkv][d]; idx int32 [nq][max_rows] ascending; state fp32 [nq][Hq][d+4]."""
    nq, Hq, d = q.shape
    chunk = k_stage.shape[0]
    _check("skv_prefill_attend", _load().skv_prefill_attend(
        nq, Hq, Hkv, d, _ptr(q), _addr(k_src), _addr(v_src), int(n_tokens), _ptr(k_stage), _ptr(v_stage),
        int(chunk), _ptr(idx), idx.shape[1], _ptr(count), float(softmax_scale), _ptr(state), _ptr(out),
        _ptr(status), _stream(stream)))
    return out


# ---- pressure-driven residency -----------------------------------------------------

RESIDENCY_FULL, RESIDENCY_MIXED, RESIDENCY_NONE = 0, 1, 2


class Residency:
    """Handle on a native residency manager (see skv_residency_*); the methods
    marshal arguments only.  Page lists are numpy int32 arrays."""

    def __init__(self, n_blocks, page, max_requests, max_pages, tail_pages=1):
        self.page, self.max_requests, self.max_pages = page, max_requests, max_pages
        h = ctypes.c_void_p()
        _check("skv_residency_create", _load().skv_residency_create(n_blocks, page, max_requests, max_pages,
                                                                   tail_pages, ctypes.byref(h)))
        self._h = h

    def close(self):
        if self._h:
            _load().skv_residency_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def add(self, b, n_tokens, host_prefix=False):
        _check("skv_residency_add", _load().skv_residency_add(self._h, b, int(n_tokens), int(bool(host_prefix))))

    def remove(self, b):
        _check("skv_residency_remove", _load().skv_residency_remove(self._h, b))

    def append(self, b, n=1):
        _check("skv_residency_append", _load().skv_residency_append(self._h, b, int(n)))

    def _list(self, name, b):
        import numpy as np
        out = np.zeros((self.max_pages,), np.int32)
        n = ctypes.c_int(0)
        _check(name, getattr(_load(), name)(self._h, b, out.ctypes.data_as(ctypes.c_void_p), self.max_pages,
                                            ctypes.byref(n)))
        return out[:n.value].copy()

    def pending(self, b):
        return self._list("skv_residency_pending", b)

    def fills(self, b):
        return self._list("skv_residency_fills", b)

    def mark_copied(self, b, pages):
        import numpy as np
        p = np.ascontiguousarray(pages, np.int32)
        _check("skv_residency_mark_copied", _load().skv_residency_mark_copied(
            self._h, b, p.ctypes.data_as(ctypes.c_void_p), p.size))

    def mark_filled(self, b, pages):
        import numpy as np
        p = np.ascontiguousarray(pages, np.int32)
        _check("skv_residency_mark_filled", _load().skv_residency_mark_filled(
            self._h, b, p.ctypes.data_as(ctypes.c_void_p), p.size))

    def lease_hot(self, b, n_pages):
        """Leases n_pages pool blocks as slot b's hot buffer; returns their numbers."""
        import numpy as np
        out = np.zeros((n_pages,), np.int32)
        _check("skv_residency_lease_hot", _load().skv_residency_lease_hot(
            self._h, b, int(n_pages), out.ctypes.data_as(ctypes.c_void_p)))
        return out

    def reclaim(self, n):
        import numpy as np
        out = np.zeros((max(n, 1), 2), np.int32)
        k = ctypes.c_int(0)
        _check("skv_residency_reclaim", _load().skv_residency_reclaim(
            self._h, int(n), out.ctypes.data_as(ctypes.c_void_p), ctypes.byref(k)))
        return out[:k.value].copy()

    def block_table(self):
        import numpy as np
        out = np.zeros((self.max_requests, self.max_pages), np.int32)
        _check("skv_residency_block_table", _load().skv_residency_block_table(
            self._h, out.ctypes.data_as(ctypes.c_void_p)))
        return out

    def state(self, b):
        return int(_load().skv_residency_state(self._h, b))

    def free_blocks(self):
        return int(_load().skv_residency_free_blocks(self._h))


def _page_copy(name, pages, page, block_table, pool, host, t_cap, status, stream):
    n_pool_rows, row_bytes = pool.shape
    B, n_pages = block_table.shape
    _check(name, getattr(_load(), name)(
        pages.shape[0], _ptr(pages), B, page, _ptr(block_table), n_pages, _ptr(pool), row_bytes, n_pool_rows,
        _addr(host), int(t_cap), _ptr(status), _stream(stream)))


def materialize_pages(pages, page, block_table, pool, host, t_cap, status=None, stream=None):
    """pages int32 [n][2] (slot, page), device; pool u8 [rows][row_bytes]; host: tensor or alias (int)."""
    _page_copy("skv_materialize_pages", pages, page, block_table, pool, host, t_cap, status, stream)


def fill_pages(pages, page, block_table, pool, host, t_cap, status=None, stream=None):
    _page_copy("skv_fill_pages", pages, page, block_table, pool, host, t_cap, status, stream)


# ---- host tier -------------------------------------------------------------------

def host_register(host_ptr: int, nbytes: int) -> int:
    """Page-lock existing host memory and return its device alias (an int)."""
    alias = ctypes.c_void_p()
    _check("skv_host_register", _load().skv_host_register(ctypes.c_void_p(host_ptr), nbytes,
                                                          ctypes.byref(alias)))
    return int(alias.value)


def host_unregister(host_ptr: int) -> None:
    _check("skv_host_unregister", _load().skv_host_unregister(ctypes.c_void_p(host_ptr)))


class HostView:
    """A shaped handle on the device alias of registered host memory.

    It stands in for a tensor argument that a call reads through its pointer
    (and, for `pool_keys`, its shape), so K/V rows or raw indexer keys can be
    read zero-copy from the host tier.  Nothing is copied.
    """

    def __init__(self, alias: int, shape, element_size: int):
        self.alias, self.shape, self._es = int(alias), tuple(int(s) for s in shape), int(element_size)

    def data_ptr(self) -> int:
        return self.alias

    def element_size(self) -> int:
        return self._es

    def numel(self) -> int:
        n = 1
        for s in self.shape:
            n *= s
        return n
