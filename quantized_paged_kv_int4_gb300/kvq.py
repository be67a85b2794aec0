"""Python binding of libkvq (include/kvq.h): argument marshalling only.

Every function takes CUDA torch tensors, checks dtype / device / layout, and passes raw device
pointers plus the current torch stream to the C ABI; all compute runs in libkvq's kernels.
There is no fallback: if libkvq.so cannot be built or loaded, or a call returns an error status,
an exception is raised.
"""

import ctypes
import os
import threading

import torch

from . import build as _build

KVQ_OK = 0
KVQ_ERR_INVALID_ARG = 1
KVQ_ERR_UNSUPPORTED = 2
KVQ_ERR_WORKSPACE = 3
KVQ_ERR_OUT_OF_RANGE = 4
KVQ_ERR_CUDA = 5
KVQ_BF16, KVQ_F16, KVQ_F32 = 0, 1, 2

# the C API's declared functions, in header order
C_FUNCTIONS = ("kvq_status_string", "kvq_abi_version", "kvq_write_int4", "kvq_decode_workspace_bytes",
               "kvq_decode_int4", "kvq_decode_int4_mods", "kvq_decode_int4_noalloc", "kvq_decode_tq",
               "kvq_decode_tq_mse_workspace_bytes", "kvq_decode_tq_mse", "kvq_kpool_write",
               "kvq_kpool_seed_tail", "kvq_kpool_decode_update", "kvq_fwht128", "kvq_device_error")
KVQ_NOALLOC_SCRATCH_BYTES = 16 << 20

_lock = threading.Lock()
_handle = None

c_i32, c_i64, c_sz, c_p, c_f32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_float


class ScoreMods(ctypes.Structure):
    """kvq_score_mods (include/kvq.h)."""
    _fields_ = [("sliding_window", c_i32), ("softcap", c_f32), ("sinks", c_p), ("alibi_slopes", c_p),
                ("q_len", c_i32)]


_SIGS = {
    "kvq_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "kvq_abi_version": (c_i32, []),
    "kvq_write_int4": (ctypes.c_int, [c_p, c_p, c_i64, c_i64, c_i64, c_i64, c_p, c_p, c_p, c_p, c_p, c_p,
                                      c_i32, c_i32, c_i32, c_i32, c_i64, c_p]),
    "kvq_decode_workspace_bytes": (c_sz, [c_i32, c_i32, c_i32, c_i32, c_i32]),
    "kvq_decode_int4": (ctypes.c_int, [c_p, c_p, c_p, c_p, c_p, c_p, c_i32, c_p, c_p, c_f32, c_i32, c_p, c_sz,
                                       c_p, ctypes.c_int, c_i32, c_i32, c_i32, c_i32, c_i32, c_i64, c_p]),
    "kvq_decode_int4_mods": (ctypes.c_int, [c_p, c_p, c_p, c_p, c_p, c_p, c_i32, c_p, c_p, c_f32, c_i32, c_p, c_sz,
                                            c_p, ctypes.c_int, c_i32, c_i32, c_i32, c_i32, c_i32, c_i64,
                                            ctypes.POINTER(ScoreMods), c_p]),
    "kvq_decode_int4_noalloc": (ctypes.c_int, [c_p, c_p, c_p, c_p, c_p, c_p, c_i32, c_p, c_p, c_f32, c_i32, c_p,
                                               ctypes.c_int, c_i32, c_i32, c_i32, c_i32, c_i32, c_i64, c_p]),
    "kvq_decode_tq": (ctypes.c_int, [c_p, c_p, c_i32, c_i32, c_p, c_i32, c_p, c_f32, c_i32, c_p, c_sz, c_p,
                                     c_i32, c_i32, c_i32, c_i32, c_i32, c_i64, c_p]),
    "kvq_decode_tq_mse_workspace_bytes": (c_sz, [c_i32, c_i32, c_i32, c_i32, c_i32]),
    "kvq_decode_tq_mse": (ctypes.c_int, [c_p, c_p, c_p, c_p, c_i32, c_i32, c_i32, c_i32, c_i32, c_p, c_i32, c_p,
                                         c_f32, c_i32, c_p, c_sz, c_p, c_i32, c_i32, c_i32, c_i32, c_i32, c_i64,
                                         c_p]),
    "kvq_kpool_write": (ctypes.c_int, [c_p, c_p, c_p, c_p, c_p, c_p, c_i64, c_i32, c_i32, c_i32, c_i64, c_i32, c_p]),
    "kvq_kpool_seed_tail": (ctypes.c_int, [c_p, c_i64, c_i64, c_i32, c_i64, c_p, c_p, c_p, c_i64, c_i32, c_i32, c_p]),
    "kvq_kpool_decode_update": (ctypes.c_int, [c_p, c_i32, c_i64, c_p, c_i64, c_i64, c_i32, c_i64, c_p, c_p, c_i64,
                                               c_i64, c_p, c_i64, c_i64, c_p, c_p, c_p, c_i32, c_i32, c_i32, c_i32,
                                               c_i32, c_p]),
    "kvq_fwht128": (ctypes.c_int, [c_p, c_p, c_p, c_i64, c_p]),
    "kvq_device_error": (ctypes.c_int, [c_p, ctypes.POINTER(ctypes.c_uint32)]),
}


class KvqError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__("%s: %s" % (where, kvq_status_string(status)))


def library_path():
    return _build.LIB


def lib():
    """The loaded libkvq (built in-tree on first use if it is missing or stale)."""
    global _handle
    h = _handle
    if h is not None:
        return h
    with _lock:
        if _handle is None:
            path = _build.build()
            h = ctypes.CDLL(path)
            for name, (res, args) in _SIGS.items():
                fn = getattr(h, name)
                fn.restype = res
                fn.argtypes = args
            _handle = h
        return _handle


def kvq_status_string(status):
    return lib().kvq_status_string(int(status)).decode()


def kvq_abi_version():
    return int(lib().kvq_abi_version())


def _check(status, where):
    if status != KVQ_OK:
        raise KvqError(status, where)


def _ptr(t):
    return t.data_ptr() if t is not None else None


def _stream(stream):
    return (torch.cuda.current_stream() if stream is None else stream).cuda_stream


def _need(t, name, dtype=None, contiguous=True):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError("%s must be a CUDA tensor" % name)
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if contiguous and not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)


def _out_code(dtype):
    return {torch.bfloat16: KVQ_BF16, torch.float16: KVQ_F16, torch.float32: KVQ_F32}[dtype]


def kvq_write_int4(key, value, k_cache, v_cache, k_scale, v_scale, slot_mapping, rht_signs=None, stream=None):
    """reshape_and_cache_int4: key/value [T, Hk, D] bf16 (last dim contiguous) into the paged cache."""
    _need(key, "key", torch.bfloat16, contiguous=False)
    _need(value, "value", torch.bfloat16, contiguous=False)
    if key.stride(-1) != 1 or value.stride(-1) != 1 or key.shape != value.shape:
        raise ValueError("key/value must have the same shape and a contiguous last dim")
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, n, torch.uint8)
    for t, n in ((k_scale, "k_scale"), (v_scale, "v_scale")):
        _need(t, n, torch.float32)
    _need(slot_mapping, "slot_mapping", torch.int64)
    if rht_signs is not None:
        _need(rht_signs, "rht_signs", torch.float32)
    T, Hk, D = key.shape
    nb, bs = k_cache.shape[0], k_cache.shape[1]
    if tuple(k_cache.shape) != (nb, bs, Hk, D // 2) or tuple(k_scale.shape) != (nb, bs, Hk):
        raise ValueError("cache shapes do not match key")
    _check(lib().kvq_write_int4(_ptr(key), _ptr(value), key.stride(0), key.stride(1), value.stride(0),
                                value.stride(1), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
                                _ptr(slot_mapping), _ptr(rht_signs), T, Hk, D, bs, nb, _stream(stream)),
           "kvq_write_int4")


def kvq_decode_workspace_bytes(B, Hq, Hk, D, num_splits=0):
    return int(lib().kvq_decode_workspace_bytes(B, Hq, Hk, D, num_splits))


def decode_workspace(B, Hq, Hk, D, num_splits=0, device=None):
    """A workspace for kvq_decode_int4 / kvq_decode_tq (reusable across calls on one stream)."""
    need = kvq_decode_workspace_bytes(B, Hq, Hk, D, num_splits)
    if need == 0:
        raise ValueError("unsupported decode shape")
    return torch.empty((need,), dtype=torch.uint8, device=device)


def _workspace(workspace, B, Hq, Hk, D, num_splits, device):
    """The caller's workspace (its size is checked by the library), or a new one of the needed size."""
    if workspace is None:
        need = kvq_decode_workspace_bytes(B, Hq, Hk, D, num_splits)
        return torch.empty((max(need, 16),), dtype=torch.uint8, device=device)
    _need(workspace, "workspace", torch.uint8)
    return workspace


def kvq_decode_int4(q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, rht_signs, softmax_scale,
                    out=None, workspace=None, num_splits=0, out_dtype=None, stream=None,
                    sliding_window=0, softcap=0.0, sinks=None, alibi_slopes=None, q_len=1):
    """unified_attention_int4 (decode): q [B * q_len, Hq, D] bf16 -> out [B * q_len, Hq, D]. Returns out.

    sliding_window / softcap / sinks ([Hq] fp32) / alibi_slopes ([Hq] fp32): the score modifiers
    (kvq_decode_int4_mods); all off by default. q_len > 1: multi-token (causal) decode."""
    _need(q, "q", torch.bfloat16)
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, n, torch.uint8)
    for t, n in ((k_scale, "k_scale"), (v_scale, "v_scale")):
        _need(t, n, torch.float32)
    _need(block_table, "block_table", torch.int32)
    _need(seq_lens, "seq_lens", torch.int32)
    if rht_signs is not None:
        _need(rht_signs, "rht_signs", torch.float32)
    BQ, Hq, D = q.shape
    if q_len < 1 or BQ % q_len:
        raise ValueError("q must hold q_len rows per sequence")
    B = BQ // q_len
    nb, bs, Hk = k_cache.shape[0], k_cache.shape[1], k_cache.shape[2]
    if out is None:
        out = torch.empty((BQ, Hq, D), dtype=out_dtype or torch.float32, device=q.device)
    _need(out, "out")
    workspace = _workspace(workspace, B, q_len * Hq, Hk, D, num_splits, q.device)
    if sliding_window or softcap or sinks is not None or alibi_slopes is not None or q_len > 1:
        for t, n in ((sinks, "sinks"), (alibi_slopes, "alibi_slopes")):
            if t is not None:
                _need(t, n, torch.float32)
                if t.numel() != Hq:
                    raise ValueError("%s must have Hq = %d entries" % (n, Hq))
        mods = ScoreMods(int(sliding_window), float(softcap), _ptr(sinks), _ptr(alibi_slopes), int(q_len))
        _check(lib().kvq_decode_int4_mods(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
                                          _ptr(block_table), block_table.shape[1], _ptr(seq_lens), _ptr(rht_signs),
                                          float(softmax_scale), num_splits, _ptr(workspace), workspace.numel(),
                                          _ptr(out), _out_code(out.dtype), B, Hq, Hk, D, bs, nb, ctypes.byref(mods),
                                          _stream(stream)),
               "kvq_decode_int4_mods")
        return out
    _check(lib().kvq_decode_int4(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
                                 _ptr(block_table), block_table.shape[1], _ptr(seq_lens), _ptr(rht_signs),
                                 float(softmax_scale), num_splits, _ptr(workspace), workspace.numel(),
                                 _ptr(out), _out_code(out.dtype), B, Hq, Hk, D, bs, nb, _stream(stream)),
           "kvq_decode_int4")
    return out


def kvq_decode_int4_noalloc(q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, rht_signs,
                            softmax_scale, out, num_splits=0, stream=None):
    """kvq_decode_int4 without a caller workspace: the library's own device scratch array is used
    (KVQ_NOALLOC_SCRATCH_BYTES per GPU, shared by every call: order such calls on one stream).
    For callers that cannot allocate device memory; `out` must be given. Returns out."""
    _need(q, "q", torch.bfloat16)
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, n, torch.uint8)
    for t, n in ((k_scale, "k_scale"), (v_scale, "v_scale")):
        _need(t, n, torch.float32)
    _need(block_table, "block_table", torch.int32)
    _need(seq_lens, "seq_lens", torch.int32)
    _need(out, "out")
    if rht_signs is not None:
        _need(rht_signs, "rht_signs", torch.float32)
    B, Hq, D = q.shape
    nb, bs, Hk = k_cache.shape[0], k_cache.shape[1], k_cache.shape[2]
    _check(lib().kvq_decode_int4_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
                                         _ptr(block_table), block_table.shape[1], _ptr(seq_lens), _ptr(rht_signs),
                                         float(softmax_scale), num_splits, _ptr(out), _out_code(out.dtype),
                                         B, Hq, Hk, D, bs, nb, _stream(stream)),
           "kvq_decode_int4_noalloc")
    return out


def kvq_decode_tq(q, kv_cache, value_bits, block_table, seq_lens, attn_scale, out=None, workspace=None,
                  num_splits=0, stream=None):
    """TurboQuant FP8-key decode: q [B, Hq, D] fp32, kv_cache [nb, 16, Hk, slot_bytes] uint8."""
    _need(q, "q", torch.float32)
    _need(kv_cache, "kv_cache", torch.uint8)
    _need(block_table, "block_table", torch.int32)
    _need(seq_lens, "seq_lens", torch.int32)
    B, Hq, D = q.shape
    nb, bs, Hk, slot_bytes = kv_cache.shape
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float32, device=q.device)
    _need(out, "out", torch.float32)
    workspace = _workspace(workspace, B, Hq, Hk, D, num_splits, q.device)
    _check(lib().kvq_decode_tq(_ptr(q), _ptr(kv_cache), slot_bytes, value_bits, _ptr(block_table),
                               block_table.shape[1], _ptr(seq_lens), float(attn_scale), num_splits,
                               _ptr(workspace), workspace.numel(), _ptr(out), B, Hq, Hk, D, bs, nb,
                               _stream(stream)),
           "kvq_decode_tq")
    return out


def kvq_decode_tq_mse_workspace_bytes(B, Hq, Hk, D, num_splits=0):
    return int(lib().kvq_decode_tq_mse_workspace_bytes(B, Hq, Hk, D, num_splits))


def kvq_decode_tq_mse(q, rotation, centroids, kv_cache, key_bits, key_packed_size, value_bits, block_table,
                      seq_lens, attn_scale, norm_correction=False, out=None, workspace=None, num_splits=0,
                      stream=None):
    """TurboQuant decode with MSE keys: q [B, Hq, D] fp32 (original query), rotation [D, D] fp32 (Pi),
    centroids [2^key_bits] fp32, kv_cache [nb, 16, Hk, slot_bytes] uint8."""
    _need(q, "q", torch.float32)
    _need(rotation, "rotation", torch.float32)
    _need(centroids, "centroids", torch.float32)
    _need(kv_cache, "kv_cache", torch.uint8)
    _need(block_table, "block_table", torch.int32)
    _need(seq_lens, "seq_lens", torch.int32)
    B, Hq, D = q.shape
    nb, bs, Hk, slot_bytes = kv_cache.shape
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float32, device=q.device)
    _need(out, "out", torch.float32)
    if workspace is None:
        workspace = torch.empty((max(kvq_decode_tq_mse_workspace_bytes(B, Hq, Hk, D, num_splits), 16),),
                                dtype=torch.uint8, device=q.device)
    _need(workspace, "workspace", torch.uint8)
    _check(lib().kvq_decode_tq_mse(_ptr(q), _ptr(rotation), _ptr(centroids), _ptr(kv_cache), slot_bytes, key_bits,
                                   key_packed_size, value_bits, int(bool(norm_correction)), _ptr(block_table),
                                   block_table.shape[1], _ptr(seq_lens), float(attn_scale), num_splits,
                                   _ptr(workspace), workspace.numel(), _ptr(out), B, Hq, Hk, D, bs, nb,
                                   _stream(stream)),
           "kvq_decode_tq_mse")
    return out


def kvq_kpool_write(kv_cache, slot_k, slot_score, ape, loc, write_mask=None, round_scale=True, stream=None):
    """kpool_compress_and_write_cache: kv_cache [num_blocks, page_size, 132] uint8 written in place;
    slot_k [n, pool, 128] bf16, slot_score [n, pool, 128] fp32, ape [pool, 128] fp32, loc [n] int64."""
    _need(kv_cache, "kv_cache", torch.uint8)
    _need(slot_k, "slot_k", torch.bfloat16)
    _need(slot_score, "slot_score", torch.float32)
    _need(ape, "ape", torch.float32)
    _need(loc, "loc", torch.int64)
    if write_mask is not None:
        _need(write_mask, "write_mask", torch.bool)
    n, pool, hd = slot_k.shape
    if tuple(slot_score.shape) != (n, pool, hd) or tuple(ape.shape) != (pool, hd) or loc.numel() != n:
        raise ValueError("slot_score / ape / loc shapes do not match slot_k")
    nb, ps, row = kv_cache.shape
    if row != hd + 4:
        raise ValueError("kv_cache rows must be head_dim + 4 bytes")
    _check(lib().kvq_kpool_write(_ptr(kv_cache), _ptr(slot_k), _ptr(slot_score), _ptr(ape), _ptr(loc),
                                 _ptr(write_mask), n, pool, hd, ps, nb, int(bool(round_scale)), _stream(stream)),
           "kvq_kpool_write")


def _tail_geometry(tail):
    """(block stride, half stride, ring, blocks) of a bf16 tail cache [blocks, 2, ring, 128] view."""
    if not isinstance(tail, torch.Tensor) or not tail.is_cuda or tail.dtype != torch.bfloat16 or tail.dim() != 4:
        raise TypeError("tail must be a CUDA bf16 tensor [blocks, 2, ring, 128]")
    if tail.shape[1] != 2 or tail.shape[3] != 128 or tail.stride(3) != 1 or tail.stride(2) != 128:
        raise ValueError("tail must be [blocks, 2, ring, 128] with contiguous rows")
    return tail.stride(0), tail.stride(1), tail.shape[2], tail.shape[0]


def kvq_kpool_seed_tail(tail, key, gate_score, tslot, kpool, stream=None):
    """kpool_seed_tail_cache: tail bf16 [blocks, 2, ring, 128] (a view; strides are honoured),
    key / gate_score bf16 [n, 128], tslot int32 [n]."""
    bs, hs, ring, nblk = _tail_geometry(tail)
    _need(key, "key", torch.bfloat16)
    _need(gate_score, "gate_score", torch.bfloat16)
    _need(tslot, "tslot", torch.int32)
    n = tslot.numel()
    if tuple(key.shape) != (n, 128) or tuple(gate_score.shape) != (n, 128):
        raise ValueError("key / gate_score must be [n, 128]")
    _check(lib().kvq_kpool_seed_tail(_ptr(tail), bs, hs, ring, nblk, _ptr(key), _ptr(gate_score), _ptr(tslot), n,
                                     kpool, 128, _stream(stream)), "kvq_kpool_seed_tail")


def kvq_kpool_decode_update(kv_cache, tail, tail_slot_mapping, key, slot_score, ape, slot_mapping, positions,
                            pool_size, round_scale=True, stream=None):
    """kpool_decode_update_and_maybe_write_cache_batched: key / slot_score bf16 [R, next_n, 128];
    tail_slot_mapping / slot_mapping / positions int32 [R, next_n]; ape fp32 [pool, 128]."""
    bs, hs, ring, nblk = _tail_geometry(tail)
    _need(kv_cache, "kv_cache", torch.uint8)
    for t, n in ((key, "key"), (slot_score, "slot_score")):
        _need(t, n, torch.bfloat16, contiguous=False)
        if t.dim() != 3 or t.shape[2] != 128 or t.stride(2) != 1:
            raise ValueError("%s must be [R, next_n, 128] with a contiguous last dim" % n)
    _need(ape, "ape", torch.float32)
    for t, n in ((tail_slot_mapping, "tail_slot_mapping"), (slot_mapping, "slot_mapping"), (positions, "positions")):
        _need(t, n, torch.int32)
        if tuple(t.shape) != tuple(key.shape[:2]):
            raise ValueError("%s must be [R, next_n]" % n)
    R, next_n = key.shape[0], key.shape[1]
    nb, ps, row = kv_cache.shape
    _check(lib().kvq_kpool_decode_update(_ptr(kv_cache), ps, nb, _ptr(tail), bs, hs, ring, nblk, _ptr(tail_slot_mapping),
                                         _ptr(key), key.stride(0), key.stride(1), _ptr(slot_score), slot_score.stride(0),
                                         slot_score.stride(1), _ptr(ape), _ptr(slot_mapping), _ptr(positions), R, next_n,
                                         pool_size, 128, int(bool(round_scale)), _stream(stream)),
           "kvq_kpool_decode_update")


def kvq_fwht128(x, y=None, row_scale=None, stream=None):
    """fwht128_quant_fp8: x [rows, 128] bf16 -> (y [rows, 128] float8_e4m3fn, scale [rows, 1] fp32)."""
    _need(x, "x", torch.bfloat16)
    if x.dim() != 2 or x.shape[1] != 128:
        raise ValueError("x must be [rows, 128]")
    rows = x.shape[0]
    if y is None:
        y = torch.empty((rows, 128), dtype=torch.float8_e4m3fn, device=x.device)
    if row_scale is None:
        row_scale = torch.empty((rows, 1), dtype=torch.float32, device=x.device)
    _need(y, "y")
    _need(row_scale, "row_scale", torch.float32)
    _check(lib().kvq_fwht128(_ptr(x), _ptr(y), _ptr(row_scale), rows, _stream(stream)), "kvq_fwht128")
    return y, row_scale


def kvq_device_error(stream=None):
    """(status, flags): synchronizes the stream, reads and clears the device-side index flags."""
    flags = ctypes.c_uint32(0)
    st = lib().kvq_device_error(_stream(stream), ctypes.byref(flags))
    return int(st), int(flags.value)
