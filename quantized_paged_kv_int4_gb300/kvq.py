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
               "kvq_decode_int4", "kvq_decode_int4_mods", "kvq_decode_int4_mods_workspace_bytes",
               "kvq_decode_int4_noalloc", "kvq_decode_tq",
               "kvq_decode_tq_lse", "kvq_decode_tq_mse_workspace_bytes", "kvq_decode_tq_mse", "kvq_kpool_write",
               "kvq_kpool_seed_tail", "kvq_kpool_decode_update", "kvq_fwht128", "kvq_copy_async",
               "kvq_debug_set_wait", "kvq_device_error")
KVQ_NOALLOC_SCRATCH_BYTES = 16 << 20

_lock = threading.Lock()
_handle = None

c_i32, c_i64, c_sz, c_p, c_f32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_float


class ScoreMods(ctypes.Structure):
    """kvq_score_mods (include/kvq.h)."""
    _fields_ = [("sliding_window", c_i32), ("softcap", c_f32), ("sinks", c_p), ("alibi_slopes", c_p),
                ("q_len", c_i32), ("lse_out", c_p), ("query_start_loc", c_p), ("total_q", c_i32)]


_SIGS = {
    "kvq_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "kvq_abi_version": (c_i32, []),
    "kvq_copy_async": (ctypes.c_int, [c_p, c_p, ctypes.c_size_t, c_p]),
    "kvq_write_int4": (ctypes.c_int, [c_p, c_p, c_i64, c_i64, c_i64, c_i64, c_p, c_p, c_p, c_p, c_p, c_p,
                                      c_i32, c_i32, c_i32, c_i32, c_i64, c_p]),
    "kvq_decode_workspace_bytes": (c_sz, [c_i32, c_i32, c_i32, c_i32, c_i32]),
    "kvq_decode_int4": (ctypes.c_int, [c_p, c_p, c_p, c_p, c_p, c_p, c_i32, c_p, c_p, c_f32, c_i32, c_p, c_sz,
                                       c_p, ctypes.c_int, c_i32, c_i32, c_i32, c_i32, c_i32, c_i64, c_p]),
    "kvq_decode_int4_mods": (ctypes.c_int, [c_p, c_p, c_p, c_p, c_p, c_p, c_i32, c_p, c_p, c_f32, c_i32, c_p, c_sz,
                                            c_p, ctypes.c_int, c_i32, c_i32, c_i32, c_i32, c_i32, c_i64,
                                            ctypes.POINTER(ScoreMods), c_p]),
    "kvq_decode_int4_mods_workspace_bytes": (c_sz, [c_i32, c_i32, c_i32, c_i32, c_i32, ctypes.POINTER(ScoreMods)]),
    "kvq_decode_int4_noalloc": (ctypes.c_int, [c_p, c_p, c_p, c_p, c_p, c_p, c_i32, c_p, c_p, c_f32, c_i32, c_p,
                                               ctypes.c_int, c_i32, c_i32, c_i32, c_i32, c_i32, c_i64, c_p]),
    "kvq_decode_tq": (ctypes.c_int, [c_p, c_p, c_i32, c_i32, c_p, c_i32, c_p, c_f32, c_i32, c_p, c_sz, c_p,
                                     c_i32, c_i32, c_i32, c_i32, c_i32, c_i64, c_p]),
    "kvq_decode_tq_lse": (ctypes.c_int, [c_p, c_p, c_i32, c_i32, c_p, c_i32, c_p, c_f32, c_i32, c_p, c_sz, c_p,
                                         c_p, c_i32, c_i32, c_i32, c_i32, c_i32, c_i64, c_p]),
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
    "kvq_debug_set_wait": (ctypes.c_int, [ctypes.c_uint64, c_i32]),
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


_OUT_CODES = {torch.bfloat16: KVQ_BF16, torch.float16: KVQ_F16, torch.float32: KVQ_F32}


def _out_code(dtype):
    if dtype not in _OUT_CODES:
        raise TypeError("out must be bfloat16, float16 or float32, got %s" % dtype)
    return _OUT_CODES[dtype]


def _check_int4_decode_args(q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, out, q_len=1,
                            ragged=False):
    """Shape agreement of an INT4 decode call: q / out [B * q_len, Hq, D] (ragged: [total_q, Hq, D]),
    caches [nb, bs, Hk, D/2], scales [nb, bs, Hk], block_table [B, max_blocks], seq_lens [B]."""
    if q.dim() != 3:
        raise ValueError("q must be [B, Hq, D]")
    BQ, Hq, D = q.shape
    if k_cache.dim() != 4 or tuple(v_cache.shape) != tuple(k_cache.shape) or k_cache.shape[3] * 2 != D:
        raise ValueError("k_cache / v_cache must both be [num_blocks, block_size, Hk, D/2]")
    nb, bs, Hk = k_cache.shape[0], k_cache.shape[1], k_cache.shape[2]
    for t, n in ((k_scale, "k_scale"), (v_scale, "v_scale")):
        if tuple(t.shape) != (nb, bs, Hk):
            raise ValueError("%s must be [num_blocks, block_size, Hk] = %s" % (n, (nb, bs, Hk)))
    B = block_table.shape[0] if ragged else BQ // q_len
    if block_table.dim() != 2 or block_table.shape[0] != B:
        raise ValueError("block_table must be [B, max_blocks] with B = %d" % B)
    if seq_lens.dim() != 1 or seq_lens.numel() != B:
        raise ValueError("seq_lens must have B = %d entries" % B)
    if out is not None:
        if tuple(out.shape) != tuple(q.shape):
            raise ValueError("out must have q's shape %s, got %s" % (tuple(q.shape), tuple(out.shape)))
        _out_code(out.dtype)


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


def kvq_decode_int4_mods_workspace_bytes(B, Hq, Hk, D, num_splits=0, mods=None):
    return int(lib().kvq_decode_int4_mods_workspace_bytes(B, Hq, Hk, D, num_splits,
                                                          None if mods is None else ctypes.byref(mods)))


def kvq_decode_int4(q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, rht_signs, softmax_scale,
                    out=None, workspace=None, num_splits=0, out_dtype=None, stream=None,
                    sliding_window=0, softcap=0.0, sinks=None, alibi_slopes=None, q_len=1, lse_out=None,
                    query_start_loc=None):
    """unified_attention_int4 (decode): q [B * q_len, Hq, D] bf16 -> out [B * q_len, Hq, D]. Returns out.

    sliding_window / softcap / sinks ([Hq] fp32) / alibi_slopes ([Hq] fp32): the score modifiers
    (kvq_decode_int4_mods); all off by default. q_len > 1: multi-token (causal) decode;
    query_start_loc (int32 [B + 1], the varlen cu_seqlens_q): ragged multi-token decode with q and
    out [total_q, Hq, D]. lse_out: an fp32 [rows, Hq] tensor that receives each row's log-sum-exp."""
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
    ragged = query_start_loc is not None
    if ragged:
        _need(query_start_loc, "query_start_loc", torch.int32)
        B = block_table.shape[0]
        if query_start_loc.numel() != B + 1:
            raise ValueError("query_start_loc must have B + 1 = %d entries" % (B + 1))
    else:
        if q_len < 1 or BQ % q_len:
            raise ValueError("q must hold q_len rows per sequence")
        B = BQ // q_len
    _check_int4_decode_args(q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, out, q_len, ragged)
    nb, bs, Hk = k_cache.shape[0], k_cache.shape[1], k_cache.shape[2]
    if out is None:
        out = torch.empty((BQ, Hq, D), dtype=out_dtype or torch.float32, device=q.device)
    _need(out, "out")
    mq = ragged or q_len > 1
    if workspace is None and mq:
        probe = ScoreMods(0, 0.0, None, None, int(q_len), None, _ptr(query_start_loc), int(BQ))
        need = kvq_decode_int4_mods_workspace_bytes(B, Hq, Hk, D, num_splits, probe)
        workspace = torch.empty((max(need, 16),), dtype=torch.uint8, device=q.device)
    else:
        workspace = _workspace(workspace, B, Hq, Hk, D, num_splits, q.device)
    if lse_out is not None:
        _need(lse_out, "lse_out", torch.float32)
        if tuple(lse_out.shape) != (BQ, Hq):
            raise ValueError("lse_out must be [%d, %d]" % (BQ, Hq))
    if (sliding_window or softcap or sinks is not None or alibi_slopes is not None or mq
            or lse_out is not None):
        for t, n in ((sinks, "sinks"), (alibi_slopes, "alibi_slopes")):
            if t is not None:
                _need(t, n, torch.float32)
                if t.numel() != Hq:
                    raise ValueError("%s must have Hq = %d entries" % (n, Hq))
        mods = ScoreMods(int(sliding_window), float(softcap), _ptr(sinks), _ptr(alibi_slopes), int(q_len),
                         _ptr(lse_out), _ptr(query_start_loc), int(BQ))
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
    _check_int4_decode_args(q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, out)
    B, Hq, D = q.shape
    nb, bs, Hk = k_cache.shape[0], k_cache.shape[1], k_cache.shape[2]
    _check(lib().kvq_decode_int4_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
                                         _ptr(block_table), block_table.shape[1], _ptr(seq_lens), _ptr(rht_signs),
                                         float(softmax_scale), num_splits, _ptr(out), _out_code(out.dtype),
                                         B, Hq, Hk, D, bs, nb, _stream(stream)),
           "kvq_decode_int4_noalloc")
    return out


def kvq_decode_tq(q, kv_cache, value_bits, block_table, seq_lens, attn_scale, out=None, workspace=None,
                  num_splits=0, stream=None, lse_out=None):
    """TurboQuant FP8-key decode: q [B, Hq, D] fp32, kv_cache [nb, 16, Hk, slot_bytes] uint8.
    lse_out: an fp32 [B, Hq] tensor that receives each row's log-sum-exp (kvq_decode_tq_lse), or None."""
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
    if lse_out is not None:
        _need(lse_out, "lse_out", torch.float32)
        if tuple(lse_out.shape) != (B, Hq):
            raise ValueError("lse_out must be [%d, %d]" % (B, Hq))
        _check(lib().kvq_decode_tq_lse(_ptr(q), _ptr(kv_cache), slot_bytes, value_bits, _ptr(block_table),
                                       block_table.shape[1], _ptr(seq_lens), float(attn_scale), num_splits,
                                       _ptr(workspace), workspace.numel(), _ptr(out), _ptr(lse_out), B, Hq, Hk,
                                       D, bs, nb, _stream(stream)),
               "kvq_decode_tq_lse")
        return out
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


def kvq_debug_set_wait(wait_limit_ns=0, withhold_stage=-1):
    """Error-path tests only: the decode's bounded-wait limit (0: default) and a ring stage the next
    INT4 decode call withholds in its first CTA (kvq_debug_set_wait in include/kvq.h)."""
    _check(lib().kvq_debug_set_wait(int(wait_limit_ns), int(withhold_stage)), "kvq_debug_set_wait")


def kvq_device_error(stream=None):
    """(status, flags): synchronizes the stream, reads and clears the device-side index flags."""
    flags = ctypes.c_uint32(0)
    st = lib().kvq_device_error(_stream(stream), ctypes.byref(flags))
    return int(st), int(flags.value)


# ----------------------------------------------------------------------------------------------
# Prepared calls: the tensors that stay the same from step to step (caches, scales, block table,
# lengths, rotation signs, workspace) are checked once and their pointers packed once; each call
# checks and passes only the per-step tensors. For serving loops whose buffers live across steps.
# ----------------------------------------------------------------------------------------------
class Int4Writer:
    """kvq_write_int4 into fixed caches: writer(key, value, slot_mapping[, stream])."""

    def __init__(self, k_cache, v_cache, k_scale, v_scale, rht_signs=None):
        for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
            _need(t, n, torch.uint8)
        for t, n in ((k_scale, "k_scale"), (v_scale, "v_scale")):
            _need(t, n, torch.float32)
        if rht_signs is not None:
            _need(rht_signs, "rht_signs", torch.float32)
        nb, bs, Hk, half = k_cache.shape
        if tuple(v_cache.shape) != tuple(k_cache.shape) or tuple(k_scale.shape) != (nb, bs, Hk) or \
                tuple(v_scale.shape) != (nb, bs, Hk):
            raise ValueError("cache / scale shapes disagree")
        self.kv_shape = (Hk, 2 * half)
        self._keep = (k_cache, v_cache, k_scale, v_scale, rht_signs)
        self._fn = lib().kvq_write_int4
        self._caches = (k_cache.data_ptr(), v_cache.data_ptr(), k_scale.data_ptr(), v_scale.data_ptr())
        self._tail = (_ptr(rht_signs),)
        self._dims = (Hk, 2 * half, bs, nb)

    def __call__(self, key, value, slot_mapping, stream=None):
        if key.dtype != torch.bfloat16 or value.dtype != torch.bfloat16 or not key.is_cuda or not value.is_cuda:
            raise TypeError("key / value must be CUDA bf16 tensors")
        if key.shape[1:] != self.kv_shape or value.shape != key.shape or key.stride(-1) != 1 or value.stride(-1) != 1:
            raise ValueError("key / value must be [T, %d, %d] with a contiguous last dim" % self.kv_shape)
        if slot_mapping.dtype != torch.int64 or not slot_mapping.is_cuda or not slot_mapping.is_contiguous() or \
                slot_mapping.numel() != key.shape[0]:
            raise ValueError("slot_mapping must be a contiguous CUDA int64 [T] tensor")
        Hk, D, bs, nb = self._dims
        _check(self._fn(key.data_ptr(), value.data_ptr(), key.stride(0), key.stride(1), value.stride(0),
                        value.stride(1), *self._caches, slot_mapping.data_ptr(), *self._tail, key.shape[0], Hk, D,
                        bs, nb, _stream(stream)), "kvq_write_int4")


class Int4Decoder:
    """kvq_decode_int4 over fixed caches, block table, lengths and workspace:
    decoder(q, out[, stream]) with q [B, Hq, D] bf16 and out [B, Hq, D] (bf16 / f16 / f32).
    The block table's and lengths' contents may change between calls; their buffers may not."""

    def __init__(self, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, rht_signs, softmax_scale, Hq,
                 num_splits=0, workspace=None):
        for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
            _need(t, n, torch.uint8)
        for t, n in ((k_scale, "k_scale"), (v_scale, "v_scale")):
            _need(t, n, torch.float32)
        _need(block_table, "block_table", torch.int32)
        _need(seq_lens, "seq_lens", torch.int32)
        if rht_signs is not None:
            _need(rht_signs, "rht_signs", torch.float32)
        nb, bs, Hk, half = k_cache.shape
        D = 2 * half
        B = block_table.shape[0]
        if tuple(v_cache.shape) != tuple(k_cache.shape) or tuple(k_scale.shape) != (nb, bs, Hk) or \
                tuple(v_scale.shape) != (nb, bs, Hk) or seq_lens.numel() != B or block_table.dim() != 2:
            raise ValueError("cache / scale / table shapes disagree")
        if workspace is None:
            workspace = decode_workspace(B, Hq, Hk, D, num_splits, device=k_cache.device)
        _need(workspace, "workspace", torch.uint8)
        self.q_shape = (B, Hq, D)
        self._keep = (k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, rht_signs, workspace)
        self._fn = lib().kvq_decode_int4
        self._head = (k_cache.data_ptr(), v_cache.data_ptr(), k_scale.data_ptr(), v_scale.data_ptr(),
                      block_table.data_ptr(), block_table.shape[1], seq_lens.data_ptr(), _ptr(rht_signs),
                      float(softmax_scale), int(num_splits), workspace.data_ptr(), workspace.numel())
        self._dims = (B, Hq, Hk, D, bs, nb)

    def __call__(self, q, out, stream=None):
        if q.dtype != torch.bfloat16 or not q.is_cuda or not q.is_contiguous() or tuple(q.shape) != self.q_shape:
            raise ValueError("q must be a contiguous CUDA bf16 tensor of shape %s" % (self.q_shape,))
        if not out.is_cuda or not out.is_contiguous() or tuple(out.shape) != self.q_shape:
            raise ValueError("out must be a contiguous CUDA tensor of shape %s" % (self.q_shape,))
        _check(self._fn(q.data_ptr(), *self._head, out.data_ptr(), _out_code(out.dtype), *self._dims,
                        _stream(stream)), "kvq_decode_int4")
        return out


def kvq_copy(dst, src, stream=None):
    """Copy src into dst (the same number of bytes) with the library's copy kernel on `stream`.
    Each tensor may be a CUDA tensor or a pinned CPU tensor (read or written by the SMs over the
    chip-to-chip link), so inside a captured step the copies are kernel nodes like the rest.
    Both contiguous, 16-byte aligned, a multiple of 16 bytes. Returns dst."""
    for t, n in ((dst, "dst"), (src, "src")):
        if not isinstance(t, torch.Tensor):
            raise TypeError("%s must be a tensor" % n)
        if not t.is_contiguous():
            raise ValueError("%s must be contiguous" % n)
        if not t.is_cuda and not t.is_pinned():
            raise ValueError("%s must be a CUDA tensor or a pinned CPU tensor" % n)
    nbytes = dst.numel() * dst.element_size()
    if src.numel() * src.element_size() != nbytes:
        raise ValueError("dst and src differ in size: %d vs %d bytes" % (nbytes, src.numel() * src.element_size()))
    _check(lib().kvq_copy_async(_ptr(dst), _ptr(src), nbytes, _stream(stream)), "kvq_copy_async")
    return dst


class CapturedStep:
    """A fixed sequence of calls on one stream, replayed as one CUDA graph.

    step = CapturedStep(fn, stream) runs fn() once eagerly (which also sets the kernels' one-time
    attributes), then captures fn() on `stream`; step() replays the capture on that stream,
    asynchronously. fn must only enqueue work on `stream` (library calls, tensor copies between
    fixed buffers -- e.g. a pinned host staging buffer to its device twin and an output back to
    pinned memory); the buffers it touches keep their addresses, and their contents at replay
    time are what the replay reads. A decode step whose inputs change from step to step copies
    them into the same buffers before each replay, or inside fn."""

    def __init__(self, fn, stream):
        self.stream = stream
        with torch.cuda.stream(stream):
            fn()
        stream.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=stream):
            fn()
        self._keep = fn

    def __call__(self):
        with torch.cuda.stream(self.stream):
            self.graph.replay()
