"""ctypes binding of libkvd.so — argument marshalling only.

Every function here has the name of the C entry point it calls and does
nothing but turn torch tensors into device pointers, pick the current CUDA
stream and raise ``KvdError`` on a non-OK status.  All computation happens in
the CUDA kernels behind the C ABI; there is no fallback path.
"""

from __future__ import annotations

import ctypes
import os

KVD_OK, KVD_ERR_INVALID, KVD_ERR_UNSUPPORTED, KVD_ERR_NOMEM, KVD_ERR_CUDA, KVD_ERR_OOB, KVD_ERR_TIMEOUT = range(7)
KVD_BF16, KVD_FP8_E4M3, KVD_F32, KVD_FP8_E5M2, KVD_MIXED, KVD_INT4, KVD_INT2, KVD_ANGLE = 0, 1, 2, 3, 4, 5, 6, 7
KVD_EARLY_START = 1   # kvd_decode_attn flags
KVD_PLANNED = 2

SYMBOLS = [
    "kvd_status_string", "kvd_pool_bytes", "kvd_pool_create", "kvd_pool_destroy", "kvd_append_kv",
    "kvd_decode_workspace_bytes", "kvd_decode_attn", "kvd_combine_splits", "kvd_accum_scores",
    "kvd_get_device_error", "kvd_selftest_wait_timeout", "kvd_decode_attn_noalloc",
    "kvd_tier_bytes", "kvd_pool_attach_host_tier", "kvd_tier_prefetch", "kvd_tier_plan", "kvd_tier_move",
    "kvd_tier_reassign", "kvd_measure_read_stream", "kvd_pool_set_block_formats", "kvd_decode_plan",
]
NOALLOC_SCRATCH_BYTES = 16 << 20


class KvdError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn}: {msg} (status {status})")
        self.status = status


class ScoresDesc(ctypes.Structure):
    _fields_ = [("scores", ctypes.c_void_p), ("scores_stride", ctypes.c_int64), ("inv_LH", ctypes.c_float)]


class PoolDesc(ctypes.Structure):
    _fields_ = [("num_layers", ctypes.c_int32), ("n_kv", ctypes.c_int32), ("d_h", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("num_blocks", ctypes.c_int64), ("kv_dtype", ctypes.c_int32),
                ("group_size", ctypes.c_int32)]


_lib = None


def lib_path() -> str:
    return os.path.join(os.path.dirname(os.path.abspath(__file__)), "_build", "libkvd.so")


def load(build_if_missing: bool = True):
    """Load libkvd.so (building it first if absent).  Raises if it cannot be built or loaded."""
    global _lib
    if _lib is not None:
        return _lib
    path = lib_path()
    if build_if_missing:
        from . import build as _build
        _build.build()
    if not os.path.exists(path):
        raise RuntimeError(f"libkvd.so not found at {path}; build it with paged_gqa_decode_kvd_gb300.build")
    lib = ctypes.CDLL(path)
    P, i32, i64, sz, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
    lib.kvd_status_string.restype = ctypes.c_char_p
    lib.kvd_status_string.argtypes = [i32]
    lib.kvd_pool_bytes.restype = i32
    lib.kvd_pool_bytes.argtypes = [ctypes.POINTER(PoolDesc), ctypes.POINTER(sz), ctypes.POINTER(sz)]
    lib.kvd_pool_create.restype = i32
    lib.kvd_pool_create.argtypes = [ctypes.POINTER(PoolDesc), P, sz, ctypes.POINTER(P)]
    lib.kvd_pool_destroy.restype = None
    lib.kvd_pool_destroy.argtypes = [P]
    lib.kvd_tier_bytes.restype = i32
    lib.kvd_tier_bytes.argtypes = [ctypes.POINTER(PoolDesc), i64, ctypes.POINTER(sz), ctypes.POINTER(sz)]
    lib.kvd_pool_attach_host_tier.restype = i32
    lib.kvd_pool_attach_host_tier.argtypes = [P, P, sz, P, sz, i64]
    lib.kvd_tier_prefetch.restype = i32
    lib.kvd_tier_prefetch.argtypes = [P, i32, P]
    lib.kvd_tier_plan.restype = i32
    lib.kvd_tier_plan.argtypes = [P, i64, P, i32, i32, i32, i32, i32, P, P, P]
    lib.kvd_tier_move.restype = i32
    lib.kvd_tier_move.argtypes = [P, P, P, i32, P]
    lib.kvd_tier_reassign.restype = i32
    lib.kvd_tier_reassign.argtypes = [i64, i64, P, P, i32, i32, P, P, P, P, P, P, P, P]
    lib.kvd_append_kv.restype = i32
    lib.kvd_append_kv.argtypes = [P, i32, P, P, P, i32, P]
    lib.kvd_decode_workspace_bytes.restype = i32
    lib.kvd_decode_workspace_bytes.argtypes = [P, i32, i32, i32, i32, ctypes.POINTER(i32), ctypes.POINTER(sz)]
    lib.kvd_decode_attn.restype = i32
    lib.kvd_decode_attn.argtypes = [P, i32, P, i32, P, P, P, i32, P, i32, i32, i32, P, f32, P, sz, P, i32, P, P, i64,
                                    P, ctypes.c_uint, P]
    lib.kvd_combine_splits.restype = i32
    lib.kvd_combine_splits.argtypes = [P, P, P, P, i32, i32, i32, i32, P, i32, P, P]
    lib.kvd_accum_scores.restype = i32
    lib.kvd_accum_scores.argtypes = [P, i64, P, P, i32, i32, f32, P, i64, P]
    lib.kvd_get_device_error.restype = i32
    lib.kvd_get_device_error.argtypes = [P, P, ctypes.POINTER(ctypes.c_int32)]
    lib.kvd_selftest_wait_timeout.restype = i32
    lib.kvd_selftest_wait_timeout.argtypes = [P, i64, P]
    lib.kvd_decode_attn_noalloc.restype = i32
    lib.kvd_decode_attn_noalloc.argtypes = [P, i32, P, i32, P, P, P, i32, P, i32, i32, i32, P, f32, P, i32, P, P,
                                            i64, P, ctypes.c_uint, P]
    lib.kvd_pool_set_block_formats.restype = i32
    lib.kvd_pool_set_block_formats.argtypes = [P, P, i64]
    lib.kvd_decode_plan.restype = i32
    lib.kvd_decode_plan.argtypes = [P, i32, P, i32, P, i32, i32, i32, P, P, sz, P]
    lib.kvd_measure_read_stream.restype = i32
    lib.kvd_measure_read_stream.argtypes = [P, sz, P, sz, P]
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().kvd_status_string(status).decode()


def _check(fn: str, status: int):
    if status != KVD_OK:
        raise KvdError(fn, status, status_string(status))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def kvd_pool_bytes(num_layers: int, n_kv: int, num_blocks: int, kv_dtype: int, d_h: int = 128, block_size: int = 16,
                   group_size: int = 0):
    """(pool_bytes, kv_bytes) of a pool: buffer size to allocate, and closed-form K/V bytes; host only.
    group_size: values per scale group of a KVD_INT4 / KVD_INT2 pool (32, 64 or 128)."""
    d = PoolDesc(num_layers, n_kv, d_h, block_size, num_blocks, kv_dtype, group_size)
    pool, kv = ctypes.c_size_t(), ctypes.c_size_t()
    _check("kvd_pool_bytes", load().kvd_pool_bytes(ctypes.byref(d), ctypes.byref(pool), ctypes.byref(kv)))
    return pool.value, kv.value


def kvd_tier_bytes(num_layers: int, n_kv: int, num_blocks: int, kv_dtype: int, host_blocks: int, d_h: int = 128,
                   block_size: int = 16):
    """(host_bytes, staging_bytes) of a host tier of host_blocks blocks; host only."""
    d = PoolDesc(num_layers, n_kv, d_h, block_size, num_blocks, kv_dtype)
    h, st = ctypes.c_size_t(), ctypes.c_size_t()
    _check("kvd_tier_bytes", load().kvd_tier_bytes(ctypes.byref(d), int(host_blocks), ctypes.byref(h), ctypes.byref(st)))
    return h.value, st.value


def kvd_pool_attach_host_tier(handle, host_mem, staging, host_blocks):
    """host_mem: pinned host tensor; staging: device tensor, or None for direct reads (both
    caller-owned, sized by kvd_tier_bytes)."""
    _check("kvd_pool_attach_host_tier", load().kvd_pool_attach_host_tier(
        handle, _ptr(host_mem), 0 if host_mem is None else host_mem.numel() * host_mem.element_size(),
        _ptr(staging), 0 if staging is None else staging.numel() * staging.element_size(), int(host_blocks)))


def kvd_tier_prefetch(handle, layer, stream=None):
    _check("kvd_tier_prefetch", load().kvd_tier_prefetch(handle, int(layer), _stream(stream)))


def kvd_tier_plan(scores, seq_lens, max_blocks_per_seq, protect_prompt, protect_recent, t1_blocks, tier,
                  importance=None, stream=None):
    """Tier plan: tier (int8 [B][max_blocks], device) gets 1 for the t1_blocks least important
    unprotected blocks of each request, 0 for the others, -1 past the context; importance
    (f32, same shape, optional) gets the per-block score sums.  scores: f32 [B][stride]."""
    _check("kvd_tier_plan", load().kvd_tier_plan(_ptr(scores), int(scores.stride(0)), _ptr(seq_lens),
                                                 int(seq_lens.shape[0]), int(max_blocks_per_seq),
                                                 int(protect_prompt), int(protect_recent), int(t1_blocks),
                                                 _ptr(importance), _ptr(tier), _stream(stream)))


def kvd_tier_move(handle, from_ids, to_ids, stream=None):
    """Copy every layer's records of physical block from_ids[i] to to_ids[i] (int32 device tensors)."""
    n = int(from_ids.numel())
    if int(to_ids.numel()) != n:
        raise ValueError("from_ids and to_ids differ in length")
    _check("kvd_tier_move", load().kvd_tier_move(handle, _ptr(from_ids), _ptr(to_ids), n, _stream(stream)))


def kvd_tier_reassign(num_blocks, host_blocks, tier, block_table, hbm_free, hbm_free_n, host_free, host_free_n,
                      retain_mask=None):
    """Host-side reassignment (numpy arrays, updated in place: block_table, hbm_free, host_free,
    retain_mask).  Returns (status, from_ids, to_ids, hbm_free_n, host_free_n); raises only for
    KVD_ERR_INVALID."""
    import numpy as np

    tier = np.ascontiguousarray(tier, dtype=np.int8)
    for a, dt in ((block_table, np.int32), (hbm_free, np.int32), (host_free, np.int32)):
        if a.dtype != dt or not a.flags.c_contiguous:
            raise TypeError("block_table, hbm_free and host_free must be contiguous int32 arrays")
    if retain_mask is not None and (retain_mask.dtype != np.uint16 or not retain_mask.flags.c_contiguous):
        raise TypeError("retain_mask must be a contiguous uint16 array")
    if tier.shape != block_table.shape or tier.ndim != 2:
        raise ValueError("tier and block_table must both be [batch][max_blocks_per_seq]")
    if hbm_free.size < num_blocks or host_free.size < host_blocks:
        raise ValueError("free lists need capacity num_blocks and host_blocks")
    batch, mb = block_table.shape
    frm = np.empty(max(1, batch * mb), np.int32)
    to = np.empty(max(1, batch * mb), np.int32)
    hn, tn, n = ctypes.c_int32(int(hbm_free_n)), ctypes.c_int32(int(host_free_n)), ctypes.c_int32()
    ptr = lambda a: None if a is None else a.ctypes.data_as(ctypes.c_void_p)
    st = load().kvd_tier_reassign(int(num_blocks), int(host_blocks), ptr(tier), ptr(block_table), batch, mb,
                                  ptr(hbm_free), ctypes.byref(hn), ptr(host_free), ctypes.byref(tn),
                                  ptr(retain_mask), ptr(frm), ptr(to), ctypes.byref(n))
    if st == KVD_ERR_INVALID:
        raise KvdError("kvd_tier_reassign", st, status_string(st))
    return st, frm[:n.value].copy(), to[:n.value].copy(), hn.value, tn.value


def kvd_pool_create(num_layers, n_kv, num_blocks, kv_dtype, mem, d_h=128, block_size=16, group_size=0):
    """Wrap a caller-owned device tensor (any dtype, pool_bytes long) as a pool; returns the handle (c_void_p)."""
    d = PoolDesc(num_layers, n_kv, d_h, block_size, num_blocks, kv_dtype, group_size)
    h = ctypes.c_void_p()
    n = mem.numel() * mem.element_size()
    _check("kvd_pool_create", load().kvd_pool_create(ctypes.byref(d), _ptr(mem), n, ctypes.byref(h)))
    return h


def kvd_pool_set_block_formats(handle, block_fmt):
    """Mixed pool: block_fmt (uint8 device tensor, one KVD_BF16 / KVD_FP8_E4M3 / KVD_FP8_E5M2
    code per physical block) gives every block's storage format; the pool reads it on every
    later append and decode, so keep the tensor alive."""
    _check("kvd_pool_set_block_formats", load().kvd_pool_set_block_formats(handle, _ptr(block_fmt),
                                                                           int(block_fmt.numel())))


def kvd_pool_destroy(handle):
    load().kvd_pool_destroy(handle)


def kvd_append_kv(handle, layer, k_new, v_new, slot_mapping, stream=None):
    n = 0 if k_new is None else k_new.shape[0]
    _check("kvd_append_kv", load().kvd_append_kv(handle, layer, _ptr(k_new), _ptr(v_new), _ptr(slot_mapping), n,
                                                 _stream(stream)))


def kvd_decode_workspace_bytes(handle, n_q, batch, max_seq_len, num_splits=0):
    s, b = ctypes.c_int(), ctypes.c_size_t()
    _check("kvd_decode_workspace_bytes",
           load().kvd_decode_workspace_bytes(handle, n_q, batch, max_seq_len, num_splits, ctypes.byref(s),
                                             ctypes.byref(b)))
    return s.value, b.value


def _scores_desc(scores, inv_LH):
    if scores is None:
        return None
    return ctypes.byref(ScoresDesc(scores.data_ptr(), scores.shape[-1], float(inv_LH)))


def kvd_decode_plan(handle, n_q, block_table, seq_lens, max_seq_len, workspace, num_splits=0, retain_mask=None,
                    stream=None):
    """The step plan into the workspace's plan region, for kvd_decode_attn(..., planned=True) calls that
    share block_table, seq_lens and retain_mask."""
    _check("kvd_decode_plan", load().kvd_decode_plan(
        handle, int(n_q), _ptr(block_table), block_table.shape[1], _ptr(seq_lens), int(seq_lens.shape[0]),
        int(max_seq_len), int(num_splits), _ptr(retain_mask), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def kvd_decode_attn(handle, layer, q, block_table, seq_lens, max_seq_len, workspace, out, num_splits=0,
                    retain_mask=None, softmax_scale=None, lse_out=None, logits_out=None, k_new=None, v_new=None,
                    scores=None, inv_LH=None, early_start=False, planned=False, stream=None):
    batch, n_q, d_h = q.shape
    if softmax_scale is None:
        softmax_scale = d_h ** -0.5
    out_dtype = KVD_F32 if out is not None and out.element_size() == 4 else KVD_BF16
    lstride = 0 if logits_out is None else logits_out.shape[-1]
    _check("kvd_decode_attn", load().kvd_decode_attn(
        handle, layer, _ptr(q), n_q, _ptr(k_new), _ptr(v_new), _ptr(block_table), block_table.shape[1],
        _ptr(seq_lens), batch,
        int(max_seq_len), int(num_splits), _ptr(retain_mask), float(softmax_scale), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(out), out_dtype, _ptr(lse_out), _ptr(logits_out),
        lstride, _scores_desc(scores, inv_LH), (KVD_EARLY_START if early_start else 0) | (KVD_PLANNED if planned else 0),
        _stream(stream)))


def kvd_combine_splits(part_o, part_lse, unit_first, unit_count, batch, n_q, n_kv, out, lse_out=None, stream=None):
    out_dtype = KVD_F32 if out.element_size() == 4 else KVD_BF16
    _check("kvd_combine_splits", load().kvd_combine_splits(
        _ptr(part_o), _ptr(part_lse), _ptr(unit_first), _ptr(unit_count), batch, n_q, n_kv, 128, _ptr(out),
        out_dtype, _ptr(lse_out), _stream(stream)))


def kvd_accum_scores(logits, lse, seq_lens, inv_LH, scores, stream=None):
    batch, n_q, lstride = logits.shape
    _check("kvd_accum_scores", load().kvd_accum_scores(
        _ptr(logits), lstride, _ptr(lse), _ptr(seq_lens), batch, n_q, float(inv_LH), _ptr(scores),
        scores.shape[-1], _stream(stream)))


def kvd_get_device_error(handle, stream=None) -> int:
    c = ctypes.c_int32()
    _check("kvd_get_device_error", load().kvd_get_device_error(handle, _stream(stream), ctypes.byref(c)))
    return c.value


def kvd_selftest_wait_timeout(handle, timeout_ns, stream=None):
    _check("kvd_selftest_wait_timeout", load().kvd_selftest_wait_timeout(handle, int(timeout_ns), _stream(stream)))


def kvd_decode_attn_noalloc(handle, layer, q, block_table, seq_lens, max_seq_len, out, num_splits=0,
                            retain_mask=None, softmax_scale=None, lse_out=None, logits_out=None, k_new=None,
                            v_new=None, scores=None, inv_LH=None, early_start=False, stream=None):
    """kvd_decode_attn without a workspace argument: the library's fixed device scratch array is used."""
    batch, n_q, d_h = q.shape
    if softmax_scale is None:
        softmax_scale = d_h ** -0.5
    out_dtype = KVD_F32 if out is not None and out.element_size() == 4 else KVD_BF16
    lstride = 0 if logits_out is None else logits_out.shape[-1]
    _check("kvd_decode_attn_noalloc", load().kvd_decode_attn_noalloc(
        handle, layer, _ptr(q), n_q, _ptr(k_new), _ptr(v_new), _ptr(block_table), block_table.shape[1],
        _ptr(seq_lens), batch,
        int(max_seq_len), int(num_splits), _ptr(retain_mask), float(softmax_scale), _ptr(out), out_dtype,
        _ptr(lse_out), _ptr(logits_out), lstride, _scores_desc(scores, inv_LH),
        KVD_EARLY_START if early_start else 0, _stream(stream)))


def kvd_measure_read_stream(buf, sink, stream=None):
    """Read every byte of the device tensor buf once (read-only HBM stream); sink: device
    tensor of at least 32 KiB that receives one word per CTA."""
    _check("kvd_measure_read_stream", load().kvd_measure_read_stream(
        _ptr(buf), buf.numel() * buf.element_size(), _ptr(sink), sink.numel() * sink.element_size(),
        _stream(stream)))
