"""ctypes wrapper over the C oracle (``kvd_oracle.c``) — TEST INFRASTRUCTURE.

Every array crossing into C is a contiguous numpy array of the C type.  The
oracle owns its pool (``OraclePool``) in its own plain layout
[num_blocks][n_kv][block_size][d_h]; it never reads the CUDA library's pool.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvd_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "libkvd_oracle.so")
_lock = threading.Lock()
_lib = None

ERR_INDEX = 1
ERR_EMPTY = 2


def lib_path() -> str:
    return _LIB


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FMA contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            i32, i64, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_double
            lib.kvdo_e4m3_decode.restype = f64
            lib.kvdo_e4m3_decode.argtypes = [ctypes.c_uint8]
            lib.kvdo_e4m3_encode.restype = ctypes.c_uint8
            lib.kvdo_e4m3_encode.argtypes = [ctypes.c_float]
            lib.kvdo_e4m3_decode_array.argtypes = [P, i64, P]
            lib.kvdo_e4m3_encode_array.argtypes = [P, i64, P]
            lib.kvdo_quantize_rows.argtypes = [P, i64, i32, P, P]
            lib.kvdo_append.restype = i32
            lib.kvdo_append.argtypes = [i32, i32, i32, i64, i32, P, P, P, i64, P, P, P, P, P, P]
            lib.kvdo_dequant_pool.argtypes = [P, P, i64, i32, P]
            lib.kvdo_decode.restype = i32
            lib.kvdo_decode.argtypes = [i32, i32, i32, i32, i64, P, P, P, P, i32, P, i32, P, f64,
                                        P, P, P, P, i64]
            lib.kvdo_score_update.argtypes = [P, i32, i32, i32, P, i64, P]
            lib.kvdo_tier_plan.argtypes = [P, i64, P, i32, i32, i32, i32, i32, i32, P, P]
            lib.kvdo_e5m2_decode.restype = f64
            lib.kvdo_e5m2_decode.argtypes = [ctypes.c_uint8]
            lib.kvdo_e5m2_encode.restype = ctypes.c_uint8
            lib.kvdo_e5m2_encode.argtypes = [ctypes.c_float]
            lib.kvdo_e5m2_decode_array.argtypes = [P, i64, P]
            lib.kvdo_e5m2_encode_array.argtypes = [P, i64, P]
            lib.kvdo_quantize_rows_fmt.argtypes = [P, i64, i32, i32, P, P]
            lib.kvdo_append_mixed.restype = i32
            lib.kvdo_append_mixed.argtypes = [i32, i32, i32, i64, P, P, P, P, i64, P, P, P, P, P, P]
            lib.kvdo_angle_key_rows.argtypes = [P, i64, i32, P, P, P]
            lib.kvdo_angle_query.argtypes = [P, i64, i32, P]
            lib.kvdo_append_angle.restype = i32
            lib.kvdo_append_angle.argtypes = [i32, i32, i32, i64, P, P, P, i64, P, P, P, P, P]
            lib.kvdo_round_half_sat.restype = f64
            lib.kvdo_round_half_sat.argtypes = [f64]
            lib.kvdo_round_half_sat_array.argtypes = [P, i64, P]
            lib.kvdo_quantize_rows_lowbit.argtypes = [P, i64, i32, i32, i32, P, P, P]
            lib.kvdo_append_lowbit.restype = i32
            lib.kvdo_append_lowbit.argtypes = [i32, i32, i32, i64, i32, i32, P, P, P, i64, P, P, P, P, P, P, P, P]
            _lib = lib
    return _lib


def _c(a, dtype):
    return np.asarray(a, dtype=dtype, order="C")


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def e4m3_decode(codes) -> np.ndarray:
    """float64 value of each uint8 E4M3 code."""
    c = _c(codes, np.uint8)
    out = np.empty(c.shape, np.float64)
    _load().kvdo_e4m3_decode_array(_p(c), c.size, _p(out))
    return out


def e4m3_encode(y) -> np.ndarray:
    """Nearest (ties to even) saturating E4M3 code of each float32 value."""
    a = _c(y, np.float32)
    out = np.empty(a.shape, np.uint8)
    _load().kvdo_e4m3_encode_array(_p(a), a.size, _p(out))
    return out


FMT_BF16, FMT_E4M3, FMT_E5M2 = 0, 1, 2   # block precision codes of a mixed pool


def e5m2_decode(codes) -> np.ndarray:
    c = _c(codes, np.uint8)
    out = np.empty(c.shape, np.float64)
    _load().kvdo_e5m2_decode_array(_p(c), c.size, _p(out))
    return out


def e5m2_encode(y) -> np.ndarray:
    a = _c(y, np.float32)
    out = np.empty(a.shape, np.uint8)
    _load().kvdo_e5m2_encode_array(_p(a), a.size, _p(out))
    return out


def quantize_rows_fmt(x, fmt: int) -> tuple[np.ndarray, np.ndarray]:
    """Per-row absmax quantise of float32 [..., d] to E4M3 (fmt 1) or E5M2 (fmt 2)."""
    a = _c(x, np.float32)
    d = a.shape[-1]
    rows = a.size // d
    codes = np.empty(a.shape, np.uint8)
    scales = np.empty(a.shape[:-1], np.float32)
    _load().kvdo_quantize_rows_fmt(_p(a), rows, d, int(fmt), _p(codes), _p(scales))
    return codes, scales


def quantize_rows(x) -> tuple[np.ndarray, np.ndarray]:
    """Per-row absmax FP8 quantise of float32 [..., d]: (codes [..., d] uint8, scales [...] float32)."""
    a = _c(x, np.float32)
    d = a.shape[-1]
    rows = a.size // d
    codes = np.empty(a.shape, np.uint8)
    scales = np.empty(a.shape[:-1], np.float32)
    _load().kvdo_quantize_rows(_p(a), rows, d, _p(codes), _p(scales))
    return codes, scales


def round_half_sat(x) -> np.ndarray:
    """Nearest IEEE half-precision value of each float64, ties to even, saturated at ±65,504."""
    a = _c(x, np.float64)
    out = np.empty(a.shape, np.float64)
    _load().kvdo_round_half_sat_array(_p(a), a.size, _p(out))
    return out


def quantize_rows_lowbit(x, bits: int, group: int) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Low-bit group quantise of float32 [..., d]: (codes [..., d] uint8 in [0, 2^bits - 1],
    scales [..., d/group] float32, zeros [..., d/group] float32), value = code·scale + zero."""
    a = _c(x, np.float32)
    d = a.shape[-1]
    rows = a.size // d
    codes = np.empty(a.shape, np.uint8)
    scales = np.empty(a.shape[:-1] + (d // group,), np.float32)
    zeros = np.empty(a.shape[:-1] + (d // group,), np.float32)
    _load().kvdo_quantize_rows_lowbit(_p(a), rows, d, int(bits), int(group), _p(codes), _p(scales), _p(zeros))
    return codes, scales, zeros


def angle_key_rows(x) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Angle-domain key rows of float32 [..., d]: (E4M3 direction codes [..., d], the logit factor
    w = fp32(r̃ / ||d||) [...], the half-precision radius r̃ [...]); the key attention sees is w·d."""
    a = _c(x, np.float32)
    d = a.shape[-1]
    rows = a.size // d
    codes = np.empty(a.shape, np.uint8)
    w = np.empty(a.shape[:-1], np.float32)
    r = np.empty(a.shape[:-1], np.float32)
    _load().kvdo_angle_key_rows(_p(a), rows, d, _p(codes), _p(w), _p(r))
    return codes, w, r


def angle_query(q) -> np.ndarray:
    """Each row q (float32 [..., d]) as (||q|| / ||d_q||)·d_q in fp64, d_q its E4M3 direction code's
    values: the query of an angle-domain logit."""
    a = _c(q, np.float32)
    out = np.empty(a.shape, np.float64)
    _load().kvdo_angle_query(_p(a), a.size // a.shape[-1], a.shape[-1], _p(out))
    return out


class OraclePool:
    """The oracle's own paged pool for one layer: [num_blocks][n_kv][block_size][d_h].

    block_fmt (uint8 [num_blocks], optional) makes it a mixed-precision pool: block p holds
    BF16 values (0), E4M3 codes (1) or E5M2 codes (2), each 8-bit row with its own scale.
    lowbit = (bits, group) makes it a low-bit pool: every row of K and V holds bits-wide codes
    with a scale and a zero point per group of `group` values.
    angle=True makes it an angle-domain pool: K rows hold E4M3 direction codes with the factor
    w = r̃/||d|| in k_scales (radius r̃ in k_radius), V rows FP8; decode it with a query passed
    through angle_query."""

    def __init__(self, num_blocks: int, n_kv: int, d_h: int, block_size: int = 16, fp8: bool = False,
                 block_fmt=None, lowbit=None, angle: bool = False):
        self.num_blocks, self.n_kv, self.d_h, self.block_size, self.fp8 = num_blocks, n_kv, d_h, block_size, fp8
        shape = (num_blocks, n_kv, block_size, d_h)
        self.block_fmt = None
        self.lowbit = None
        self.angle = bool(angle)
        if self.angle:
            self.fp8 = True
            self.k_codes = np.zeros(shape, np.uint8)
            self.v_codes = np.zeros(shape, np.uint8)
            self.k_scales = np.zeros(shape[:-1], np.float32)
            self.v_scales = np.ones(shape[:-1], np.float32)
            self.k_radius = np.zeros(shape[:-1], np.float32)
            self.k = self.v = None
        elif lowbit is not None:
            self.lowbit = (int(lowbit[0]), int(lowbit[1]))
            ng = d_h // self.lowbit[1]
            assert ng * self.lowbit[1] == d_h and self.lowbit[0] in (2, 4)
            self.k = np.zeros(shape, np.float64)
            self.v = np.zeros(shape, np.float64)
            self.k_codes = np.zeros(shape, np.uint8)
            self.v_codes = np.zeros(shape, np.uint8)
            self.k_scales = np.ones(shape[:-1] + (ng,), np.float32)
            self.k_zeros = np.zeros(shape[:-1] + (ng,), np.float32)
            self.v_scales = np.ones(shape[:-1] + (ng,), np.float32)
            self.v_zeros = np.zeros(shape[:-1] + (ng,), np.float32)
        elif block_fmt is not None:
            self.block_fmt = _c(block_fmt, np.uint8)
            assert self.block_fmt.shape == (num_blocks,) and int(self.block_fmt.max(initial=0)) <= FMT_E5M2
            self.k = np.zeros(shape, np.float64)
            self.v = np.zeros(shape, np.float64)
            self.k_codes = np.zeros(shape, np.uint8)
            self.v_codes = np.zeros(shape, np.uint8)
            self.k_scales = np.ones(shape[:-1], np.float32)
            self.v_scales = np.ones(shape[:-1], np.float32)
        elif fp8:
            self.k_codes = np.zeros(shape, np.uint8)
            self.v_codes = np.zeros(shape, np.uint8)
            self.k_scales = np.ones(shape[:-1], np.float32)
            self.v_scales = np.ones(shape[:-1], np.float32)
            self.k = self.v = None
        else:
            self.k = np.zeros(shape, np.float64)
            self.v = np.zeros(shape, np.float64)
            self.k_codes = self.v_codes = self.k_scales = self.v_scales = None

    def append(self, k_new, v_new, slot_mapping) -> int:
        """Write tokens: k_new, v_new float32 [N][n_kv][d_h] (bf16 values), slot_mapping int64 [N]."""
        k = _c(k_new, np.float32)
        v = _c(v_new, np.float32)
        s = _c(slot_mapping, np.int64)
        if self.angle:
            return _load().kvdo_append_angle(self.n_kv, self.d_h, self.block_size, self.num_blocks, _p(k), _p(v),
                                             _p(s), s.size, _p(self.k_codes), _p(self.v_codes), _p(self.k_scales),
                                             _p(self.v_scales), _p(self.k_radius))
        if self.lowbit is not None:
            return _load().kvdo_append_lowbit(self.n_kv, self.d_h, self.block_size, self.num_blocks, self.lowbit[0],
                                              self.lowbit[1], _p(k), _p(v), _p(s), s.size, _p(self.k), _p(self.v),
                                              _p(self.k_codes), _p(self.v_codes), _p(self.k_scales),
                                              _p(self.k_zeros), _p(self.v_scales), _p(self.v_zeros))
        if self.block_fmt is not None:
            return _load().kvdo_append_mixed(self.n_kv, self.d_h, self.block_size, self.num_blocks,
                                             _p(self.block_fmt), _p(k), _p(v), _p(s), s.size, _p(self.k), _p(self.v),
                                             _p(self.k_codes), _p(self.v_codes), _p(self.k_scales),
                                             _p(self.v_scales))
        return _load().kvdo_append(self.n_kv, self.d_h, self.block_size, self.num_blocks, int(self.fp8),
                                   _p(k), _p(v), _p(s), s.size,
                                   _p(self.k), _p(self.v), _p(self.k_codes), _p(self.v_codes),
                                   _p(self.k_scales), _p(self.v_scales))

    def values(self) -> tuple[np.ndarray, np.ndarray]:
        """fp64 K and V as read by attention (FP8: code value × row scale)."""
        if not self.fp8 or self.block_fmt is not None or self.lowbit is not None:
            return self.k, self.v
        rows = self.num_blocks * self.n_kv * self.block_size
        kd = np.empty(self.k_codes.shape, np.float64)
        vd = np.empty(self.v_codes.shape, np.float64)
        lib = _load()
        lib.kvdo_dequant_pool(_p(self.k_codes), _p(self.k_scales), rows, self.d_h, _p(kd))
        lib.kvdo_dequant_pool(_p(self.v_codes), _p(self.v_scales), rows, self.d_h, _p(vd))
        return kd, vd


def decode(pool: OraclePool, q, n_q: int, block_table, seq_lens, retain=None, softmax_scale=None,
           want_alpha: bool = False, want_logits: bool = False, kv_values=None):
    """fp64 decode attention.  Returns dict(out [B][n_q][d_h], lse [B][n_q], status[, alpha, logits])."""
    qd = _c(q, np.float64)
    B = qd.shape[0]
    bt = _c(block_table, np.int32)
    sl = _c(seq_lens, np.int32)
    rt = None if retain is None else _c(np.asarray(retain) & 0xFFFF, np.uint16)
    if softmax_scale is None:
        softmax_scale = 1.0 / np.sqrt(pool.d_h)
    kv, vv = pool.values() if kv_values is None else kv_values
    kv = _c(kv, np.float64)
    vv = _c(vv, np.float64)
    out = np.zeros((B, n_q, pool.d_h), np.float64)
    lse = np.zeros((B, n_q), np.float64)
    stride = int(sl.max()) if sl.size else 0
    alpha = np.zeros((B, n_q, stride), np.float64) if want_alpha else None
    logits = np.full((B, n_q, stride), -np.inf, np.float64) if want_logits else None
    st = _load().kvdo_decode(n_q, pool.n_kv, pool.d_h, pool.block_size, pool.num_blocks,
                             _p(qd), _p(kv), _p(vv), _p(bt), bt.shape[1], _p(sl), B, _p(rt),
                             float(softmax_scale), _p(out), _p(lse), _p(alpha), _p(logits), stride)
    res = {"out": out, "lse": lse, "status": st}
    if want_alpha:
        res["alpha"] = alpha
    if want_logits:
        res["logits"] = logits
    return res


def score_update(s, alpha_layers, seq_lens) -> np.ndarray:
    """One step of s_i += (1/L) Σ_ℓ (1/H) Σ_h α; alpha_layers [L][B][H][stride], s [B][stride] (updated copy)."""
    a = _c(alpha_layers, np.float64)
    L, B, H, stride = a.shape
    out = _c(s, np.float64).copy()
    assert out.shape == (B, stride)
    sl = _c(seq_lens, np.int32)
    _load().kvdo_score_update(_p(a), L, B, H, _p(sl), stride, _p(out))
    return out


def tier_plan(scores, seq_lens, max_blocks: int, protect_prompt: int, protect_recent: int, t1: int,
              block_size: int = 16) -> tuple[np.ndarray, np.ndarray]:
    """Per-block importance (fp32 [B][max_blocks]) and tier (int8: 1 host, 0 HBM, -1 past the
    context) from cumulative scores [B][stride] (fp32)."""
    sc = _c(scores, np.float32)
    B, stride = sc.shape
    sl = _c(seq_lens, np.int32)
    assert sl.shape == (B,)
    imp = np.zeros((B, max_blocks), np.float32)
    tier = np.zeros((B, max_blocks), np.int8)
    _load().kvdo_tier_plan(_p(sc), stride, _p(sl), B, int(max_blocks), int(block_size), int(protect_prompt),
                           int(protect_recent), int(t1), _p(imp), _p(tier))
    return imp, tier


def decode_dense_inputs(k_logical, v_logical, q, seq_lens, n_q, evicted=None, fp8=False, softmax_scale=None):
    """Run the oracle on logical (unpaged) K/V by paging them into an identity-ordered pool.

    k_logical, v_logical: list over requests of float32 [ctx_b][n_kv][d_h] (bf16 values);
    evicted: optional list over requests of position arrays.  Used for sampled checks of
    large workloads, where only the sampled requests are regenerated on the host.
    """
    bs = 16
    n_kv, d_h = k_logical[0].shape[1], k_logical[0].shape[2]
    nblk = [-(-int(c) // bs) for c in seq_lens]
    nb = sum(nblk)
    bt = np.full((len(seq_lens), max(nblk)), -1, np.int32)
    pool = OraclePool(nb, n_kv, d_h, bs, fp8)
    off = 0
    retain = None
    if evicted is not None:
        retain = np.full(nb, 0xFFFF, np.int64)
    for b, c in enumerate(seq_lens):
        bt[b, :nblk[b]] = np.arange(off, off + nblk[b])
        slots = np.arange(c, dtype=np.int64) + off * bs
        pool.append(k_logical[b], v_logical[b], slots)
        if evicted is not None:
            for pos in np.asarray(evicted[b]).tolist():
                retain[off + pos // bs] &= ~(1 << (pos % bs))
        off += nblk[b]
    return decode(pool, q, n_q, bt, seq_lens, retain, softmax_scale, want_alpha=True, want_logits=True)
