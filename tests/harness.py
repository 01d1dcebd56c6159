"""Helpers for GPU parity tests: fill a device pool through the C ABI, run the oracle
on the same seeded inputs, unpack the device pool's documented layout, and compare
within the stated tolerances."""

from __future__ import annotations

import numpy as np
import torch

import oracle
import paged_gqa_decode_kvd_gb300 as kvd
from kvd_inputs import Workload

# Output parity: max |err| <= 2e-3 absolute + 1e-2 relative (bf16 outputs, fp32 accumulation).
OUT_ATOL, OUT_RTOL = 2e-3, 1e-2
# Importance scores: 1e-5 relative.
SCORE_RTOL = 1e-5
# Split vs non-split device results (fp32 output).
SPLIT_ATOL = 1e-3


def assert_out_close(gpu, ref, atol=OUT_ATOL, rtol=OUT_RTOL, what="out"):
    g = np.asarray(gpu, np.float64)
    r = np.asarray(ref, np.float64)
    err = np.abs(g - r)
    bound = atol + rtol * np.abs(r)
    bad = err > bound
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} outside {atol}+{rtol}|ref|; "
                           f"max err {err.max():.3e} at {np.unravel_index(err.argmax(), err.shape)}")
    return float(err.max())


def dtype_code(w: Workload) -> int:
    return {"bf16": kvd.KVD_BF16, "fp8_e4m3": kvd.KVD_FP8_E4M3, "mixed": kvd.KVD_MIXED, "int4": kvd.KVD_INT4,
            "int2": kvd.KVD_INT2, "angle": kvd.KVD_ANGLE}[w.kv_dtype]


FORMAT_CODES = (kvd.KVD_BF16, kvd.KVD_FP8_E4M3, kvd.KVD_FP8_E5M2)   # index = oracle format code


def make_pool(w: Workload, layers: int | None = None, poison: bool = True) -> kvd.KVPool:
    pool = kvd.KVPool(layers or w.L, w.n_kv, w.num_blocks(), dtype_code(w), group_size=w.group_size)
    if poison:   # NaN everywhere first (codes, bf16 values, fp32 scales): unwritten slots must never leak
        pool.mem.fill_(0xFF)
    if w.kv_dtype == "mixed":
        codes = torch.tensor([FORMAT_CODES[f] for f in w.block_formats().tolist()], dtype=torch.uint8)
        pool.set_block_formats(codes.to(pool.mem.device))
    return pool


def fill_layer(pool: kvd.KVPool, w: Workload, layer: int, bt_cpu: torch.Tensor, upto: list[int], dev,
               pool_layer: int | None = None):
    """Append positions [0, upto[b]) of every request of `layer` through kvd_append_kv."""
    for b in range(w.batch):
        n = upto[b]
        if n <= 0:
            continue
        k, v = w.kv(layer, b, 0, n, dev)
        slots = w.slot_mapping(b, 0, n, bt_cpu).to(dev)
        kvd.kvd_append_kv(pool.handle, layer if pool_layer is None else pool_layer, k.contiguous(), v.contiguous(),
                          slots)


def device_inputs(w: Workload, dev, step: int = 0):
    bt = w.block_table()
    seq = torch.tensor(w.seq_lens(step), dtype=torch.int32)
    retain = w.retain_mask(bt)
    return bt, bt.to(dev), seq, seq.to(dev), None if retain is None else retain_bits(retain).to(dev)


def retain_bits(mask: torch.Tensor) -> torch.Tensor:
    """int32 values 0..65535 -> int16 tensor holding the same 16 bits (the C side reads uint16)."""
    return torch.from_numpy(mask.numpy().astype(np.uint16).view(np.int16))


def workspace(pool: kvd.KVPool, n_q: int, batch: int, max_seq: int, num_splits: int = 0, dev="cuda"):
    s, nbytes = kvd.kvd_decode_workspace_bytes(pool.handle, n_q, batch, max_seq, num_splits)
    return s, torch.empty(nbytes, dtype=torch.uint8, device=dev)


def oracle_layer(w: Workload, layer: int, bt_cpu: torch.Tensor, seq_lens: list[int], retain=None, step: int = 0,
                 want_alpha=False, want_logits=False, q=None):
    """fp64 oracle over the oracle's own pool filled from the same seeded inputs."""
    if w.kv_dtype == "mixed":
        pool = oracle.OraclePool(w.num_blocks(), w.n_kv, w.d_h, 16, block_fmt=w.block_formats())
    elif w.lowbit:
        pool = oracle.OraclePool(w.num_blocks(), w.n_kv, w.d_h, 16, lowbit=w.lowbit)
    elif w.kv_dtype == "angle":
        pool = oracle.OraclePool(w.num_blocks(), w.n_kv, w.d_h, 16, angle=True)
    else:
        pool = oracle.OraclePool(w.num_blocks(), w.n_kv, w.d_h, 16, w.kv_dtype != "bf16")
    for b in range(w.batch):
        k, v = w.kv(layer, b, 0, seq_lens[b])
        slots = w.slot_mapping(b, 0, seq_lens[b], bt_cpu).numpy()
        assert pool.append(k.float().numpy(), v.float().numpy(), slots) == 0
    if q is None:
        q = w.q(layer, step)
    qn = q.float().numpy()
    if w.kv_dtype == "angle":   # the query of an angle-domain logit: its own direction code, rescaled
        qn = oracle.angle_query(qn)
    return oracle.decode(pool, qn, w.n_q, bt_cpu.numpy(), seq_lens,
                         None if retain is None else retain.numpy(), 1.0 / np.sqrt(w.d_h),
                         want_alpha=want_alpha, want_logits=want_logits)


# ---------------------------------------------------------------- pool layout
def _tile_perm(kind: str, fp8: bool) -> np.ndarray:
    """index[t, d] of element (token t, dim d) inside a K or V tile (documented layout)."""
    t = np.arange(16)[:, None]
    d = np.arange(128)[None, :]
    i = d // 16
    if kind == "k":
        c = d % 16
        lane = 4 * (t % 8) + (c % 8) // 2
        e = (c % 2) + 2 * (t // 8) + 4 * (c // 8)
    else:
        r = d % 16
        lane = 4 * (r % 8) + (t % 8) // 2
        e = (t % 2) + 2 * (r // 8) + 4 * (t // 8)
    if fp8:
        return ((i // 2) * 32 + lane) * 16 + (i % 2) * 8 + e
    return (i * 32 + lane) * 8 + e


def read_record(pool: kvd.KVPool, layer: int, block: int, head: int):
    """(K, V) of one (layer, block, head) record, each [16][128], as stored (bf16 tensor or uint8 codes)."""
    fp8 = pool.kv_dtype in (kvd.KVD_FP8_E4M3, kvd.KVD_ANGLE)
    rb = pool.record_bytes
    off = ((layer * pool.num_blocks + block) * pool.n_kv + head) * rb
    raw = pool.mem[off:off + rb].cpu()
    if fp8:
        kt, vt = raw[:2048].numpy(), raw[2048:4096].numpy()
        return kt[_tile_perm("k", True)], vt[_tile_perm("v", True)]
    vals = raw.view(torch.bfloat16)
    kt, vt = vals[:2048], vals[2048:]
    return kt[torch.from_numpy(_tile_perm("k", False))], vt[torch.from_numpy(_tile_perm("v", False))]


def read_scales(pool: kvd.KVPool, layer: int, block: int, head: int):
    """(K scales, V scales) [16] fp32 stored after the tiles of an FP8 record."""
    off = ((layer * pool.num_blocks + block) * pool.n_kv + head) * pool.record_bytes + 4096
    s = pool.mem[off:off + 128].cpu().view(torch.float32).numpy()
    return s[:16], s[16:]


def _lowbit_positions(bits: int, kind: str):
    """(byte index, bit shift) [16][128] of the code of (token t, dim d) in a low-bit K or V tile,
    from the layout the header documents."""
    t = np.arange(16)[:, None]
    d = np.arange(128)[None, :]
    per = 8 // bits
    kg = d // (16 * per)
    h = (d // 16) % per
    c = d % 16
    if kind == "k":
        lane = 4 * (t % 8) + (c % 8) // 2
        j = (c % 2) + 2 * (c // 8)
    else:
        lane = 4 * (c % 8) + (t % 8) // 2
        j = (t % 2) + 2 * (c // 8)
    th = t // 8
    byte = (((kg // 2) * 32 + lane) * 4 + (kg % 2) * 2 + th) * 4 + j
    return np.broadcast_to(byte, (16, 128)), np.broadcast_to(h * bits, (16, 128))


def read_lowbit_record(pool: kvd.KVPool, layer: int, block: int, head: int):
    """(K codes, V codes [16][128] uint8, K scales, K zeros, V scales, V zeros [16][ng] float32) of one
    record of a low-bit pool, unpacked from the documented layout."""
    bits = 4 if pool.kv_dtype == kvd.KVD_INT4 else 2
    ng = 128 // pool.group_size
    rb = pool.record_bytes
    tile = 256 * bits
    off = ((layer * pool.num_blocks + block) * pool.n_kv + head) * rb
    raw = pool.mem[off:off + rb].cpu().numpy()
    out = []
    for kind, base in (("k", 0), ("v", tile)):
        byte, shift = _lowbit_positions(bits, kind)
        out.append(((raw[base + byte] >> shift) & ((1 << bits) - 1)).astype(np.uint8))
    meta = raw[2 * tile:].view(np.float16).astype(np.float32).reshape(2, 16, ng, 2)
    return out[0], out[1], meta[0, ..., 0], meta[0, ..., 1], meta[1, ..., 0], meta[1, ..., 1]
