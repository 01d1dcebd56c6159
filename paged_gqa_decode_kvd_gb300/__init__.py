"""Paged GQA decode attention for GB300 (sm_103a).

The computation lives in ``libkvd.so`` (hand-written CUDA behind a C ABI,
``include/kvd.h``); this package is its Python binding plus a small owner of
pool memory.  Importing it does not touch the GPU; the first call that needs
the library loads it and fails loudly if it is missing or cannot be built.
"""

from __future__ import annotations

from ._lib import (  # noqa: F401
    KVD_ANGLE,
    KVD_BF16,
    KVD_EARLY_START,
    KVD_PLANNED,
    KVD_F32,
    KVD_FP8_E4M3,
    KVD_FP8_E5M2,
    KVD_INT2,
    KVD_INT4,
    KVD_MIXED,
    KVD_OK,
    KVD_ERR_CUDA,
    KVD_ERR_INVALID,
    KVD_ERR_NOMEM,
    KVD_ERR_OOB,
    KVD_ERR_TIMEOUT,
    KVD_ERR_UNSUPPORTED,
    SYMBOLS,
    NOALLOC_SCRATCH_BYTES,
    KvdError,
    kvd_accum_scores,
    kvd_append_kv,
    kvd_pool_attach_host_tier,
    kvd_tier_bytes,
    kvd_tier_prefetch,
    kvd_tier_plan,
    kvd_tier_move,
    kvd_tier_reassign,
    kvd_combine_splits,
    kvd_decode_attn,
    kvd_decode_attn_noalloc,
    kvd_decode_plan,
    kvd_decode_workspace_bytes,
    kvd_measure_read_stream,
    kvd_get_device_error,
    kvd_pool_bytes,
    kvd_pool_create,
    kvd_pool_destroy,
    kvd_pool_set_block_formats,
    kvd_selftest_wait_timeout,
    lib_path,
    load,
    status_string,
)


class KVPool:
    """Device memory for a paged KV pool (torch allocations) plus its library handle."""

    def __init__(self, num_layers: int, n_kv: int, num_blocks: int, kv_dtype: int = KVD_BF16, device="cuda",
                 group_size: int = 0):
        import torch

        self.num_layers, self.n_kv, self.num_blocks, self.kv_dtype = num_layers, n_kv, num_blocks, kv_dtype
        self.group_size = group_size
        pool_bytes, self.kv_bytes = kvd_pool_bytes(num_layers, n_kv, num_blocks, kv_dtype, group_size=group_size)
        self.mem = torch.empty(pool_bytes, dtype=torch.uint8, device=device)
        self.handle = kvd_pool_create(num_layers, n_kv, num_blocks, kv_dtype, self.mem, group_size=group_size)

    @property
    def record_bytes(self) -> int:
        """Bytes of one (layer, block, KV head) record slot: K tile, V tile and (FP8) 32 fp32 scales,
        (INT4 / INT2) 2·16·(128/group_size) scale-and-zero words; a mixed pool sizes every slot for BF16."""
        if self.kv_dtype in (KVD_INT4, KVD_INT2):
            bits = 4 if self.kv_dtype == KVD_INT4 else 2
            return 2 * 256 * bits + 2 * 64 * (128 // self.group_size)
        return 4096 + 128 if self.kv_dtype in (KVD_FP8_E4M3, KVD_ANGLE) else 8192

    def set_block_formats(self, block_fmt):
        """Mixed pool: one precision code per physical block (uint8 device tensor, kept alive here)."""
        self.block_fmt = block_fmt
        kvd_pool_set_block_formats(self.handle, block_fmt)

    def attach_host_tier(self, host_blocks: int, staged: bool = False):
        """Give the pool host_blocks host-tier blocks (ids num_blocks ..): their records in
        pinned host memory, read by the decode kernel in place over the host link, or
        (staged) copied per layer by kvd_tier_prefetch into two HBM staging slots."""
        import torch

        host_bytes, staging_bytes = kvd_tier_bytes(self.num_layers, self.n_kv, self.num_blocks, self.kv_dtype,
                                                   host_blocks)
        self.host_mem = torch.empty(host_bytes, dtype=torch.uint8, pin_memory=True)
        self.staging = torch.empty(staging_bytes, dtype=torch.uint8, device=self.mem.device) if staged else None
        kvd_pool_attach_host_tier(self.handle, self.host_mem, self.staging, host_blocks)
        self.host_blocks = host_blocks

    def close(self):
        if self.handle is not None:
            kvd_pool_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
