"""kvd_decode_attn_noalloc: decode attention for callers that may not allocate device memory.

Such callers (a host framework whose allocator owns all device memory, a latency-critical
loop that cannot take cudaMalloc's synchronisation) pass only inputs and outputs; the split
scratch lives in a fixed array inside the library.  The entry point runs the same kernels
with the same split plan as kvd_decode_attn, so its results must be the same bits.  Two
calls in a row, with different shapes, pool types and a fused score update, must each match
the workspace-taking entry point, so nothing stale from one call leaks into the next.  This
file is collected last on purpose.
"""

import numpy as np
import pytest
import torch

import paged_gqa_decode_kvd_gb300 as kvd
from kvd_inputs import Workload
from tests import harness as H

pytestmark = pytest.mark.gpu


def _workload(name, n_q, n_kv, lens, seed, kv_dtype="bf16", **kw):
    w = Workload(name, L=1, n_q=n_q, n_kv=n_kv, d_h=128, batch=len(lens), kv_dtype=kv_dtype, seed=seed, **kw)
    w._ctx0 = list(lens)
    return w


def _both(w, dev, scores=False):
    """The same call through both entry points; returns each one's (out, lse[, scores])."""
    bt, bt_d, seq, seq_d, ret_d = H.device_inputs(w, dev)
    pool = H.make_pool(w)
    H.fill_layer(pool, w, 0, bt, w.seq_lens(), dev)
    q = w.q(0, 0, dev)
    max_len = max(w.seq_lens())
    _, ws = H.workspace(pool, w.n_q, w.batch, max_len, 0, dev)
    base = torch.rand(w.batch, max_len, dtype=torch.float32, device=dev) if scores else None
    res = []
    for noalloc in (False, True):
        out = torch.full((w.batch, w.n_q, 128), float("nan"), dtype=torch.float32, device=dev)
        lse = torch.full((w.batch, w.n_q), float("nan"), dtype=torch.float32, device=dev)
        kw = dict(retain_mask=ret_d, lse_out=lse)
        sc = None
        if scores:
            sc = base.clone()
            kw.update(logits_out=torch.empty(w.batch, w.n_q, max_len, dtype=torch.float32, device=dev), scores=sc,
                      inv_LH=1.0 / w.n_q)
        if noalloc:
            kvd.kvd_decode_attn_noalloc(pool.handle, 0, q, bt_d, seq_d, max_len, out, **kw)
        else:
            kvd.kvd_decode_attn(pool.handle, 0, q, bt_d, seq_d, max_len, ws, out, **kw)
        assert kvd.kvd_get_device_error(pool.handle) == 0
        res.append((out.cpu(), lse.cpu(), None if sc is None else sc.cpu()))
    ref = H.oracle_layer(w, 0, bt, w.seq_lens(), retain=w.retain_mask(bt))
    return res, ref, pool


def test_noalloc_matches_workspace_entry_point_on_two_calls(cuda_device):
    calls = [
        (_workload("noalloc_a", 32, 8, [3000, 17, 1200, 640], seed=1), False),
        (_workload("noalloc_b", 28, 4, [5, 2047, 800], seed=2, kv_dtype="fp8_e4m3", outlier_p=0.01,
                   outlier_factor=20.0), False),
        (_workload("noalloc_c", 28, 4, [3000, 700, 16], seed=3, evict_frac=0.05, protect_prompt=64,
                   protect_recent=32, scores=True), True),
    ]
    for w, scores in calls:
        (ws_res, na_res), ref, _ = _both(w, cuda_device, scores)
        for a, b in zip(ws_res, na_res):
            if a is not None:
                assert torch.equal(a, b), f"{w.name}: the no-alloc result differs from the workspace path"
        H.assert_out_close(na_res[0].numpy(), ref["out"], what=f"{w.name} out")
        np.testing.assert_allclose(na_res[1].numpy(), ref["lse"], rtol=1e-5, atol=1e-4)


def test_noalloc_call_allocates_no_device_memory(cuda_device):
    w = _workload("noalloc_mem", 32, 8, [4000, 900], seed=4)
    bt, bt_d, seq, seq_d, _ = H.device_inputs(w, cuda_device)
    pool = H.make_pool(w)
    H.fill_layer(pool, w, 0, bt, w.seq_lens(), cuda_device)
    q = w.q(0, 0, cuda_device)
    out = torch.empty(w.batch, w.n_q, 128, dtype=torch.bfloat16, device=cuda_device)
    kvd.kvd_decode_attn_noalloc(pool.handle, 0, q, bt_d, seq_d, 4000, out)   # first call: address lookup
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info(cuda_device)[0]
    for _ in range(3):
        kvd.kvd_decode_attn_noalloc(pool.handle, 0, q, bt_d, seq_d, 4000, out)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info(cuda_device)[0] == free0
    assert kvd.kvd_get_device_error(pool.handle) == 0


def test_noalloc_rejects_shapes_beyond_its_scratch_and_a_null_output(cuda_device):
    w = _workload("noalloc_big", 64, 8, [16], seed=3)
    pool = H.make_pool(w)
    big_batch = 2048                                  # needs far more than the fixed scratch
    need = kvd.kvd_decode_workspace_bytes(pool.handle, 64, big_batch, 1 << 17, 4096)[1]
    assert need > kvd.NOALLOC_SCRATCH_BYTES
    q = torch.zeros(big_batch, 64, 128, dtype=torch.bfloat16, device=cuda_device)
    bt = torch.zeros(big_batch, 1, dtype=torch.int32, device=cuda_device)
    seq = torch.ones(big_batch, dtype=torch.int32, device=cuda_device)
    out = torch.empty(big_batch, 64, 128, dtype=torch.bfloat16, device=cuda_device)
    with pytest.raises(kvd.KvdError) as e:
        kvd.kvd_decode_attn_noalloc(pool.handle, 0, q, bt, seq, 1 << 17, out, num_splits=4096)
    assert e.value.status == kvd.KVD_ERR_NOMEM
    with pytest.raises(kvd.KvdError) as e:
        kvd.kvd_decode_attn_noalloc(pool.handle, 0, q[:1], bt[:1], seq[:1], 16, None)
    assert e.value.status == kvd.KVD_ERR_INVALID
    # a shape whose planned workspace (five partial slots a split) exceeds the scratch but whose
    # unplanned one fits: accepted, since the entry point never takes a plan
    need_planned = kvd.kvd_decode_workspace_bytes(pool.handle, 64, 16, 16, 1500)[1]
    assert need_planned > kvd.NOALLOC_SCRATCH_BYTES
    bt_w = w.block_table()
    H.fill_layer(pool, w, 0, bt_w, [16], cuda_device)            # request 0's 16 tokens, shared by all 16
    bt16 = bt_w[:1].repeat(16, 1).to(cuda_device)
    seq16 = torch.full((16,), 16, dtype=torch.int32, device=cuda_device)
    q16 = w.q(0, 0, cuda_device).repeat(16, 1, 1).contiguous()
    out16 = torch.empty(16, 64, 128, dtype=torch.float32, device=cuda_device)
    kvd.kvd_decode_attn_noalloc(pool.handle, 0, q16, bt16, seq16, 16, out16, num_splits=1500)
    assert kvd.kvd_get_device_error(pool.handle) == 0
    ref = H.oracle_layer(w, 0, bt_w, [16])["out"][0]
    for b in range(16):
        H.assert_out_close(out16[b].cpu().numpy(), ref, what=f"request {b}")
