"""kvd_decode_attn_noalloc: decode attention for callers that may not allocate device memory.

Such callers (a host framework whose allocator owns all device memory, a latency-critical
loop that cannot take cudaMalloc's synchronisation) pass only inputs and outputs; the split
scratch lives in a fixed array inside the library.  Two calls in a row, with different
shapes, must each match the workspace-taking entry point, so nothing stale from the first
call leaks into the second.  This file is collected last on purpose.
"""

import numpy as np
import pytest
import torch

import paged_gqa_decode_kvd_gb300 as kvd
from kvd_inputs import Workload
from tests import harness as H

pytestmark = pytest.mark.gpu


def _workload(name, n_q, n_kv, lens, seed):
    w = Workload(name, L=1, n_q=n_q, n_kv=n_kv, d_h=128, batch=len(lens), kv_dtype="bf16", seed=seed)
    w._ctx0 = list(lens)
    return w


def _both(w, dev):
    bt, bt_d, seq, seq_d, _ = H.device_inputs(w, dev)
    pool = H.make_pool(w)
    H.fill_layer(pool, w, 0, bt, w.seq_lens(), dev)
    q = w.q(0, 0, dev)
    max_len = max(w.seq_lens())
    _, ws = H.workspace(pool, w.n_q, w.batch, max_len, 0, dev)
    ref = torch.empty(w.batch, w.n_q, 128, dtype=torch.float32, device=dev)
    ref_lse = torch.empty(w.batch, w.n_q, dtype=torch.float32, device=dev)
    kvd.kvd_decode_attn(pool.handle, 0, q, bt_d, seq_d, max_len, ws, ref, lse_out=ref_lse)
    out = torch.full_like(ref, float("nan"))
    lse = torch.full_like(ref_lse, float("nan"))
    kvd.kvd_decode_attn_noalloc(pool.handle, 0, q, bt_d, seq_d, max_len, out, lse_out=lse)
    assert kvd.kvd_get_device_error(pool.handle) == 0
    return out.cpu().numpy(), lse.cpu().numpy(), ref.cpu().numpy(), ref_lse.cpu().numpy()


def test_noalloc_matches_workspace_entry_point_on_two_calls(cuda_device):
    first = _workload("noalloc_a", 32, 8, [3000, 17, 1200, 640], seed=1)
    second = _workload("noalloc_b", 16, 2, [5, 2047, 800], seed=2)
    for w in (first, second):
        out, lse, ref, ref_lse = _both(w, cuda_device)
        H.assert_out_close(out, ref, what=f"{w.name} out")
        np.testing.assert_allclose(lse, ref_lse, rtol=1e-5, atol=1e-4)


def test_noalloc_rejects_shapes_beyond_its_scratch(cuda_device):
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
