"""The seeded input generator: determinism, addressability and the workload recipes."""

import numpy as np
import torch

import kvd_inputs as ki
from kvd_inputs import gen


def test_hash_matches_python_reference():
    idx = torch.arange(0, 1000, dtype=torch.int64) * 977 + 5
    key = gen.stream_key(3, "k", 1)
    h = gen.hash_index(key, idx).numpy().astype(np.uint64)
    ref = [gen.mix64(key + int(i)) for i in idx.tolist()]
    assert [int(x) for x in h] == ref


def test_normal_is_standard_and_slices_are_addressable():
    key = gen.stream_key(0, "x")
    full = gen.normal(key, gen.index_range(0, 1 << 20, "cpu"))
    assert abs(full.mean().item()) < 5e-3 and abs(full.std().item() - 1) < 5e-3
    part = gen.normal(key, gen.index_range(12345, 1000, "cpu"))
    assert torch.equal(part, full[12345:13345])


def test_workload_shapes_and_structure():
    w = ki.get("tiny")
    bt = w.block_table()
    assert bt.shape == (1, 128) and len(set(bt[0].tolist())) == 128 and int(bt.max()) < 256
    w = ki.get("llama8b")
    bt = w.block_table()
    assert sorted(bt.flatten().tolist()) == list(range(16384))
    assert w.kv_bytes_per_step() == 32 * 8192 * 131072          # 131,072 B per token over 32 layers
    w = ki.get("ragged")
    lens = w.seq_lens()
    assert len(lens) == 64 and min(lens) >= 256 and max(lens) <= 32768
    assert any(c % 16 for c in lens)
    w = ki.get("tiered")
    assert w.seq_lens(0)[0] == 16385 and w.seq_lens(63)[0] == 16448 and w.max_blocks() == 1028
    ev = w.evicted_positions(0)
    assert ev.numel() == 468 and int(ev.min()) >= 512 and int(ev.max()) < 16128
    m = w.retain_mask()
    assert sum(bin(0xFFFF & ~x).count("1") for x in m.tolist()) == 8 * 468


def test_kv_values_are_deterministic_and_slice_consistent():
    w = ki.get("llama70b_fp8")
    k1, v1 = w.kv(3, 0, 100, 164)
    k2, v2 = w.kv(3, 0, 0, 200)
    assert torch.equal(k1, k2[100:164]) and torch.equal(v1, v2[100:164])
    f = w._outlier_factor(3, "k", "cpu")
    assert set(f.unique().tolist()) <= {1.0, 20.0}


def test_mixed_workload_bytes_count_each_token_at_its_blocks_width():
    """K/V bytes of a mixed pool: 2·L·n_kv·d_h·w_kv per token with w_kv = 2 for a token in a BF16
    block and 1 in an E4M3 / E5M2 block (scales counted apart: 8 B per token and KV head)."""
    from kvd_inputs import Workload

    w = Workload("mixed_bytes", L=3, n_q=8, n_kv=2, d_h=128, batch=3, kv_dtype="mixed", seed=4,
                 mixed_probs=(0.3, 0.4, 0.3))
    w._ctx0 = [37, 300, 16]
    fmt = w.block_formats()
    assert set(fmt.tolist()) <= {0, 1, 2} and len(fmt) == w.num_blocks()
    bt = w.block_table()
    wide = narrow = 0
    for b, n in enumerate(w.seq_lens()):
        for t in range(n):
            if fmt[int(bt[b, t // 16])] == 0:
                wide += 1
            else:
                narrow += 1
    assert w.kv_bytes_per_step() == 2 * 3 * 2 * 128 * (2 * wide + narrow)
    assert w.scale_bytes_per_step() == 2 * 3 * 2 * 4 * narrow
    import pytest
    with pytest.raises(ValueError):
        w.w_kv
