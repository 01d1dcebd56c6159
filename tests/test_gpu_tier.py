"""Host tier (T1): blocks whose records live in pinned host memory and are staged into HBM
before each layer's attention give outputs bit-identical to the same blocks kept in HBM
(page "기술 요약: 모든 사고가 HBM 을 필요로 하는 것은 아님", section "3. 제로-근사오차
오프로딩", Prop. 1: the output depends on the evicted set only, not on the HBM/host split)."""

import numpy as np
import pytest
import torch

import harness as H
import paged_gqa_decode_kvd_gb300 as kvd
from kvd_inputs import Workload


def _workload(kv_dtype):
    w = Workload(f"tier_{kv_dtype}", L=2, n_q=16, n_kv=4, d_h=128, batch=5, kv_dtype=kv_dtype, seed=31,
                 evict_frac=0.05, protect_prompt=32, protect_recent=16,
                 outlier_p=0.01 if kv_dtype != "bf16" else 0.0, outlier_factor=20.0)
    w._ctx0 = [700, 333, 1500, 17, 48]
    return w


def _tiered_table(w, bt, frac=0.3, seed=3):
    """Move a seeded fraction of every request's logical blocks (always request 0's last one,
    which the step's append writes) to host-tier ids num_blocks + i."""
    n = w.num_blocks()
    bt2 = bt.clone()
    moved = []   # (original physical block, host-tier id)
    rng = np.random.default_rng(seed)
    for b, ln in enumerate(w.seq_lens()):
        nb = (ln + 15) // 16
        pick = set(int(j) for j in rng.choice(nb, size=max(1, int(frac * nb)), replace=False))
        if b == 0:
            pick.add(nb - 1)
        for j in sorted(pick):
            moved.append((int(bt[b, j]), n + len(moved)))
            bt2[b, j] = moved[-1][1]
    return bt2, moved


def _run_layer(pool, w, layer, bt_d, seq_d, ret_d, k_new, v_new, dev, splits):
    lens = w.seq_lens()
    S = max(lens)
    _, ws = H.workspace(pool, w.n_q, w.batch, S, splits, dev)
    out = torch.empty(w.batch, w.n_q, 128, dtype=torch.float32, device=dev)
    lse = torch.empty(w.batch, w.n_q, dtype=torch.float32, device=dev)
    logits = torch.zeros(w.batch, w.n_q, S, dtype=torch.float32, device=dev)   # unattended columns stay 0
    kvd.kvd_decode_attn(pool.handle, layer, w.q(layer, 0, dev), bt_d, seq_d, S, ws, out, num_splits=splits,
                        retain_mask=ret_d, lse_out=lse, logits_out=logits, k_new=k_new, v_new=v_new)
    torch.cuda.synchronize()
    assert kvd.kvd_get_device_error(pool.handle) == 0
    return out.cpu(), lse.cpu(), logits.cpu()


@pytest.mark.gpu
@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
def test_host_tier_is_bitwise_identical_to_hbm(cuda_device, kv_dtype):
    dev = cuda_device
    w = _workload(kv_dtype)
    lens = w.seq_lens()
    bt = w.block_table()
    bt2, moved = _tiered_table(w, bt)
    retain = w.retain_mask(bt)
    ret2 = torch.cat([retain, retain[[p for p, _ in moved]]])
    seq_d = torch.tensor(lens, dtype=torch.int32, device=dev)
    prefix = [c - 1 for c in lens]
    pos = w.append_pos(0)

    hbm = H.make_pool(w)
    tier = H.make_pool(w)
    tier.attach_host_tier(len(moved))
    tier.host_mem.fill_(0xFF)   # unwritten host slots hold NaN, like the poisoned pool
    for layer in range(w.L):
        H.fill_layer(hbm, w, layer, bt, prefix, dev)
        H.fill_layer(tier, w, layer, bt2, prefix, dev)
    torch.cuda.synchronize()

    for layer in range(w.L):   # layers 0 and 1 use staging slots 0 and 1
        ks, vs = zip(*[w.kv(layer, b, pos[b], pos[b] + 1, dev) for b in range(w.batch)])
        k_new, v_new = torch.cat(ks).contiguous(), torch.cat(vs).contiguous()
        kvd.kvd_tier_prefetch(tier.handle, layer)
        for splits in (0, 7):
            a = _run_layer(hbm, w, layer, bt.to(dev), seq_d, H.retain_bits(retain).to(dev), k_new, v_new, dev,
                           splits)
            b = _run_layer(tier, w, layer, bt2.to(dev), seq_d, H.retain_bits(ret2).to(dev), k_new, v_new, dev,
                           splits)
            for x, y in zip(a, b):
                assert torch.equal(x, y)
        ref = H.oracle_layer(w, layer, bt, lens, retain=retain)
        H.assert_out_close(b[0].numpy(), ref["out"])

    # every host record equals its HBM twin byte for byte (the appended token included)
    rb, nkv, nb, nh = hbm.record_bytes, w.n_kv, w.num_blocks(), len(moved)
    host = tier.host_mem
    for layer in range(w.L):
        for orig, hid in moved:
            for h in range(nkv):
                off_a = ((layer * nb + orig) * nkv + h) * rb
                off_b = ((layer * nh + (hid - nb)) * nkv + h) * rb
                assert torch.equal(hbm.mem[off_a:off_a + rb].cpu(), host[off_b:off_b + rb])


@pytest.mark.gpu
def test_host_tier_attach_checks_its_buffers(cuda_device):
    pool = kvd.KVPool(1, 2, 8, kvd.KVD_BF16, device=cuda_device)
    host_bytes, staging_bytes = kvd.kvd_tier_bytes(1, 2, 8, kvd.KVD_BF16, 4)
    pinned = torch.empty(host_bytes, dtype=torch.uint8, pin_memory=True)
    staging = torch.empty(staging_bytes, dtype=torch.uint8, device=cuda_device)
    with pytest.raises(kvd.KvdError):   # missing host buffer
        kvd.kvd_pool_attach_host_tier(pool.handle, None, staging, 4)
    with pytest.raises(kvd.KvdError):   # staging too small
        kvd.kvd_pool_attach_host_tier(pool.handle, pinned, staging[:staging_bytes // 2], 4)
    with pytest.raises(kvd.KvdError):   # host buffer too small
        kvd.kvd_pool_attach_host_tier(pool.handle, pinned[:host_bytes - 16], staging, 4)
    kvd.kvd_pool_attach_host_tier(pool.handle, pinned, staging, 4)
    kvd.kvd_tier_prefetch(pool.handle, 0)
    torch.cuda.synchronize()
    assert kvd.kvd_get_device_error(pool.handle) == 0
    kvd.kvd_pool_attach_host_tier(pool.handle, None, None, 0)   # detach
