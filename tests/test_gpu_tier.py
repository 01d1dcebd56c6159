"""Host tier (T1): blocks whose records live in pinned host memory — read by the decode kernel
in place, or staged into HBM before each layer's attention — give outputs bit-identical to the
same blocks kept in HBM
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
@pytest.mark.parametrize("staged", [False, True], ids=["direct", "staged"])
@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
def test_host_tier_is_bitwise_identical_to_hbm(cuda_device, kv_dtype, staged):
    dev = cuda_device
    w = _workload(kv_dtype)
    lens = w.seq_lens()
    bt = w.block_table()
    bt2, moved = _tiered_table(w, bt)
    retain = w.retain_mask(bt)
    ret2 = torch.cat([retain, retain[[p for p, _ in moved]]])
    prefix = [c - 1 for c in lens]

    hbm = H.make_pool(w)
    tier = H.make_pool(w)
    tier.attach_host_tier(len(moved), staged=staged)
    tier.host_mem.fill_(0xFF)   # unwritten host slots hold NaN, like the poisoned pool
    for layer in range(w.L):
        H.fill_layer(hbm, w, layer, bt, prefix, dev)
        H.fill_layer(tier, w, layer, bt2, prefix, dev)
    torch.cuda.synchronize()

    _compare_layers(hbm, tier, w, bt, bt2, retain, ret2, moved, dev)


def _compare_layers(hbm, tier, w, bt, bt2, retain, ret2, moved, dev):
    """Decode every layer (fused append included, with and without splits) on the all-HBM pool
    and on the tiered one: outputs, LSE and logits bit-identical, and every host record equal to
    its HBM twin afterwards (the appended token included)."""
    lens = w.seq_lens()
    seq_d = torch.tensor(lens, dtype=torch.int32, device=dev)
    pos = w.append_pos(0)
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

    rb, nkv, nb, nh = hbm.record_bytes, w.n_kv, w.num_blocks(), tier.host_blocks
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
    kvd.kvd_pool_attach_host_tier(pool.handle, pinned, None, 4)   # direct reads: no staging, prefetch a no-op
    kvd.kvd_tier_prefetch(pool.handle, 0)
    kvd.kvd_pool_attach_host_tier(pool.handle, None, None, 0)   # detach


@pytest.mark.gpu
@pytest.mark.parametrize("case", ["mixed", "stride_cut", "max_blocks"])
def test_tier_plan_matches_oracle(cuda_device, case):
    """Block importance bit-identical (fp32 sums in position order on both sides) and the tier
    of every block equal to the oracle's (page "기술 요약: 모든 사고가 HBM 을 필요로 하는
    것은 아님", sections "1. 4 단계 분류" and "4. 시스템 구현")."""
    import oracle
    rng = np.random.default_rng(41)
    if case == "mixed":
        lens, mb, stride, pp, pr, t1 = [0, 1, 16, 17, 700, 4096, 4097, 5000], 300, 4800, 64, 48, 40
    elif case == "stride_cut":
        lens, mb, stride, pp, pr, t1 = [1000, 1200, 333], 80, 1004, 16, 0, 7
    else:   # the largest plan: one request of 16384 blocks
        lens, mb, stride, pp, pr, t1 = [262144], 16384, 262144, 4, 64, 9000
    s = rng.exponential(1e-4, size=(len(lens), stride)).astype(np.float32)
    s[:, ::3] = np.round(s[:, ::3], 5)   # repeated values, so block importances tie
    s[:, 160:320] = 0.0                  # ten all-zero blocks per request: a tie at 0
    imp_ref, tier_ref = oracle.tier_plan(s, lens, mb, pp, pr, t1)
    dev = cuda_device
    sd = torch.from_numpy(s).to(dev)
    ld = torch.tensor(lens, dtype=torch.int32, device=dev)
    tier = torch.full((len(lens), mb), 7, dtype=torch.int8, device=dev)
    imp = torch.full((len(lens), mb), float("nan"), dtype=torch.float32, device=dev)
    kvd.kvd_tier_plan(sd, ld, mb, pp, pr, t1, tier, importance=imp)
    torch.cuda.synchronize()
    assert np.array_equal(imp.cpu().numpy().view(np.uint32), imp_ref.view(np.uint32))
    assert np.array_equal(tier.cpu().numpy(), tier_ref)


@pytest.mark.gpu
def test_tier_plan_rejects_bad_arguments(cuda_device):
    s = torch.zeros(1, 64, device=cuda_device)
    ln = torch.tensor([64], dtype=torch.int32, device=cuda_device)
    with pytest.raises(kvd.KvdError):
        kvd.kvd_tier_plan(s, ln, 16385, 0, 0, 1, torch.empty(1, 16385, dtype=torch.int8, device=cuda_device))
    with pytest.raises(kvd.KvdError):
        kvd.kvd_tier_plan(s, ln, 4, -1, 0, 1, torch.empty(1, 4, dtype=torch.int8, device=cuda_device))


def _record_view(mem, layer, block, h, nblk, nkv, rb):
    off = ((layer * nblk + block) * nkv + h) * rb
    return mem[off:off + rb]


@pytest.mark.gpu
@pytest.mark.parametrize("dtype_code", [kvd.KVD_BF16, kvd.KVD_FP8_E4M3])
def test_tier_move_copies_whole_records(cuda_device, dtype_code):
    """Every layer's and head's record of each source block lands on its destination, between
    and within tiers; untouched blocks keep their bytes; a bad id is reported and skipped."""
    L, nkv, nblk, nh = 3, 2, 40, 12
    pool = kvd.KVPool(L, nkv, nblk, dtype_code, device=cuda_device)
    pool.attach_host_tier(nh)
    g = torch.Generator().manual_seed(5)
    pool.mem.copy_(torch.randint(0, 256, pool.mem.shape, generator=g, dtype=torch.uint8))
    pool.host_mem.copy_(torch.randint(0, 256, pool.host_mem.shape, generator=g, dtype=torch.uint8))
    torch.cuda.synchronize()
    rb = pool.record_bytes
    before_hbm, before_host = pool.mem.cpu().clone(), pool.host_mem.clone()
    pairs = [(3, nblk + 0), (7, nblk + 5), (nblk + 2, 11), (nblk + 9, 30), (20, 21), (nblk + 10, nblk + 11)]
    frm = torch.tensor([a for a, _ in pairs], dtype=torch.int32, device=cuda_device)
    to = torch.tensor([b for _, b in pairs], dtype=torch.int32, device=cuda_device)
    kvd.kvd_tier_move(pool.handle, frm, to)
    torch.cuda.synchronize()
    assert kvd.kvd_get_device_error(pool.handle) == 0

    def rec(mem_hbm, mem_host, layer, blk, h):
        if blk < nblk:
            return _record_view(mem_hbm, layer, blk, h, nblk, nkv, rb)
        return _record_view(mem_host, layer, blk - nblk, h, nh, nkv, rb)

    want_hbm, want_host = before_hbm.clone(), before_host.clone()
    for a, b in pairs:
        for layer in range(L):
            for h in range(nkv):
                rec(want_hbm, want_host, layer, b, h).copy_(rec(before_hbm, before_host, layer, a, h))
    assert torch.equal(pool.mem.cpu(), want_hbm)
    assert torch.equal(pool.host_mem, want_host)

    bad_from = torch.tensor([nblk + nh, 1], dtype=torch.int32, device=cuda_device)
    bad_to = torch.tensor([2, 4], dtype=torch.int32, device=cuda_device)
    kvd.kvd_tier_move(pool.handle, bad_from, bad_to)
    torch.cuda.synchronize()
    assert kvd.kvd_get_device_error(pool.handle) == kvd.KVD_ERR_OOB
    for layer in range(L):   # the valid pair still moved, the bad one did not
        for h in range(nkv):
            assert torch.equal(_record_view(pool.mem, layer, 4, h, nblk, nkv, rb).cpu(),
                               _record_view(want_hbm, layer, 1, h, nblk, nkv, rb))
            assert torch.equal(_record_view(pool.mem, layer, 2, h, nblk, nkv, rb).cpu(),
                               _record_view(want_hbm, layer, 2, h, nblk, nkv, rb))


@pytest.mark.gpu
@pytest.mark.parametrize("staged", [False, True], ids=["direct", "staged"])
@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
def test_plan_move_decode_is_bitwise_identical_to_hbm(cuda_device, kv_dtype, staged):
    """A re-tiering round as a caller runs it: plan from the scores, move the planned blocks to
    host-tier ids, patch the block tables, poison the vacated HBM blocks; the next decode step
    is bit-identical to the all-HBM pool."""
    dev = cuda_device
    w = _workload(kv_dtype)
    lens = w.seq_lens()
    bt = w.block_table()
    retain = w.retain_mask(bt)
    prefix = [c - 1 for c in lens]
    mb, nb = bt.shape[1], w.num_blocks()
    hbm = H.make_pool(w)
    tier = H.make_pool(w)
    for layer in range(w.L):
        H.fill_layer(hbm, w, layer, bt, prefix, dev)
        H.fill_layer(tier, w, layer, bt, prefix, dev)

    rng = np.random.default_rng(17)
    scores = torch.from_numpy(rng.exponential(1e-3, size=(w.batch, max(lens))).astype(np.float32)).to(dev)
    seq_d = torch.tensor(lens, dtype=torch.int32, device=dev)
    plan = torch.empty(w.batch, mb, dtype=torch.int8, device=dev)
    kvd.kvd_tier_plan(scores, seq_d, mb, 32, 16, 6, plan)
    plan = plan.cpu()
    bt2 = bt.clone()
    moved = []
    for b in range(w.batch):
        for j in range(mb):
            if plan[b, j] == 1:
                moved.append((int(bt[b, j]), nb + len(moved)))
                bt2[b, j] = moved[-1][1]
    assert len(moved) > 10 and all(plan[b, (lens[b] - 1) // 16] == 0 for b in range(w.batch))

    tier.attach_host_tier(len(moved), staged=staged)
    tier.host_mem.fill_(0xFF)
    frm = torch.tensor([a for a, _ in moved], dtype=torch.int32, device=dev)
    to = torch.tensor([h for _, h in moved], dtype=torch.int32, device=dev)
    kvd.kvd_tier_move(tier.handle, frm, to)
    rb = tier.record_bytes
    for layer in range(w.L):   # the vacated HBM blocks now hold NaN (all heads' records are adjacent)
        for orig, _ in moved:
            off = (layer * nb + orig) * w.n_kv * rb
            tier.mem[off:off + w.n_kv * rb].fill_(0xFF)
    torch.cuda.synchronize()
    assert kvd.kvd_get_device_error(tier.handle) == 0
    ret2 = torch.cat([retain, retain[[p for p, _ in moved]]])
    _compare_layers(hbm, tier, w, bt, bt2, retain, ret2, moved, dev)


def _poison(pool, w, ids):
    """NaN bytes into every layer's records of the given block ids (pool or host tier)."""
    torch.cuda.synchronize()   # host-tier bytes are written by the CPU: the moves must have run
    nb, rb = w.num_blocks(), pool.record_bytes
    for layer in range(w.L):
        for p in ids:
            if p < nb:
                off = (layer * nb + p) * w.n_kv * rb
                pool.mem[off:off + w.n_kv * rb].fill_(0xFF)
            else:
                off = (layer * pool.host_blocks + (p - nb)) * w.n_kv * rb
                pool.host_mem[off:off + w.n_kv * rb].fill_(0xFF)


@pytest.mark.gpu
@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
def test_reassignment_rounds_are_bitwise_identical_to_hbm(cuda_device, kv_dtype):
    """Two reassignment rounds as a serving loop runs them every Δ steps: plan on the device,
    kvd_tier_reassign on the host (free lists, table and retain patch), kvd_tier_move, vacated
    blocks poisoned.  The second round's plan differs, so blocks are promoted back to HBM and
    others demoted; after each round the decode is bit-identical to the all-HBM pool."""
    dev = cuda_device
    w = _workload(kv_dtype)
    lens = w.seq_lens()
    bt = w.block_table()
    retain = w.retain_mask(bt)
    prefix = [c - 1 for c in lens]
    mb, nb, nh = bt.shape[1], w.num_blocks(), 64
    hbm = H.make_pool(w)
    tier = H.make_pool(w)
    for layer in range(w.L):
        H.fill_layer(hbm, w, layer, bt, prefix, dev)
        H.fill_layer(tier, w, layer, bt, prefix, dev)
    tier.attach_host_tier(nh)
    tier.host_mem.fill_(0xFF)

    bt_host = bt.numpy().astype(np.int32).copy()
    used = set(int(x) for x in bt_host.ravel() if x >= 0)
    hbm_free = np.zeros(nb, np.int32)
    free = [i for i in range(nb) if i not in used]
    hbm_free[:len(free)] = free
    hn = len(free)
    host_free = np.arange(nb, nb + nh, dtype=np.int32)
    tn = nh
    ret_host = np.concatenate([retain.numpy().astype(np.uint16), np.full(nh, 0xFFFF, np.uint16)])
    seq_d = torch.tensor(lens, dtype=torch.int32, device=dev)
    promoted = 0
    for seed in (17, 23):
        rng = np.random.default_rng(seed)
        scores = torch.from_numpy(rng.exponential(1e-3, size=(w.batch, max(lens))).astype(np.float32)).to(dev)
        plan = torch.empty(w.batch, mb, dtype=torch.int8, device=dev)
        kvd.kvd_tier_plan(scores, seq_d, mb, 32, 16, 6, plan)
        st, frm, to, hn, tn = kvd.kvd_tier_reassign(nb, nh, plan.cpu().numpy(), bt_host, hbm_free, hn, host_free, tn,
                                                     ret_host)
        assert st == kvd.KVD_OK and len(frm) > 0
        promoted += int(((frm >= nb) & (to < nb)).sum())
        kvd.kvd_tier_move(tier.handle, torch.from_numpy(frm).to(dev), torch.from_numpy(to).to(dev))
        _poison(tier, w, frm.tolist())
        torch.cuda.synchronize()
        assert kvd.kvd_get_device_error(tier.handle) == 0
        moved = [(int(bt[b, j]), int(bt_host[b, j])) for b in range(w.batch) for j in range(mb)
                 if bt_host[b, j] >= nb]
        _compare_layers(hbm, tier, w, bt, torch.from_numpy(bt_host.copy()), retain,
                        torch.from_numpy(ret_host.astype(np.int32)), moved, dev)
    assert promoted > 0
