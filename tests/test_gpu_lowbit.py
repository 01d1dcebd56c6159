"""Low-bit KV pools (4-bit and 2-bit codes, a half-precision scale and zero point per group of
32, 64 or 128 values of a (token, KV head) row) on the GPU against the oracle's low-bit pool.

"The KV Cache Is the New Memory Wall", §4.2, §4.6 and Tab. 7 name INT4 and 2-bit KV with group
scales; the oracle (OraclePool(lowbit=(bits, group))) quantises each group in single precision
and reads back code·scale + zero.  The CUDA pool must hold the same codes, scales and zero points
bit for bit, and attention over it must match the oracle's fp64 attention over the read-back
values within the output tolerance.
"""

import numpy as np
import pytest
import torch

import paged_gqa_decode_kvd_gb300 as kvd
from kvd_inputs import Workload
from tests import harness as H

pytestmark = pytest.mark.gpu

KINDS = [("int4", 32), ("int4", 64), ("int4", 128), ("int2", 32), ("int2", 64), ("int2", 128)]


def _custom(name, n_q, n_kv, lens, kv_dtype, group, seed=0, L=1, **kw):
    w = Workload(name, L=L, n_q=n_q, n_kv=n_kv, d_h=128, batch=len(lens), kv_dtype=kv_dtype, group_size=group,
                 seed=seed, **kw)
    w._ctx0 = list(lens)
    return w


def _decode(pool, w, bt_d, seq_d, splits=0, retain=None, k_new=None, v_new=None, logits=None, out_f32=True):
    max_len = max(w.seq_lens())
    _, ws = H.workspace(pool, w.n_q, w.batch, max_len, splits)
    out = torch.empty(w.batch, w.n_q, 128, dtype=torch.float32 if out_f32 else torch.bfloat16, device=bt_d.device)
    lse = torch.empty(w.batch, w.n_q, dtype=torch.float32, device=bt_d.device)
    kvd.kvd_decode_attn(pool.handle, 0, w.q(0, 0, bt_d.device), bt_d, seq_d, max_len, ws, out, num_splits=splits,
                        retain_mask=retain, lse_out=lse, k_new=k_new, v_new=v_new, logits_out=logits)
    assert kvd.kvd_get_device_error(pool.handle) == 0
    return out.float().cpu().numpy(), lse.cpu().numpy()


def _oracle_pool(w, bt, lens):
    import oracle

    pool = oracle.OraclePool(w.num_blocks(), w.n_kv, w.d_h, 16, lowbit=w.lowbit)
    for b in range(w.batch):
        k, v = w.kv(0, b, 0, lens[b])
        assert pool.append(k.float().numpy(), v.float().numpy(), w.slot_mapping(b, 0, lens[b], bt).numpy()) == 0
    return pool


@pytest.mark.parametrize("kind,group", KINDS)
def test_lowbit_codes_scales_and_zeros_are_bit_exact(cuda_device, kind, group):
    """kvd_append_kv writes the oracle's codes, scales and zero points, for every written slot of
    a sample of blocks; rows with 20x outlier channels, a zero row and a constant row included."""
    w = _custom(f"lb_codes_{kind}_{group}", 32, 8, [700, 33, 1601], kind, group, seed=group, outlier_p=0.02,
                outlier_factor=20.0)
    bt, bt_d, seq, seq_d, _ = H.device_inputs(w, cuda_device)
    pool = H.make_pool(w)
    H.fill_layer(pool, w, 0, bt, w.seq_lens(), cuda_device)
    # a zero row and a constant row, appended over position 5 of request 0
    k0 = torch.zeros(1, w.n_kv, 128, dtype=torch.bfloat16)
    v0 = torch.full((1, w.n_kv, 128), 1.25, dtype=torch.bfloat16)
    slot = w.slot_mapping(0, 5, 6, bt)
    kvd.kvd_append_kv(pool.handle, 0, k0.to(cuda_device), v0.to(cuda_device), slot.to(cuda_device))
    assert kvd.kvd_get_device_error(pool.handle) == 0
    opool = _oracle_pool(w, bt, w.seq_lens())
    assert opool.append(k0.float().numpy(), v0.float().numpy(), slot.numpy()) == 0
    written = {}
    for b, n in enumerate(w.seq_lens()):
        for t in range(n):
            written.setdefault(int(bt[b, t // 16]), []).append(t % 16)
    blocks = sorted(written)[:: max(1, len(written) // 12)] + [int(bt[0, 0])]
    for p in blocks:
        sl = sorted(written[p])
        for h in range(w.n_kv):
            kc, vc, ks, kz, vs, vz = H.read_lowbit_record(pool, 0, p, h)
            assert np.array_equal(kc[sl], opool.k_codes[p, h][sl]), (p, h)
            assert np.array_equal(vc[sl], opool.v_codes[p, h][sl]), (p, h)
            assert np.array_equal(ks[sl], opool.k_scales[p, h][sl]) and np.array_equal(kz[sl], opool.k_zeros[p, h][sl])
            assert np.array_equal(vs[sl], opool.v_scales[p, h][sl]) and np.array_equal(vz[sl], opool.v_zeros[p, h][sl])


@pytest.mark.parametrize("kind,group", KINDS)
@pytest.mark.parametrize("g", [1, 4, 7, 8])
def test_lowbit_attention_matches_oracle(cuda_device, kind, group, g):
    """Ragged lengths (partial last blocks, a 1-token request), outlier channels, several split
    counts: fp32 output and LSE against the oracle's fp64 attention over read-back values."""
    n_kv = 4
    w = _custom(f"lb_attn_{kind}_{group}_{g}", g * n_kv, n_kv, [2100, 17, 700, 1, 1601], kind, group, seed=g,
                outlier_p=0.01, outlier_factor=20.0)
    bt, bt_d, seq, seq_d, _ = H.device_inputs(w, cuda_device)
    pool = H.make_pool(w)
    H.fill_layer(pool, w, 0, bt, w.seq_lens(), cuda_device)
    ref = H.oracle_layer(w, 0, bt, w.seq_lens())
    for splits in (0, 7, 1):
        out, lse = _decode(pool, w, bt_d, seq_d, splits)
        H.assert_out_close(out, ref["out"], what=f"{kind} G{group} g {g} splits {splits}")
        np.testing.assert_allclose(lse, ref["lse"], rtol=1e-5, atol=1e-4)


@pytest.mark.parametrize("kind,group", [("int4", 32), ("int2", 128)])
def test_lowbit_fused_append_evicted_slots_and_logits(cuda_device, kind, group):
    """The decode call's fused append writes the new token exactly as kvd_append_kv does (pool bytes
    equal), evicted slots drop out, and the logits written for the score update match the oracle's
    (−inf exactly where evicted)."""
    w = _custom(f"lb_fused_{kind}", 28, 4, [3000, 700, 16, 4100], kind, group, seed=5, evict_frac=0.05,
                protect_prompt=64, protect_recent=32)
    dev = cuda_device
    bt, bt_d, seq, seq_d, ret_d = H.device_inputs(w, dev)
    lens = w.seq_lens()
    prefix = [n - 1 for n in lens]
    ks, vs = zip(*[w.kv(0, b, n - 1, n, dev) for b, n in enumerate(lens)])
    kn, vn = torch.cat(ks).contiguous(), torch.cat(vs).contiguous()
    stride = max(lens) + 5
    runs = []
    for fused in (True, False):
        pool = H.make_pool(w)
        H.fill_layer(pool, w, 0, bt, prefix, dev)
        if not fused:
            slots = torch.cat([w.slot_mapping(b, n - 1, n, bt) for b, n in enumerate(lens)]).to(dev)
            kvd.kvd_append_kv(pool.handle, 0, kn, vn, slots)
        logits = torch.full((w.batch, w.n_q, stride), 7.0, dtype=torch.float32, device=dev)
        out, lse = _decode(pool, w, bt_d, seq_d, 0, retain=ret_d, k_new=kn if fused else None,
                           v_new=vn if fused else None, logits=logits)
        runs.append((pool, out, lse, logits.cpu().numpy()))
    assert torch.equal(runs[0][0].mem, runs[1][0].mem)
    assert np.array_equal(runs[0][1], runs[1][1])
    retain = w.retain_mask(bt).numpy()
    ref = H.oracle_layer(w, 0, bt, lens, retain=torch.from_numpy(retain), want_logits=True)
    H.assert_out_close(runs[0][1], ref["out"], what=f"{kind} fused append")
    np.testing.assert_allclose(runs[0][2], ref["lse"], rtol=1e-5, atol=1e-4)
    got = runs[0][3]
    for b, n in enumerate(lens):
        rl = ref["logits"][b][:, :n]
        gl = got[b][:, :n]
        assert np.array_equal(np.isneginf(gl), np.isneginf(rl))
        fin = np.isfinite(rl)
        np.testing.assert_allclose(gl[fin], rl[fin], rtol=1e-5, atol=1e-5)
        assert np.all(got[b][:, n:] == 7.0)   # nothing written past the context


@pytest.mark.parametrize("kind", ["int4", "int2"])
def test_lowbit_relabelling_is_bitwise_invariant_and_split_agrees(cuda_device, kind):
    """Paging is lossless: another placement of the same blocks gives the same bits (the per-block
    work does not depend on where a block lies); split and non-split agree within 1e-3."""
    w = _custom(f"lb_perm_{kind}", 32, 8, [3333, 900, 64], kind, 32, seed=9)
    bt, bt_d, seq, seq_d, _ = H.device_inputs(w, cuda_device)
    pool = H.make_pool(w)
    H.fill_layer(pool, w, 0, bt, w.seq_lens(), cuda_device)
    a, la = _decode(pool, w, bt_d, seq_d, 41)
    perm = torch.randperm(w.num_blocks(), generator=torch.Generator().manual_seed(3)).to(torch.int32)
    bt2 = torch.where(bt >= 0, perm[bt.clamp(min=0).long()], bt)
    pool2 = H.make_pool(w)
    H.fill_layer(pool2, w, 0, bt2, w.seq_lens(), cuda_device)
    b, lb = _decode(pool2, w, bt2.to(cuda_device), seq_d, 41)
    assert np.array_equal(a, b) and np.array_equal(la, lb)
    one, _ = _decode(pool, w, bt_d, seq_d, 1)
    np.testing.assert_allclose(a, one, atol=H.SPLIT_ATOL, rtol=0)


def test_lowbit_pool_arguments(cuda_device):
    for g in (0, 16, 96, 256):
        with pytest.raises(kvd.KvdError) as e:
            kvd.kvd_pool_bytes(1, 8, 64, kvd.KVD_INT4, group_size=g)
        assert e.value.status == kvd.KVD_ERR_UNSUPPORTED
    pool = kvd.KVPool(1, 8, 64, kvd.KVD_INT2, device=cuda_device, group_size=64)
    with pytest.raises(kvd.KvdError) as e:
        kvd.kvd_pool_attach_host_tier(pool.handle, torch.empty(1 << 20, dtype=torch.uint8, pin_memory=True), None, 4)
    assert e.value.status == kvd.KVD_ERR_UNSUPPORTED
