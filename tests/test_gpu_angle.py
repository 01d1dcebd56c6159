"""Angle-domain keys on the GPU against the oracle ("기술 요약: Spherical KV", §2.1, Angle-Domain
Attention): every key row is kept as the E4M3 code of its direction and its logit factor
w = half(||k||)/||d_k||, values as FP8; the kernel codes each query head the same way and computes
the logit ||q||·r̃·cos(d_q, d_k) from the codes.  The oracle's angle pool (OraclePool(angle=True))
with its query passed through angle_query computes the same logits in fp64.
"""

import numpy as np
import pytest
import torch

import oracle
import paged_gqa_decode_kvd_gb300 as kvd
from kvd_inputs import Workload
from tests import harness as H

pytestmark = pytest.mark.gpu


def _custom(name, n_q, n_kv, lens, seed=0, **kw):
    w = Workload(name, L=1, n_q=n_q, n_kv=n_kv, d_h=128, batch=len(lens), kv_dtype="angle", seed=seed, **kw)
    w._ctx0 = list(lens)
    return w


def _decode(pool, w, bt_d, seq_d, splits=0, retain=None, k_new=None, v_new=None, logits=None):
    max_len = max(w.seq_lens())
    _, ws = H.workspace(pool, w.n_q, w.batch, max_len, splits)
    out = torch.empty(w.batch, w.n_q, 128, dtype=torch.float32, device=bt_d.device)
    lse = torch.empty(w.batch, w.n_q, dtype=torch.float32, device=bt_d.device)
    kvd.kvd_decode_attn(pool.handle, 0, w.q(0, 0, bt_d.device), bt_d, seq_d, max_len, ws, out, num_splits=splits,
                        retain_mask=retain, lse_out=lse, k_new=k_new, v_new=v_new, logits_out=logits)
    assert kvd.kvd_get_device_error(pool.handle) == 0
    return out.cpu().numpy(), lse.cpu().numpy()


def test_angle_codes_factors_and_value_scales_are_bit_exact(cuda_device):
    """kvd_append_kv stores the oracle's direction codes, its logit factors w (fp64 arithmetic, so bit
    for bit) and its FP8 value codes and scales; rows with 20x outlier channels, a zero row included."""
    w = _custom("ang_codes", 32, 8, [700, 33, 1601], seed=1, outlier_p=0.02, outlier_factor=20.0)
    bt, bt_d, seq, seq_d, _ = H.device_inputs(w, cuda_device)
    pool = H.make_pool(w)
    H.fill_layer(pool, w, 0, bt, w.seq_lens(), cuda_device)
    zero = torch.zeros(1, w.n_kv, 128, dtype=torch.bfloat16)
    slot = w.slot_mapping(0, 5, 6, bt)
    kvd.kvd_append_kv(pool.handle, 0, zero.to(cuda_device), zero.to(cuda_device), slot.to(cuda_device))
    assert kvd.kvd_get_device_error(pool.handle) == 0
    opool = oracle.OraclePool(w.num_blocks(), w.n_kv, 128, 16, angle=True)
    for b, n in enumerate(w.seq_lens()):
        k, v = w.kv(0, b, 0, n)
        assert opool.append(k.float().numpy(), v.float().numpy(), w.slot_mapping(b, 0, n, bt).numpy()) == 0
    assert opool.append(zero.float().numpy(), zero.float().numpy(), slot.numpy()) == 0
    written = {}
    for b, n in enumerate(w.seq_lens()):
        for t in range(n):
            written.setdefault(int(bt[b, t // 16]), []).append(t % 16)
    for p in sorted(written)[::7] + [int(bt[0, 0])]:
        sl = sorted(written[p])
        for h in range(w.n_kv):
            kc, vc = H.read_record(pool, 0, p, h)
            kw, vs = H.read_scales(pool, 0, p, h)
            assert np.array_equal(kc[sl], opool.k_codes[p, h][sl])
            assert np.array_equal(vc[sl], opool.v_codes[p, h][sl])
            assert np.array_equal(kw[sl], opool.k_scales[p, h][sl]), (p, h)
            assert np.array_equal(vs[sl], opool.v_scales[p, h][sl])
    assert H.read_scales(pool, 0, int(bt[0, 0]), 0)[0][5] == 0.0   # the zero row: w = 0


@pytest.mark.parametrize("g", [1, 4, 7, 8])
def test_angle_attention_matches_oracle(cuda_device, g):
    """Ragged lengths (partial last blocks, a 1-token request), outlier channels, several split counts:
    fp32 output and LSE against the oracle's fp64 attention with the angle-coded query."""
    n_kv = 4
    w = _custom(f"ang_attn_{g}", g * n_kv, n_kv, [2100, 17, 700, 1, 1601], seed=g, outlier_p=0.01,
                outlier_factor=20.0)
    bt, bt_d, seq, seq_d, _ = H.device_inputs(w, cuda_device)
    pool = H.make_pool(w)
    H.fill_layer(pool, w, 0, bt, w.seq_lens(), cuda_device)
    ref = H.oracle_layer(w, 0, bt, w.seq_lens())
    for splits in (0, 7, 1):
        out, lse = _decode(pool, w, bt_d, seq_d, splits)
        H.assert_out_close(out, ref["out"], what=f"angle g {g} splits {splits}")
        np.testing.assert_allclose(lse, ref["lse"], rtol=1e-5, atol=1e-4)


def test_angle_fused_append_evicted_slots_and_logits(cuda_device):
    """The fused append writes the new token exactly as kvd_append_kv does, evicted slots drop out, and
    the logits ||q||·r̃·cos(d_q, d_k)·scale written for the score update match the oracle's (-inf where
    evicted)."""
    w = _custom("ang_fused", 28, 4, [3000, 700, 16, 4100], seed=5, evict_frac=0.05, protect_prompt=64,
                protect_recent=32)
    dev = cuda_device
    bt, bt_d, seq, seq_d, ret_d = H.device_inputs(w, dev)
    lens = w.seq_lens()
    ks, vs = zip(*[w.kv(0, b, n - 1, n, dev) for b, n in enumerate(lens)])
    kn, vn = torch.cat(ks).contiguous(), torch.cat(vs).contiguous()
    stride = max(lens) + 3
    runs = []
    for fused in (True, False):
        pool = H.make_pool(w)
        H.fill_layer(pool, w, 0, bt, [n - 1 for n in lens], dev)
        if not fused:
            slots = torch.cat([w.slot_mapping(b, n - 1, n, bt) for b, n in enumerate(lens)]).to(dev)
            kvd.kvd_append_kv(pool.handle, 0, kn, vn, slots)
        logits = torch.full((w.batch, w.n_q, stride), 7.0, dtype=torch.float32, device=dev)
        out, lse = _decode(pool, w, bt_d, seq_d, 0, retain=ret_d, k_new=kn if fused else None,
                           v_new=vn if fused else None, logits=logits)
        runs.append((pool, out, lse, logits.cpu().numpy()))
    assert torch.equal(runs[0][0].mem, runs[1][0].mem)
    assert np.array_equal(runs[0][1], runs[1][1])
    ref = H.oracle_layer(w, 0, bt, lens, retain=w.retain_mask(bt), want_logits=True)
    H.assert_out_close(runs[0][1], ref["out"], what="angle fused append")
    got = runs[0][3]
    for b, n in enumerate(lens):
        rl, gl = ref["logits"][b][:, :n], got[b][:, :n]
        assert np.array_equal(np.isneginf(gl), np.isneginf(rl))
        fin = np.isfinite(rl)
        np.testing.assert_allclose(gl[fin], rl[fin], rtol=1e-5, atol=1e-5)
        assert np.all(got[b][:, n:] == 7.0)


def test_angle_relabelling_is_bitwise_invariant(cuda_device):
    w = _custom("ang_perm", 32, 8, [3333, 900, 64], seed=9)
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
