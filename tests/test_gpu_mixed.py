"""Mixed-precision, tier-homogeneous pages on the GPU against the oracle's mixed pool.

Every physical block holds its K/V in one format — BF16 values, or E4M3 / E5M2 codes with a
per-(token, KV head) fp32 scale — named by a per-block precision byte ("The KV Cache Is the
New Memory Wall", §5.5; "기술 요약: Spherical KV", §2.2).  The oracle's mixed pool
(OraclePool(block_fmt=...)) quantises each block in its own format; the CUDA pool must hold
the same codes and scales bit for bit and attend within the output tolerance.
"""

import numpy as np
import pytest
import torch

import oracle
import paged_gqa_decode_kvd_gb300 as kvd
from kvd_inputs import Workload, gen
from tests import harness as H

pytestmark = pytest.mark.gpu

API = {oracle.FMT_BF16: kvd.KVD_BF16, oracle.FMT_E4M3: kvd.KVD_FP8_E4M3, oracle.FMT_E5M2: kvd.KVD_FP8_E5M2}


def _custom(name, n_q, n_kv, lens, seed=0, L=1, **kw):
    w = Workload(name, L=L, n_q=n_q, n_kv=n_kv, d_h=128, batch=len(lens), kv_dtype="bf16", seed=seed, **kw)
    w._ctx0 = list(lens)
    return w


def _formats(w, probs=(0.3, 0.4, 0.3)):
    """Seeded oracle format code per physical block (0 BF16, 1 E4M3, 2 E5M2)."""
    u = gen.uniform(gen.stream_key(w.seed, w.name, "fmt"), gen.index_range(0, w.num_blocks(), "cpu")).numpy()
    return np.where(u < probs[0], 0, np.where(u < probs[0] + probs[1], 1, 2)).astype(np.uint8)


def _mixed_pool(w, fmt, layers=1, dev="cuda"):
    pool = kvd.KVPool(layers, w.n_kv, w.num_blocks(), kvd.KVD_MIXED, device=dev)
    pool.mem.fill_(0xFF)
    codes = torch.tensor([API[int(f)] for f in fmt], dtype=torch.uint8, device=dev)
    pool.set_block_formats(codes)
    return pool


def _oracle_mixed(w, fmt, bt, lens, layer=0, q=None, retain=None):
    pool = oracle.OraclePool(w.num_blocks(), w.n_kv, w.d_h, 16, block_fmt=fmt)
    for b in range(w.batch):
        k, v = w.kv(layer, b, 0, lens[b])
        assert pool.append(k.float().numpy(), v.float().numpy(), w.slot_mapping(b, 0, lens[b], bt).numpy()) == 0
    if q is None:
        q = w.q(layer, 0)
    res = oracle.decode(pool, q.float().numpy(), w.n_q, bt.numpy(), lens, retain, 1.0 / np.sqrt(w.d_h))
    return pool, res


def _decode(pool, w, bt_d, seq_d, splits=0, retain=None, k_new=None, v_new=None, logits=None):
    max_len = max(w.seq_lens())
    _, ws = H.workspace(pool, w.n_q, w.batch, max_len, splits)
    out = torch.empty(w.batch, w.n_q, 128, dtype=torch.float32, device=bt_d.device)
    lse = torch.empty(w.batch, w.n_q, dtype=torch.float32, device=bt_d.device)
    kvd.kvd_decode_attn(pool.handle, 0, w.q(0, 0, bt_d.device), bt_d, seq_d, max_len, ws, out, num_splits=splits,
                        retain_mask=retain, lse_out=lse, k_new=k_new, v_new=v_new, logits_out=logits)
    assert kvd.kvd_get_device_error(pool.handle) == 0
    return out.cpu().numpy(), lse.cpu().numpy()


def _record(pool, block, head, fmt):
    """(K, V[, K scales, V scales]) of one record of layer 0 as stored, in the token × dim order."""
    off = (block * pool.n_kv + head) * 8192
    raw = pool.mem[off:off + 8192].cpu()
    if fmt == oracle.FMT_BF16:
        vals = raw.view(torch.bfloat16)
        return (vals[:2048][torch.from_numpy(H._tile_perm("k", False))],
                vals[2048:][torch.from_numpy(H._tile_perm("v", False))])
    b = raw.numpy()
    sc = raw[4096:4224].view(torch.float32).numpy()
    return b[:2048][H._tile_perm("k", True)], b[2048:4096][H._tile_perm("v", True)], sc[:16], sc[16:]


@pytest.mark.parametrize("g", [1, 4, 7, 8])
def test_mixed_pool_codes_scales_and_attention_match_oracle(cuda_device, g):
    """Ragged lengths, outlier channels (the 8-bit scales see 20x rows), every group size."""
    n_kv = 4
    w = _custom(f"mixed_g{g}", g * n_kv, n_kv, [2100, 17, 700, 33, 1601], seed=g, outlier_p=0.02,
                outlier_factor=20.0)
    fmt = _formats(w)
    bt, bt_d, seq, seq_d, _ = H.device_inputs(w, cuda_device)
    pool = _mixed_pool(w, fmt, dev=cuda_device)
    H.fill_layer(pool, w, 0, bt, w.seq_lens(), cuda_device)
    assert kvd.kvd_get_device_error(pool.handle) == 0
    opool, ref = _oracle_mixed(w, fmt, bt, w.seq_lens())
    # stored codes and scales: bit for bit, every written slot of a sample of blocks of each format
    written = {}
    for b, n in enumerate(w.seq_lens()):
        for t in range(n):
            written.setdefault(int(bt[b, t // 16]), []).append(t % 16)
    for f in (0, 1, 2):
        for p in [p for p in sorted(written) if fmt[p] == f][:6]:
            sl = sorted(written[p])
            for h in range(n_kv):
                rec = _record(pool, p, h, f)
                if f == 0:
                    assert np.array_equal(rec[0].float().numpy()[sl], opool.k[p, h][sl].astype(np.float32))
                    assert np.array_equal(rec[1].float().numpy()[sl], opool.v[p, h][sl].astype(np.float32))
                else:
                    assert np.array_equal(rec[0][sl], opool.k_codes[p, h][sl])
                    assert np.array_equal(rec[1][sl], opool.v_codes[p, h][sl])
                    assert np.array_equal(rec[2][sl], opool.k_scales[p, h][sl])
                    assert np.array_equal(rec[3][sl], opool.v_scales[p, h][sl])
    for splits in (0, 5, 1):
        out, lse = _decode(pool, w, bt_d, seq_d, splits)
        H.assert_out_close(out, ref["out"], what=f"g {g} splits {splits}")
        np.testing.assert_allclose(lse, ref["lse"], rtol=1e-5, atol=1e-4)


@pytest.mark.parametrize("f", [oracle.FMT_BF16, oracle.FMT_E4M3])
def test_single_format_mixed_pool_equals_the_plain_pool(cuda_device, f):
    """A mixed pool whose blocks are all BF16 (all E4M3) gives the plain BF16 (FP8) pool's output
    bit for bit under the same split count: the per-block path is the plain path."""
    w = _custom(f"mixed_same_{f}", 32, 8, [3000, 17, 1200, 640], seed=11)
    bt, bt_d, seq, seq_d, _ = H.device_inputs(w, cuda_device)
    pool = _mixed_pool(w, np.full(w.num_blocks(), f, np.uint8), dev=cuda_device)
    H.fill_layer(pool, w, 0, bt, w.seq_lens(), cuda_device)
    plain_w = _custom(f"mixed_same_{f}", 32, 8, [3000, 17, 1200, 640], seed=11)
    plain_w.kv_dtype = "bf16" if f == oracle.FMT_BF16 else "fp8_e4m3"
    plain = H.make_pool(plain_w)
    H.fill_layer(plain, plain_w, 0, bt, w.seq_lens(), cuda_device)
    for splits in (37, 300):
        a, la = _decode(pool, w, bt_d, seq_d, splits)
        b, lb = _decode(plain, plain_w, bt_d, seq_d, splits)
        assert np.array_equal(a, b) and np.array_equal(la, lb)


def test_mixed_pool_fused_append_and_evicted_slots(cuda_device):
    """The decode call's fused append writes the new token in its block's own format (bitwise
    equal to kvd_append_kv), and evicted slots drop out, against the oracle."""
    w = _custom("mixed_fused", 28, 4, [3000, 700, 16, 4100], seed=5, evict_frac=0.05, protect_prompt=64,
                protect_recent=32)
    fmt = _formats(w)
    dev = cuda_device
    bt, bt_d, seq, seq_d, ret_d = H.device_inputs(w, dev)
    lens = w.seq_lens()
    prefix = [n - 1 for n in lens]
    pos = [n - 1 for n in lens]
    ks, vs = zip(*[w.kv(0, b, pos[b], pos[b] + 1, dev) for b in range(w.batch)])
    kn, vn = torch.cat(ks).contiguous(), torch.cat(vs).contiguous()
    pools = []
    outs = []
    for fused in (True, False):
        pool = _mixed_pool(w, fmt, dev=dev)
        H.fill_layer(pool, w, 0, bt, prefix, dev)
        if not fused:
            slots = torch.cat([w.slot_mapping(b, pos[b], pos[b] + 1, bt) for b in range(w.batch)]).to(dev)
            kvd.kvd_append_kv(pool.handle, 0, kn, vn, slots)
        out, lse = _decode(pool, w, bt_d, seq_d, 0, retain=ret_d, k_new=kn if fused else None,
                           v_new=vn if fused else None)
        pools.append(pool)
        outs.append((out, lse))
    assert torch.equal(pools[0].mem, pools[1].mem)
    assert np.array_equal(outs[0][0], outs[1][0])
    _, ref = _oracle_mixed(w, fmt, bt, lens, retain=w.retain_mask(bt).numpy())
    H.assert_out_close(outs[0][0], ref["out"], what="mixed fused append")
    np.testing.assert_allclose(outs[0][1], ref["lse"], rtol=1e-5, atol=1e-4)


def test_mixed_pool_bad_format_code_is_reported_not_faulted(cuda_device):
    w = _custom("mixed_badfmt", 32, 8, [900, 400], seed=6)
    fmt = _formats(w)
    bt, bt_d, seq, seq_d, _ = H.device_inputs(w, cuda_device)
    pool = _mixed_pool(w, fmt, dev=cuda_device)
    H.fill_layer(pool, w, 0, bt, w.seq_lens(), cuda_device)
    bad = pool.block_fmt.clone()
    bad[int(bt[0, 3])] = 7
    pool.set_block_formats(bad)
    max_len = max(w.seq_lens())
    _, ws = H.workspace(pool, w.n_q, w.batch, max_len)
    out = torch.empty(w.batch, w.n_q, 128, dtype=torch.float32, device=cuda_device)
    kvd.kvd_decode_attn(pool.handle, 0, w.q(0, 0, cuda_device), bt_d, seq_d, max_len, ws, out)
    assert kvd.kvd_get_device_error(pool.handle) == kvd.KVD_ERR_OOB
    assert np.isfinite(out.cpu().numpy()).all()


def test_block_format_arguments_are_checked(cuda_device):
    w = _custom("mixed_args", 32, 8, [64], seed=7)
    plain = H.make_pool(w)
    codes = torch.zeros(w.num_blocks(), dtype=torch.uint8, device=cuda_device)
    with pytest.raises(kvd.KvdError) as e:
        kvd.kvd_pool_set_block_formats(plain.handle, codes)      # not a mixed pool
    assert e.value.status == kvd.KVD_ERR_INVALID
    pool = kvd.KVPool(1, w.n_kv, w.num_blocks(), kvd.KVD_MIXED, device=cuda_device)
    with pytest.raises(kvd.KvdError) as e:
        kvd.kvd_pool_set_block_formats(pool.handle, codes[:-1])  # fewer codes than blocks
    assert e.value.status == kvd.KVD_ERR_INVALID
    k, v = w.kv(0, 0, 0, 1, cuda_device)
    with pytest.raises(kvd.KvdError) as e:                       # no formats given yet
        kvd.kvd_append_kv(pool.handle, 0, k.contiguous(), v.contiguous(),
                          torch.zeros(1, dtype=torch.int64, device=cuda_device))
    assert e.value.status == kvd.KVD_ERR_INVALID
    with pytest.raises(kvd.KvdError) as e:
        kvd.kvd_pool_attach_host_tier(pool.handle, torch.empty(1 << 20, dtype=torch.uint8, pin_memory=True), None, 4)
    assert e.value.status == kvd.KVD_ERR_UNSUPPORTED
