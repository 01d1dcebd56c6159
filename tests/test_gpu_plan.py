"""The step plan (kvd_decode_plan + KVD_PLANNED): a decode that reads its split and first blocks
from the plan streams the same blocks as one that derives them (logits and fused appends bit for
bit, for every pool kind, for several layers sharing one plan, with a host tier).  With the plan the
work is balanced dynamically (the last sixth of every CTA's range is cut into pieces that any CTA
takes once its own part is done), so the partials and their merge order differ: outputs agree to
fp32 rounding and with the oracle, and repeat bit for bit (a piece's partial does not depend on the
CTA that takes it).  Bad lengths and block ids are reported the same way."""

import numpy as np
import pytest
import torch

import paged_gqa_decode_kvd_gb300 as kvd
from kvd_inputs import Workload
from tests import harness as H

pytestmark = pytest.mark.gpu


def _custom(name, n_q, n_kv, lens, kv_dtype="bf16", seed=0, L=1, **kw):
    w = Workload(name, L=L, n_q=n_q, n_kv=n_kv, d_h=128, batch=len(lens), kv_dtype=kv_dtype, seed=seed, **kw)
    w._ctx0 = list(lens)
    return w


def _run(pool, w, layer, bt_d, seq_d, ws, splits, planned, retain=None, k_new=None, v_new=None, logits=None):
    max_len = max(w.seq_lens())
    out = torch.empty(w.batch, w.n_q, 128, dtype=torch.float32, device=bt_d.device)
    lse = torch.empty(w.batch, w.n_q, dtype=torch.float32, device=bt_d.device)
    kvd.kvd_decode_attn(pool.handle, layer, w.q(layer, 0, bt_d.device), bt_d, seq_d, max_len, ws, out,
                        num_splits=splits, retain_mask=retain, lse_out=lse, k_new=k_new, v_new=v_new,
                        logits_out=logits, early_start=True, planned=planned)
    return out, lse


KINDS = [("bf16", 0), ("fp8_e4m3", 0), ("mixed", 0), ("int4", 32), ("int2", 128), ("angle", 0)]


@pytest.mark.parametrize("kind,group", KINDS)
def test_planned_decode_equals_unplanned(cuda_device, kind, group):
    """Ragged lengths (a 1-token request, partial blocks), evicted slots, fused append, logits, two
    layers decoded from one plan, several split counts: every output bit equal."""
    extra = dict(group_size=group) if group else {}
    if kind == "mixed":
        extra["mixed_probs"] = (0.3, 0.4, 0.3)
    w = _custom(f"plan_{kind}", 28, 4, [2100, 1, 700, 33, 1601], kind, seed=3, L=2, evict_frac=0.05,
                protect_prompt=64, protect_recent=32, **extra)
    dev = cuda_device
    bt, bt_d, seq, seq_d, ret_d = H.device_inputs(w, dev)
    lens = w.seq_lens()
    kn, vn = zip(*[w.kv(0, b, n - 1, n, dev) for b, n in enumerate(lens)])
    kn, vn = torch.cat(kn).contiguous(), torch.cat(vn).contiguous()
    for splits in (0, 23, 5, 1):   # 5 and 1: ranges long enough for run-time balancing
        res = []
        for planned in (False, True):
            pool = H.make_pool(w, layers=2)
            for layer in range(2):
                H.fill_layer(pool, w, layer, bt, [n - 1 for n in lens], dev)
            _, ws = H.workspace(pool, w.n_q, w.batch, max(lens), splits)
            if planned:
                kvd.kvd_decode_plan(pool.handle, w.n_q, bt_d, seq_d, max(lens), ws, num_splits=splits,
                                    retain_mask=ret_d)
            outs = []
            for layer in range(2):
                logits = torch.full((w.batch, w.n_q, max(lens)), 3.0, dtype=torch.float32, device=dev)
                out, lse = _run(pool, w, layer, bt_d, seq_d, ws, splits, planned, ret_d, kn, vn, logits)
                outs += [out.cpu(), lse.cpu(), logits.cpu()]
            assert kvd.kvd_get_device_error(pool.handle) == 0
            res.append((outs, pool.mem.cpu()))
        for i, (a, b) in enumerate(zip(res[0][0], res[1][0])):
            if i % 3 == 2:
                assert torch.equal(a, b)           # logits: the same blocks, the same arithmetic
            else:                                  # out / lse: other partials, another merge order
                torch.testing.assert_close(b, a, rtol=0, atol=H.SPLIT_ATOL)
        assert torch.equal(res[0][1], res[1][1])   # the fused appends wrote the same bytes
        if splits == 0:   # layer 0 (both layers append layer 0's new token)
            ref = H.oracle_layer(w, 0, bt, lens, retain=w.retain_mask(bt))
            H.assert_out_close(res[1][0][0].numpy(), ref["out"], what=f"{kind} planned layer 0")
            np.testing.assert_allclose(res[1][0][1].numpy(), ref["lse"], rtol=1e-5, atol=1e-4)


@pytest.mark.parametrize("staged,splits", [(False, 0), (True, 0), (False, 8)])
def test_planned_decode_with_a_host_tier(cuda_device, staged, splits):
    """8 splits: ranges of 373 blocks, so the run-time balancing's pieces (taken by any CTA) hold
    host-tier blocks read in place."""
    w = _custom("plan_tier", 32, 8, [3000, 900, 2048], seed=4)
    dev = cuda_device
    bt, bt_d, seq, seq_d, _ = H.device_inputs(w, dev)
    pool = H.make_pool(w)
    H.fill_layer(pool, w, 0, bt, w.seq_lens(), dev)
    nh = 40
    pool.attach_host_tier(nh, staged=staged)
    # move every 5th block of request 0 to the host tier
    ids = bt[0, : (w.seq_lens()[0] + 15) // 16: 5].clone()
    to = torch.arange(w.num_blocks(), w.num_blocks() + len(ids), dtype=torch.int32)
    kvd.kvd_tier_move(pool.handle, ids.to(dev), to.to(dev))
    bt2 = bt.clone()
    bt2[0, : (w.seq_lens()[0] + 15) // 16: 5] = to
    bt2_d = bt2.to(dev)
    if staged:
        kvd.kvd_tier_prefetch(pool.handle, 0)
    _, ws = H.workspace(pool, w.n_q, w.batch, max(w.seq_lens()), splits)
    a, la = _run(pool, w, 0, bt2_d, seq_d, ws, splits, False)
    kvd.kvd_decode_plan(pool.handle, w.n_q, bt2_d, seq_d, max(w.seq_lens()), ws, num_splits=splits)
    b, lb = _run(pool, w, 0, bt2_d, seq_d, ws, splits, True)
    assert kvd.kvd_get_device_error(pool.handle) == 0
    torch.testing.assert_close(b, a, rtol=0, atol=H.SPLIT_ATOL)
    torch.testing.assert_close(lb, la, rtol=1e-5, atol=1e-4)


def test_plan_reports_bad_lengths_and_ids(cuda_device):
    w = _custom("plan_bad", 32, 8, [900, 400, 64], seed=6)
    dev = cuda_device
    bt, bt_d, seq, seq_d, _ = H.device_inputs(w, dev)
    pool = H.make_pool(w)
    H.fill_layer(pool, w, 0, bt, w.seq_lens(), dev)
    _, ws = H.workspace(pool, w.n_q, w.batch, 900, 0)
    bad = bt.clone()
    bad[0, 0] = w.num_blocks() + 7            # a block id outside the pool, in some CTA's first batch
    kvd.kvd_decode_plan(pool.handle, w.n_q, bad.to(dev), seq_d, 900, ws)
    out, _ = _run(pool, w, 0, bad.to(dev), seq_d, ws, 0, True)
    assert kvd.kvd_get_device_error(pool.handle) == kvd.KVD_ERR_OOB
    assert np.isfinite(out.cpu().numpy()).all()
    seq_bad = seq.clone()
    seq_bad[2] = 0                             # a length below 1
    kvd.kvd_decode_plan(pool.handle, w.n_q, bt_d, seq_bad.to(dev), 900, ws)
    out, _ = _run(pool, w, 0, bt_d, seq_bad.to(dev), ws, 0, True)
    assert kvd.kvd_get_device_error(pool.handle) == kvd.KVD_ERR_OOB
    assert np.isfinite(out.cpu().numpy()).all()


def test_plan_arguments(cuda_device):
    w = _custom("plan_args", 32, 8, [64], seed=7)
    dev = cuda_device
    bt, bt_d, seq, seq_d, _ = H.device_inputs(w, dev)
    pool = H.make_pool(w)
    s, nbytes = kvd.kvd_decode_workspace_bytes(pool.handle, w.n_q, 1, 64)
    small = torch.empty(nbytes - 256, dtype=torch.uint8, device=dev)
    with pytest.raises(kvd.KvdError) as e:
        kvd.kvd_decode_plan(pool.handle, w.n_q, bt_d, seq_d, 64, small)
    assert e.value.status == kvd.KVD_ERR_NOMEM
    out = torch.empty(1, w.n_q, 128, dtype=torch.float32, device=dev)
    lib = kvd.load()
    import ctypes

    st = lib.kvd_decode_attn_noalloc(pool.handle, 0, ctypes.c_void_p(w.q(0, 0, dev).data_ptr()), w.n_q, None, None,
                                     ctypes.c_void_p(bt_d.data_ptr()), bt.shape[1], ctypes.c_void_p(seq_d.data_ptr()),
                                     1, 64, 0, None, 0.1, ctypes.c_void_p(out.data_ptr()), kvd.KVD_F32, None, None, 0,
                                     None, kvd.KVD_PLANNED, None)
    assert st == kvd.KVD_ERR_INVALID


@pytest.mark.parametrize("kind,splits", [("bf16", 0), ("fp8_e4m3", 0), ("bf16", 1000), ("bf16", 16), ("fp8_e4m3", 7)])
def test_planned_units_spread_over_every_cta(cuda_device, kind, splits):
    """One KV head per request and g = 8: request 0 (40,000 tokens) is one unit cut into hundreds of
    pieces, request 1 (20,000 tokens) has every slot evicted (all its pieces have lse = -inf), and
    1000 splits put more CTAs in the grid than fit at once; 16 and 7 splits give ranges long enough
    for run-time balancing.  Five launches share one plan and repeat
    bit for bit (the piece counters are back at zero after each); planned equals unplanned to fp32
    rounding; request 0 matches the oracle, request 1 is out = 0, lse = -inf."""
    w = _custom(f"spread_{kind}", 8, 1, [40000, 20000], kind, seed=11)
    dev = cuda_device
    bt, bt_d, seq, seq_d, _ = H.device_inputs(w, dev)
    lens = w.seq_lens()
    pool = H.make_pool(w)
    H.fill_layer(pool, w, 0, bt, lens, dev)
    mask = torch.full((w.num_blocks(),), 0xFFFF, dtype=torch.int32)
    mask[bt[1, : (lens[1] + 15) // 16].long()] = 0
    ret_d = H.retain_bits(mask).to(dev)
    _, ws = H.workspace(pool, w.n_q, w.batch, max(lens), splits)
    kvd.kvd_decode_plan(pool.handle, w.n_q, bt_d, seq_d, max(lens), ws, num_splits=splits, retain_mask=ret_d)
    outs = [_run(pool, w, 0, bt_d, seq_d, ws, splits, True, ret_d) for _ in range(5)]
    assert kvd.kvd_get_device_error(pool.handle) == 0
    for o, l in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(l, outs[0][1])
    out, lse = outs[0]
    assert torch.all(out[1] == 0) and torch.all(torch.isneginf(lse[1]))
    a, la = _run(pool, w, 0, bt_d, seq_d, ws, splits, False, ret_d)
    torch.testing.assert_close(out, a, rtol=0, atol=H.SPLIT_ATOL)
    torch.testing.assert_close(lse, la, rtol=1e-5, atol=1e-4)
    ref = H.oracle_layer(w, 0, bt, lens, retain=mask)
    H.assert_out_close(out[0].cpu().numpy(), ref["out"][0], what=f"{kind} spread unit")
    np.testing.assert_allclose(lse[0].cpu().numpy(), ref["lse"][0], rtol=1e-5, atol=1e-4)


@pytest.mark.parametrize("splits", [0, 4])
def test_planned_decode_with_fused_scores(cuda_device, splits):
    """The fused score update (merge launch) of a planned decode against the standalone score update
    after an unplanned one (4 splits: ranges long enough for run-time balancing); without lse_out
    the fused update is rejected before any launch (it reads the LSEs the decode kernel finished
    there)."""
    w = _custom("plan_scores", 28, 4, [5000, 700, 3100, 16], seed=12, evict_frac=0.04, protect_prompt=64,
                protect_recent=32)
    dev = cuda_device
    bt, bt_d, seq, seq_d, ret_d = H.device_inputs(w, dev)
    lens = w.seq_lens()
    pool = H.make_pool(w)
    H.fill_layer(pool, w, 0, bt, lens, dev)
    _, ws = H.workspace(pool, w.n_q, w.batch, max(lens), splits)
    stride = max(lens) + 5
    base = torch.rand(w.batch, stride, generator=torch.Generator().manual_seed(5)).to(dev)
    res = []
    for planned in (False, True):
        scores = base.clone()
        logits = torch.empty(w.batch, w.n_q, stride, dtype=torch.float32, device=dev)
        out = torch.empty(w.batch, w.n_q, 128, dtype=torch.float32, device=dev)
        lse = torch.empty(w.batch, w.n_q, dtype=torch.float32, device=dev)
        if planned:
            kvd.kvd_decode_plan(pool.handle, w.n_q, bt_d, seq_d, max(lens), ws, num_splits=splits,
                                retain_mask=ret_d)
            kvd.kvd_decode_attn(pool.handle, 0, w.q(0, 0, dev), bt_d, seq_d, max(lens), ws, out, num_splits=splits,
                                retain_mask=ret_d, lse_out=lse, logits_out=logits, scores=scores,
                                inv_LH=1.0 / (3 * w.n_q), early_start=True, planned=True)
        else:
            kvd.kvd_decode_attn(pool.handle, 0, w.q(0, 0, dev), bt_d, seq_d, max(lens), ws, out, num_splits=splits,
                                retain_mask=ret_d, lse_out=lse, logits_out=logits)
            kvd.kvd_accum_scores(logits, lse, seq_d, 1.0 / (3 * w.n_q), scores)
        assert kvd.kvd_get_device_error(pool.handle) == 0
        res.append((out.cpu(), scores.cpu()))
    torch.testing.assert_close(res[1][0], res[0][0], rtol=0, atol=H.SPLIT_ATOL)
    torch.testing.assert_close(res[1][1], res[0][1], rtol=1e-5, atol=1e-7)
    with pytest.raises(kvd.KvdError) as e:
        kvd.kvd_decode_attn(pool.handle, 0, w.q(0, 0, dev), bt_d, seq_d, max(lens), ws, out, num_splits=splits,
                            logits_out=logits, scores=scores, inv_LH=1.0, planned=True)
    assert e.value.status == kvd.KVD_ERR_INVALID
