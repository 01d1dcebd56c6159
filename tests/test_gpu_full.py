"""Full-size workloads in the launch configuration the benchmark times, checked against the
oracle on whole layers (every request, or every KV head of a long request), and by properties
that hold at any size.

Every device pool is filled through kvd_append_kv from the seeded generator running on
the GPU; the oracle regenerates each request's K/V on the host from the same counter-based
generator (bit-identical) and never reads device memory.  Oracle units run on a thread pool
(the C oracle releases the interpreter lock).
"""

import concurrent.futures as cf
import os

import numpy as np
import pytest
import torch

import oracle
import paged_gqa_decode_kvd_gb300 as kvd
from kvd_inputs import get
from tests import harness as H

pytestmark = pytest.mark.gpu


def _device_layer(w, dev, layer, pool, step=0, logits=False, splits=0):
    bt, bt_d, seq, seq_d, ret_d = H.device_inputs(w, dev, step)
    lens = w.seq_lens(step)
    max_len = max(w.seq_lens(w.steps - 1))
    S, ws = H.workspace(pool, w.n_q, w.batch, max_len, splits, dev)
    out = torch.empty(w.batch, w.n_q, 128, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(w.batch, w.n_q, dtype=torch.float32, device=dev)
    lg = torch.full((w.batch, w.n_q, max_len), float("nan"), dtype=torch.float32, device=dev) if logits else None
    kvd.kvd_decode_attn(pool.handle, layer, w.q(layer, step, dev), bt_d, seq_d, max_len, ws, out,
                        num_splits=splits, retain_mask=ret_d, lse_out=lse, logits_out=lg)
    assert kvd.kvd_get_device_error(pool.handle) == 0
    return out.float().cpu().numpy(), lse.cpu().numpy(), lg, bt, S


def _oracle_request(w, layer, b, n, step=0, heads=None, evicted=None):
    """Oracle on one request's regenerated K/V (optionally only the query heads of some KV heads)."""
    k, v = w.kv(layer, b, 0, n)
    q = w.q(layer, step)[b:b + 1]
    n_q = w.n_q
    if heads is not None:                      # restrict to KV heads `heads` and their query groups
        k, v = k[:, heads], v[:, heads]
        q = torch.cat([q[:, h * w.g:(h + 1) * w.g] for h in heads], dim=1)
        n_q = w.g * len(heads)
    return oracle.decode_dense_inputs([k.float().numpy()], [v.float().numpy()], q.float().numpy(), [n], n_q,
                                      evicted=evicted, fp8=w.kv_dtype != "bf16")


def test_llama8b_full_batch_sampled_requests(cuda_device):
    """32 requests x 8,192 tokens, 16,384-block shuffled pool, automatic split plan."""
    w = get("llama8b")
    layers = [0, 31]
    pool = H.make_pool(w)
    bt = w.block_table()
    for layer in layers:
        H.fill_layer(pool, w, layer, bt, w.seq_lens(), cuda_device)
    for layer in layers:
        out, lse, _, _, S = _device_layer(w, cuda_device, layer, pool)
        assert S > 1
        for b in (0, 13, 31):
            ref = _oracle_request(w, layer, b, 8192)
            H.assert_out_close(out[b], ref["out"][0], what=f"layer {layer} request {b}")
            np.testing.assert_allclose(lse[b], ref["lse"][0], rtol=1e-5, atol=1e-4)


def test_ragged_full_batch_sampled_requests(cuda_device):
    """64 requests, contexts log-uniform in [256, 32,768], ragged last blocks."""
    w = get("ragged")
    lens = w.seq_lens()
    pool = H.make_pool(w)
    bt = w.block_table()
    layer = 2
    H.fill_layer(pool, w, layer, bt, lens, cuda_device)
    out, lse, _, _, S = _device_layer(w, cuda_device, layer, pool)
    order = np.argsort(lens)
    for b in [int(order[0]), int(order[-1]), int(order[len(order) // 2]), 7]:
        ref = _oracle_request(w, layer, b, lens[b])
        H.assert_out_close(out[b], ref["out"][0], what=f"request {b} (context {lens[b]})")
        np.testing.assert_allclose(lse[b], ref["lse"][0], rtol=1e-5, atol=1e-4)


def test_llama70b_fp8_full_context_sampled_head(cuda_device):
    """Batch 1 x 131,072 tokens, FP8 pool with outlier channels, split across every SM."""
    w = get("llama70b_fp8")
    pool = H.make_pool(w, layers=1)
    bt = w.block_table()
    H.fill_layer(pool, w, 0, bt, w.seq_lens(), cuda_device)
    out, lse, _, _, S = _device_layer(w, cuda_device, 0, pool)
    assert S >= 152
    kvh = 5
    ref = _oracle_request(w, 0, 0, 131072, heads=[kvh])
    sl = slice(kvh * w.g, (kvh + 1) * w.g)
    H.assert_out_close(out[0, sl], ref["out"][0], what="70B FP8 KV head 5")
    np.testing.assert_allclose(lse[0, sl], ref["lse"][0], rtol=1e-5, atol=1e-4)
    # the appended token of a decode step is quantised exactly as the oracle does it
    kn, vn = w.kv(0, 0, 131071, 131072)
    kc, ks = oracle.quantize_rows(kn.float().numpy())
    p, t = int(bt[0, 131071 // 16]), 131071 % 16
    for h in range(w.n_kv):
        kr, _ = H.read_record(pool, 0, p, h)
        sk, _ = H.read_scales(pool, 0, p, h)
        assert np.array_equal(kr[t], kc[0, h]) and sk[t] == ks[0, h]


def test_tiered_scores_over_64_steps(cuda_device):
    """28 layers, 8 requests, 16,384 + t context, 3% evicted: score sum grows by exactly one per
    step for every request, evicted slots score zero, and two steps of request 0 match the oracle."""
    w = get("tiered")
    dev = cuda_device
    pool = H.make_pool(w)
    bt = w.block_table()
    prefill = [c - 1 for c in w.seq_lens(0)]
    for layer in range(w.L):
        H.fill_layer(pool, w, layer, bt, prefill, dev)
    max_len = max(w.seq_lens(w.steps - 1))
    S, ws = H.workspace(pool, w.n_q, w.batch, max_len, 0, dev)
    ret_d = H.retain_bits(w.retain_mask(bt)).to(dev)
    bt_d = bt.to(dev)
    scores = torch.zeros(w.batch, max_len, dtype=torch.float32, device=dev)
    lse = torch.empty(w.batch, w.n_q, dtype=torch.float32, device=dev)
    logits = torch.empty(w.batch, w.n_q, max_len, dtype=torch.float32, device=dev)
    out = torch.empty(w.batch, w.n_q, 128, dtype=torch.bfloat16, device=dev)
    inv = 1.0 / (w.L * w.n_q)
    kept_s = None
    for t in range(w.steps):
        pos = w.append_pos(t)
        seq_d = torch.tensor(w.seq_lens(t), dtype=torch.int32, device=dev)
        for layer in range(w.L):
            ks, vs = zip(*[w.kv(layer, b, pos[b], pos[b] + 1, dev) for b in range(w.batch)])
            slots = torch.cat([w.slot_mapping(b, pos[b], pos[b] + 1, bt) for b in range(w.batch)]).to(dev)
            kvd.kvd_append_kv(pool.handle, layer, torch.cat(ks), torch.cat(vs), slots)
            if layer % 2:   # both forms of the score update: fused into the call, or separate
                kvd.kvd_decode_attn(pool.handle, layer, w.q(layer, t, dev), bt_d, seq_d, max_len, ws, out,
                                    retain_mask=ret_d, lse_out=lse, logits_out=logits, scores=scores, inv_LH=inv)
            else:
                kvd.kvd_decode_attn(pool.handle, layer, w.q(layer, t, dev), bt_d, seq_d, max_len, ws, out,
                                    retain_mask=ret_d, lse_out=lse, logits_out=logits)
                kvd.kvd_accum_scores(logits, lse, seq_d, inv, scores)
        if t == 1:
            kept_s = scores.clone()
    assert kvd.kvd_get_device_error(pool.handle) == 0
    s = scores.double().cpu().numpy()
    np.testing.assert_allclose(s.sum(axis=1), w.steps, rtol=2e-5)
    for b in range(w.batch):
        assert np.all(s[b, w.evicted_positions(b).numpy()] == 0)
    # oracle: request 0, steps 0 and 1, every layer
    s_ref = np.zeros((1, max_len))
    for t in range(2):
        n = w.seq_lens(t)[0]
        alphas = []
        for layer in range(w.L):
            r = _oracle_request(w, layer, 0, n, step=t, evicted=[w.evicted_positions(0).numpy()])
            a = np.zeros((1, w.n_q, max_len))
            a[:, :, :n] = r["alpha"]
            alphas.append(a)
        s_ref = oracle.score_update(s_ref, np.stack(alphas), [n])
    got = kept_s[0].double().cpu().numpy()
    assert np.all(np.abs(got - s_ref[0]) <= H.SCORE_RTOL * np.abs(s_ref[0]) + 1e-12)



# ------------------------------------------------------------- whole layers, benchmark configuration
def _bench_layer(w, dev, layer, step=0, logits=False):
    """One layer as the benchmark runs it: a one-layer pool holding the context before the step,
    the step plan, then kvd_decode_attn appending the step's token itself (k_new, v_new) with early
    start and the automatic split count."""
    bt, bt_d, seq, seq_d, ret_d = H.device_inputs(w, dev, step)
    lens = w.seq_lens(step)
    pool = H.make_pool(w, layers=1)
    H.fill_layer(pool, w, layer, bt, [n - 1 for n in lens], dev, pool_layer=0)
    kn, vn = zip(*[w.kv(layer, b, n - 1, n, dev) for b, n in enumerate(lens)])
    kn, vn = torch.cat(kn).contiguous(), torch.cat(vn).contiguous()
    max_len = max(w.seq_lens(w.steps - 1))
    S, ws = H.workspace(pool, w.n_q, w.batch, max_len, 0, dev)
    kvd.kvd_decode_plan(pool.handle, w.n_q, bt_d, seq_d, max_len, ws, retain_mask=ret_d)
    out = torch.empty(w.batch, w.n_q, 128, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(w.batch, w.n_q, dtype=torch.float32, device=dev)
    kvd.kvd_decode_attn(pool.handle, 0, w.q(layer, step, dev), bt_d, seq_d, max_len, ws, out, retain_mask=ret_d,
                        lse_out=lse, k_new=kn, v_new=vn, early_start=True, planned=True)
    assert kvd.kvd_get_device_error(pool.handle) == 0
    return out.float().cpu().numpy(), lse.cpu().numpy(), S, pool


def _oracle_unit(w, layer, b, n, step=0, heads=None):
    """Oracle on one request of any pool kind: its regenerated K/V in an identity-ordered pool (a
    mixed pool keeps each block's format from the request's block table), optionally only the query
    heads of some KV heads."""
    k, v = w.kv(layer, b, 0, n)
    q = w.q(layer, step)[b:b + 1]
    n_kv = w.n_kv
    if heads is not None:
        k, v = k[:, heads], v[:, heads]
        q = torch.cat([q[:, h * w.g:(h + 1) * w.g] for h in heads], dim=1)
        n_kv = len(heads)
    q = q.float().numpy()
    nb = -(-n // 16)
    if w.lowbit:
        pool = oracle.OraclePool(nb, n_kv, w.d_h, 16, lowbit=w.lowbit)
    elif w.kv_dtype == "angle":
        pool = oracle.OraclePool(nb, n_kv, w.d_h, 16, angle=True)
        q = oracle.angle_query(q)
    elif w.kv_dtype == "mixed":
        pool = oracle.OraclePool(nb, n_kv, w.d_h, 16, block_fmt=w.block_formats()[w.block_table()[b, :nb].numpy()])
    else:
        pool = oracle.OraclePool(nb, n_kv, w.d_h, 16, w.kv_dtype != "bf16")
    assert pool.append(k.float().numpy(), v.float().numpy(), np.arange(n, dtype=np.int64)) == 0
    return oracle.decode(pool, q, w.g * n_kv, np.arange(nb, dtype=np.int32)[None], [n])


def _pool_map(fn, items):
    with cf.ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 4)) as ex:
        return list(ex.map(fn, items))


@pytest.mark.parametrize("name", ["llama8b", "ragged"])
def test_whole_layer_every_request(cuda_device, name):
    """Every request of one layer (8B: 32 x 8,192 tokens; ragged: 64 contexts in [256, 32,768])."""
    w = get(name)
    layer = w.L - 1
    out, lse, S, _ = _bench_layer(w, cuda_device, layer)
    assert S > 1
    lens = w.seq_lens()
    refs = _pool_map(lambda b: _oracle_unit(w, layer, b, lens[b]), range(w.batch))
    for b, ref in enumerate(refs):
        H.assert_out_close(out[b], ref["out"][0], what=f"{name} layer {layer} request {b}")
        np.testing.assert_allclose(lse[b], ref["lse"][0], rtol=1e-5, atol=1e-4)


@pytest.mark.parametrize("name", ["llama70b_fp8", "llama70b_int4", "llama70b_int2", "llama70b_angle"])
def test_long_context_every_head(cuda_device, name):
    """Batch 1 x 131,072 tokens split across every SM: all 8 KV heads (64 query heads) of one layer."""
    w = get(name)
    layer = w.L - 1
    out, lse, S, _ = _bench_layer(w, cuda_device, layer)
    assert S >= 152
    refs = _pool_map(lambda h: _oracle_unit(w, layer, 0, 131072, heads=[h]), range(w.n_kv))
    for h, ref in enumerate(refs):
        sl = slice(h * w.g, (h + 1) * w.g)
        H.assert_out_close(out[0, sl], ref["out"][0], what=f"{name} KV head {h}")
        np.testing.assert_allclose(lse[0, sl], ref["lse"][0], rtol=1e-5, atol=1e-4)


def test_mixed_precision_whole_layer(cuda_device):
    """8B shape with every physical block BF16 / E4M3 / E5M2: every request of one layer against the
    oracle's mixed pool (each block in the format of the physical block it occupies on the GPU)."""
    w = get("llama8b_mixed")
    layer = w.L - 1
    out, lse, S, _ = _bench_layer(w, cuda_device, layer)
    lens = w.seq_lens()
    refs = _pool_map(lambda b: _oracle_unit(w, layer, b, lens[b]), range(w.batch))
    for b, ref in enumerate(refs):
        H.assert_out_close(out[b], ref["out"][0], what=f"mixed layer request {b}")
        np.testing.assert_allclose(lse[b], ref["lse"][0], rtol=1e-5, atol=1e-4)


def test_tiered_scores_every_request_two_steps(cuda_device):
    """The tiered workload's first two steps, every layer: the importance score of every request
    and position against the oracle's (1/(L·H))·Σ_ℓ Σ_h α, evicted positions included."""
    w = get("tiered")
    dev = cuda_device
    pool = H.make_pool(w)
    bt = w.block_table()
    prefill = [c - 1 for c in w.seq_lens(0)]
    for layer in range(w.L):
        H.fill_layer(pool, w, layer, bt, prefill, dev)
    max_len = max(w.seq_lens(w.steps - 1))
    S, ws = H.workspace(pool, w.n_q, w.batch, max_len, 0, dev)
    ret_d = H.retain_bits(w.retain_mask(bt)).to(dev)
    bt_d = bt.to(dev)
    scores = torch.zeros(w.batch, max_len, dtype=torch.float32, device=dev)
    lse = torch.empty(w.batch, w.n_q, dtype=torch.float32, device=dev)
    logits = torch.empty(w.batch, w.n_q, max_len, dtype=torch.float32, device=dev)
    out = torch.empty(w.batch, w.n_q, 128, dtype=torch.bfloat16, device=dev)
    inv = 1.0 / (w.L * w.n_q)
    for t in range(2):
        pos = w.append_pos(t)
        seq_d = torch.tensor(w.seq_lens(t), dtype=torch.int32, device=dev)
        kvd.kvd_decode_plan(pool.handle, w.n_q, bt_d, seq_d, max_len, ws, retain_mask=ret_d)
        for layer in range(w.L):
            ks, vs = zip(*[w.kv(layer, b, pos[b], pos[b] + 1, dev) for b in range(w.batch)])
            kvd.kvd_decode_attn(pool.handle, layer, w.q(layer, t, dev), bt_d, seq_d, max_len, ws, out,
                                retain_mask=ret_d, lse_out=lse, logits_out=logits, k_new=torch.cat(ks).contiguous(),
                                v_new=torch.cat(vs).contiguous(), early_start=True, planned=True)
            kvd.kvd_accum_scores(logits, lse, seq_d, inv, scores)
    assert kvd.kvd_get_device_error(pool.handle) == 0
    got = scores.double().cpu().numpy()

    def alpha(args):
        layer, b, t = args
        n = w.seq_lens(t)[b]
        r = _oracle_request(w, layer, b, n, step=t, evicted=[w.evicted_positions(b).numpy()])
        return r["alpha"][0]

    for b in range(w.batch):
        s_ref = np.zeros((1, max_len))
        for t in range(2):
            n = w.seq_lens(t)[b]
            al = _pool_map(alpha, [(layer, b, t) for layer in range(w.L)])
            a = np.zeros((w.L, 1, w.n_q, max_len))
            for layer in range(w.L):
                a[layer, 0, :, :n] = al[layer]
            s_ref = oracle.score_update(s_ref, a, [n])
        assert np.all(np.abs(got[b] - s_ref[0]) <= H.SCORE_RTOL * np.abs(s_ref[0]) + 1e-12), b
