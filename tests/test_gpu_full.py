"""Full-size workloads in the launch configuration the benchmark times, checked on
sampled outputs the oracle computes one by one, and by properties that hold at any size.

Every device pool is filled through kvd_append_kv from the seeded generator running on
the GPU; the oracle regenerates the sampled requests' K/V on the host from the same
counter-based generator (bit-identical) and never reads device memory.
"""

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
