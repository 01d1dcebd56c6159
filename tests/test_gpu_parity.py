"""Parity of the CUDA path (through the C ABI) with the fp64 oracle on seeded inputs.

Sizes here run the oracle in seconds yet span many 16-token blocks, several
splits and ragged tails; the full-size workloads are in test_gpu_full.py.
"""

import numpy as np
import pytest
import torch

import oracle
import paged_gqa_decode_kvd_gb300 as kvd
from kvd_inputs import Workload, gen, get
from tests import harness as H

pytestmark = pytest.mark.gpu


def _custom(name, n_q, n_kv, lens, kv_dtype="bf16", L=1, seed=0, **kw):
    w = Workload(name, L=L, n_q=n_q, n_kv=n_kv, d_h=128, batch=len(lens), kv_dtype=kv_dtype, seed=seed, **kw)
    w._ctx0 = list(lens)
    return w


def _run(w, dev, num_splits=0, out_f32=False, want_logits=False, layer=0, pool=None, fill=True, retain=True):
    bt, bt_d, seq, seq_d, ret_d = H.device_inputs(w, dev)
    if pool is None:
        pool = H.make_pool(w, layers=layer + 1)
    if fill:
        H.fill_layer(pool, w, layer, bt, w.seq_lens(), dev)
    S, ws = H.workspace(pool, w.n_q, w.batch, max(w.seq_lens()), num_splits, dev)
    q = w.q(layer, 0, dev)
    out = torch.empty(w.batch, w.n_q, 128, dtype=torch.float32 if out_f32 else torch.bfloat16, device=dev)
    lse = torch.empty(w.batch, w.n_q, dtype=torch.float32, device=dev)
    logits = None
    if want_logits:
        logits = torch.full((w.batch, w.n_q, max(w.seq_lens())), float("nan"), dtype=torch.float32, device=dev)
    kvd.kvd_decode_attn(pool.handle, layer, q, bt_d, seq_d, max(w.seq_lens()), ws, out, num_splits=num_splits,
                        retain_mask=ret_d if retain else None, lse_out=lse, logits_out=logits)
    err = kvd.kvd_get_device_error(pool.handle)
    return dict(out=out.float().cpu().numpy(), lse=lse.cpu().numpy(), splits=S, pool=pool, err=err,
                logits=None if logits is None else logits.cpu().numpy(), bt=bt)


def test_generator_identical_on_cpu_and_cuda(cuda_device):
    w = get("llama70b_fp8")
    kc, vc = w.kv(5, 0, 1000, 1100)
    kg, vg = w.kv(5, 0, 1000, 1100, cuda_device)
    assert torch.equal(kc, kg.cpu()) and torch.equal(vc, vg.cpu())
    assert torch.equal(w.q(3, 2), w.q(3, 2, cuda_device).cpu())
    key = gen.stream_key(1, "x")
    assert torch.equal(gen.uniform(key, gen.index_range(0, 4096, "cpu")),
                       gen.uniform(key, gen.index_range(0, 4096, cuda_device)).cpu())


def test_append_bf16_stores_exact_values(cuda_device):
    w = _custom("app_bf16", 8, 4, [37, 5, 64])
    w.pool_slack_blocks = 7
    bt = w.block_table()
    pool = H.make_pool(w)
    H.fill_layer(pool, w, 0, bt, w.seq_lens(), cuda_device)
    assert kvd.kvd_get_device_error(pool.handle) == 0
    for b, n in enumerate(w.seq_lens()):
        k, v = w.kv(0, b, 0, n)
        for pos in range(n):
            p, t = int(bt[b, pos // 16]), pos % 16
            for h in range(w.n_kv):
                kr, vr = H.read_record(pool, 0, p, h)
                assert torch.equal(kr[t], k[pos, h]) and torch.equal(vr[t], v[pos, h])


def test_append_fp8_codes_and_scales_bit_exact(cuda_device):
    w = _custom("app_fp8", 8, 2, [40, 17], kv_dtype="fp8_e4m3", outlier_p=0.05, outlier_factor=20.0)
    bt = w.block_table()
    pool = H.make_pool(w)
    H.fill_layer(pool, w, 0, bt, w.seq_lens(), cuda_device)
    assert kvd.kvd_get_device_error(pool.handle) == 0
    for b, n in enumerate(w.seq_lens()):
        k, v = w.kv(0, b, 0, n)
        kc, ks = oracle.quantize_rows(k.float().numpy())
        vc, vs = oracle.quantize_rows(v.float().numpy())
        for pos in range(n):
            p, t = int(bt[b, pos // 16]), pos % 16
            for h in range(w.n_kv):
                kr, vr = H.read_record(pool, 0, p, h)
                sk, sv = H.read_scales(pool, 0, p, h)
                assert np.array_equal(kr[t], kc[pos, h]) and np.array_equal(vr[t], vc[pos, h])
                assert sk[t] == ks[pos, h] and sv[t] == vs[pos, h]


def test_fp8_quantise_matches_oracle_on_edge_rows(cuda_device):
    """Zero rows, ties, tiny and huge magnitudes, negative zero: codes and scales bit-exact."""
    n_kv = 1
    rows = []
    r = np.random.default_rng(3)
    rows.append(np.zeros(128))
    rows.append(np.r_[np.full(127, -0.0), [0.0]])
    x = r.standard_normal(128) * 1e-30
    rows.append(x)
    rows.append(r.standard_normal(128) * 1e30)
    y = np.linspace(-448, 448, 128)
    rows.append(y)
    d = oracle.e4m3_decode(np.arange(127, dtype=np.uint8))
    mids = (d[1:] + d[:-1]) / 2           # exact ties once divided by scale 1 (absmax 448)
    rows.append(np.r_[mids, [448.0, -448.0]])
    for _ in range(26):
        rows.append(r.standard_normal(128) * np.exp2(r.uniform(-20, 20)))
    xs = torch.tensor(np.array(rows), dtype=torch.float32).to(torch.bfloat16)      # [N][128]
    N = xs.shape[0]
    pool = kvd.KVPool(1, n_kv, (N + 15) // 16, kvd.KVD_FP8_E4M3)
    kd = xs.view(N, 1, 128).to(cuda_device).contiguous()
    slots = torch.arange(N, dtype=torch.int64, device=cuda_device)
    kvd.kvd_append_kv(pool.handle, 0, kd, kd, slots)
    codes, scales = oracle.quantize_rows(xs.float().numpy())
    for n in range(N):
        kr, vr = H.read_record(pool, 0, n // 16, 0)
        sk, _ = H.read_scales(pool, 0, n // 16, 0)
        assert np.array_equal(kr[n % 16], codes[n]), n
        assert sk[n % 16] == scales[n], n


def test_tiny_workload_parity(cuda_device):
    """1 layer, batch 1, n_q 32, n_kv 8, context 2,048 in 128 blocks of a shuffled 256-block pool."""
    w = get("tiny")
    r16 = _run(w, cuda_device)
    r32 = _run(w, cuda_device, out_f32=True, pool=r16["pool"], fill=False)
    assert r16["err"] == 0 and r32["err"] == 0
    ref = H.oracle_layer(w, 0, r16["bt"], w.seq_lens())
    H.assert_out_close(r16["out"], ref["out"])
    H.assert_out_close(r32["out"], ref["out"])
    np.testing.assert_allclose(r32["lse"], ref["lse"], rtol=1e-5, atol=1e-4)


def test_page_block_table_example(cuda_device):
    """Requests A, B, C of the page's example (11 physical blocks), ragged last blocks."""
    tables = {"A": [0, 4], "B": [1, 2, 5, 6, 8, 9], "C": [3, 7, 10]}
    lens = [20, 90, 33]
    w = _custom("page_example", 32, 8, lens)
    bt = torch.full((3, 6), -1, dtype=torch.int32)
    for i, name in enumerate("ABC"):
        bt[i, :len(tables[name])] = torch.tensor(tables[name])
    w.block_table = lambda: bt.clone()
    w.num_blocks = lambda: 11
    res = _run(w, cuda_device, out_f32=True)
    assert res["err"] == 0
    ref = H.oracle_layer(w, 0, bt, lens)
    H.assert_out_close(res["out"], ref["out"])


def test_relabelling_physical_blocks_is_bitwise_invariant(cuda_device):
    w = _custom("relabel", 16, 4, [300, 77, 129, 1], pool_slack_blocks=20)
    base = _run(w, cuda_device, num_splits=7, out_f32=True)
    perm = gen.permutation(gen.stream_key(9, "relabel"), w.num_blocks())
    orig = w.block_table()
    relab = torch.where(orig >= 0, perm[orig.clamp(min=0).long()].to(torch.int32), orig)
    w.block_table = lambda: relab.clone()
    other = _run(w, cuda_device, num_splits=7, out_f32=True)
    assert np.array_equal(base["out"], other["out"]) and np.array_equal(base["lse"], other["lse"])


@pytest.mark.parametrize("g", [1, 2, 4, 7, 8])
def test_ragged_lengths_every_group_size(cuda_device, g):
    lens = [1, 15, 16, 17, 31, 33, 250, 1000, 2047, 5]
    w = _custom(f"ragged_g{g}", 2 * g, 2, lens, seed=g)
    for splits in (0, 1, 13):
        res = _run(w, cuda_device, num_splits=splits, out_f32=True)
        assert res["err"] == 0
        ref = H.oracle_layer(w, 0, res["bt"], lens)
        H.assert_out_close(res["out"], ref["out"], what=f"g={g} splits={splits}")
        np.testing.assert_allclose(res["lse"], ref["lse"], rtol=1e-5, atol=1e-4)


@pytest.mark.parametrize("g", [1, 2, 4, 7, 8])
def test_fp8_ragged_lengths_every_group_size(cuda_device, g):
    """The FP8 pool (E4M3 codes, per-(token, head) scales, 20x outlier channels) for every group
    size, lengths around the block edges, one CTA, the planned split and 13 splits."""
    lens = [1, 15, 16, 17, 31, 33, 250, 1000, 2047, 5]
    w = _custom(f"fp8_ragged_g{g}", 2 * g, 2, lens, kv_dtype="fp8_e4m3", outlier_p=0.01, outlier_factor=20.0,
                seed=10 + g)
    for splits in (0, 1, 13):
        res = _run(w, cuda_device, num_splits=splits, out_f32=True)
        assert res["err"] == 0
        ref = H.oracle_layer(w, 0, res["bt"], lens)
        H.assert_out_close(res["out"], ref["out"], what=f"fp8 g={g} splits={splits}")
        np.testing.assert_allclose(res["lse"], ref["lse"], rtol=1e-5, atol=1e-4)


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
def test_maximum_batch(cuda_device, kv_dtype):
    """The largest supported batch (2,048 requests, lengths 1..48 around the block edges): the
    per-request length and prefix arrays fill 16 KB of each CTA's shared memory, and units
    of one to three blocks mostly lie inside one CTA (finished there, no merge)."""
    lens = [int(x) for x in np.random.default_rng(7).integers(1, 49, size=2048)]
    w = _custom(f"maxbatch_{kv_dtype}", 8, 2, lens, kv_dtype=kv_dtype, seed=21)
    res = _run(w, cuda_device, out_f32=True)
    assert res["err"] == 0
    ref = H.oracle_layer(w, 0, res["bt"], lens)
    H.assert_out_close(res["out"], ref["out"], what=f"{kv_dtype} batch 2048")
    np.testing.assert_allclose(res["lse"], ref["lse"], rtol=1e-5, atol=1e-4)


def test_split_and_non_split_agree(cuda_device):
    w = _custom("splits", 32, 8, [4000, 2500, 16, 1234])
    one = _run(w, cuda_device, num_splits=1, out_f32=True)
    for s in (0, 3, 64, 500):
        many = _run(w, cuda_device, num_splits=s, out_f32=True, pool=one["pool"], fill=False)
        assert np.abs(many["out"] - one["out"]).max() <= H.SPLIT_ATOL
        assert np.abs(many["lse"] - one["lse"]).max() <= 1e-4


def test_fp8_decode_parity(cuda_device):
    w = _custom("fp8", 64, 8, [2048, 700], kv_dtype="fp8_e4m3", outlier_p=0.01, outlier_factor=20.0)
    res = _run(w, cuda_device, out_f32=True)
    assert res["err"] == 0
    ref = H.oracle_layer(w, 0, res["bt"], w.seq_lens())
    H.assert_out_close(res["out"], ref["out"])
    np.testing.assert_allclose(res["lse"], ref["lse"], rtol=1e-5, atol=1e-4)


def test_fp8_many_requests_parity(cuda_device):
    """48 FP8 requests at g = 8: the per-request arrays leave no room for three 16-stage CTAs
    an SM, so this call runs the FP8 kernel with the 8-stage ring (small batches run 16)."""
    lens = [int(x) for x in np.random.default_rng(3).integers(40, 700, size=48)]
    w = _custom("fp8many", 64, 8, lens, kv_dtype="fp8_e4m3", outlier_p=0.01, outlier_factor=20.0, seed=4)
    res = _run(w, cuda_device, out_f32=True)
    assert res["err"] == 0
    ref = H.oracle_layer(w, 0, res["bt"], w.seq_lens())
    H.assert_out_close(res["out"], ref["out"])
    np.testing.assert_allclose(res["lse"], ref["lse"], rtol=1e-5, atol=1e-4)


def test_evicted_slots_logits_and_scores(cuda_device):
    """Retain mask, per-position logits and the score epilogue against the oracle."""
    w = _custom("evict", 28, 4, [1500, 900, 2100], evict_frac=0.1, protect_prompt=64, protect_recent=32,
                scores=True)
    res = _run(w, cuda_device, out_f32=True, want_logits=True)
    assert res["err"] == 0
    retain = w.retain_mask(res["bt"])
    ref = H.oracle_layer(w, 0, res["bt"], w.seq_lens(), retain=retain, want_alpha=True, want_logits=True)
    H.assert_out_close(res["out"], ref["out"])
    for b, n in enumerate(w.seq_lens()):
        lg, rl = res["logits"][b, :, :n], ref["logits"][b, :, :n]
        assert np.array_equal(np.isneginf(lg), np.isneginf(rl))
        fin = np.isfinite(rl)
        np.testing.assert_allclose(lg[fin], rl[fin], rtol=1e-5, atol=2e-5)
    # score epilogue for one layer of L = 3 (weight 1/(L·H)) into a running score array
    dev = cuda_device
    S = max(w.seq_lens())
    scores = torch.zeros(w.batch, S + 5, dtype=torch.float32, device=dev)
    kvd.kvd_accum_scores(torch.from_numpy(res["logits"]).to(dev), torch.from_numpy(res["lse"]).to(dev),
                         torch.tensor(w.seq_lens(), dtype=torch.int32, device=dev), 1.0 / (3 * w.n_q), scores)
    got = scores.cpu().numpy().astype(np.float64)
    want = np.zeros_like(got)
    for b, n in enumerate(w.seq_lens()):
        want[b, :n] = ref["alpha"][b, :, :n].sum(0) / (3 * w.n_q)
    assert np.all(np.abs(got - want) <= H.SCORE_RTOL * np.abs(want))
    assert np.all(got[:, S:] == 0)


def test_combine_of_oracle_partials_equals_full_attention(cuda_device):
    """kvd_combine_splits on partials the oracle computes over disjoint pieces of each context."""
    w = _custom("comb", 16, 4, [500, 333])
    bt = w.block_table()
    lens = w.seq_lens()
    g = w.g
    U = w.batch * w.n_kv
    cuts = [[0, 100, 260, 500], [0, 1, 333]]
    q = w.q(0, 0)
    slots_o, slots_l, first, count = [], [], np.zeros(U, np.int32), np.zeros(U, np.int32)
    for b in range(w.batch):
        k, v = w.kv(0, b, 0, lens[b])
        pieces = []
        for a, e in zip(cuts[b][:-1], cuts[b][1:]):
            r = oracle.decode_dense_inputs([k[a:e].float().numpy()], [v[a:e].float().numpy()],
                                           q[b:b + 1].float().numpy(), [e - a], w.n_q)
            pieces.append(r)
        for kvh in range(w.n_kv):
            u = b * w.n_kv + kvh
            first[u] = len(slots_o)
            count[u] = len(pieces)
            for r in pieces:
                slots_o.append(r["out"][0, kvh * g:(kvh + 1) * g])
                slots_l.append(r["lse"][0, kvh * g:(kvh + 1) * g])
    dev = cuda_device
    po = torch.tensor(np.array(slots_o), dtype=torch.float32, device=dev).contiguous()
    pl = torch.tensor(np.array(slots_l), dtype=torch.float32, device=dev).contiguous()
    out = torch.empty(w.batch, w.n_q, 128, dtype=torch.float32, device=dev)
    lse = torch.empty(w.batch, w.n_q, dtype=torch.float32, device=dev)
    kvd.kvd_combine_splits(po, pl, torch.from_numpy(first).to(dev), torch.from_numpy(count).to(dev), w.batch,
                           w.n_q, w.n_kv, out, lse)
    ref = H.oracle_layer(w, 0, bt, lens)
    np.testing.assert_allclose(out.cpu().numpy(), ref["out"], rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(lse.cpu().numpy(), ref["lse"], rtol=1e-6, atol=1e-5)


def test_out_of_range_block_id_is_reported_not_faulted(cuda_device):
    w = _custom("oob", 8, 2, [64, 40])
    bt = w.block_table()
    pool = H.make_pool(w)
    H.fill_layer(pool, w, 0, bt, w.seq_lens(), cuda_device)
    bad = bt.clone()
    bad[1, 1] = 10 ** 6                 # beyond the pool: the kernel must skip it and flag
    S, ws = H.workspace(pool, w.n_q, w.batch, 64)
    out = torch.empty(2, 8, 128, dtype=torch.float32, device=cuda_device)
    kvd.kvd_decode_attn(pool.handle, 0, w.q(0, 0, cuda_device), bad.to(cuda_device),
                        torch.tensor(w.seq_lens(), dtype=torch.int32, device=cuda_device), 64, ws, out)
    assert kvd.kvd_get_device_error(pool.handle) == kvd.KVD_ERR_OOB
    assert kvd.kvd_get_device_error(pool.handle) == 0          # reading clears the word
    ref = H.oracle_layer(w, 0, bt, w.seq_lens())
    H.assert_out_close(out[0].cpu().numpy(), ref["out"][0])     # request 0 unaffected
    # a slot beyond the pool in the append
    kvd.kvd_append_kv(pool.handle, 0, torch.zeros(1, 2, 128, dtype=torch.bfloat16, device=cuda_device),
                      torch.zeros(1, 2, 128, dtype=torch.bfloat16, device=cuda_device),
                      torch.tensor([10 ** 7], dtype=torch.int64, device=cuda_device))
    assert kvd.kvd_get_device_error(pool.handle) == kvd.KVD_ERR_OOB


def test_bad_sequence_length_is_reported(cuda_device):
    w = _custom("badlen", 8, 2, [64, 40])
    pool = H.make_pool(w)
    S, ws = H.workspace(pool, w.n_q, w.batch, 64)
    out = torch.empty(2, 8, 128, dtype=torch.float32, device=cuda_device)
    lse = torch.empty(2, 8, dtype=torch.float32, device=cuda_device)
    bt = w.block_table().to(cuda_device)
    for bad in (0, 10 ** 6, -5):
        seq = torch.tensor([bad, 40], dtype=torch.int32, device=cuda_device)
        kvd.kvd_decode_attn(pool.handle, 0, w.q(0, 0, cuda_device), bt, seq, 64, ws, out, lse_out=lse)
        assert kvd.kvd_get_device_error(pool.handle) == kvd.KVD_ERR_OOB
        assert torch.all(out[0] == 0) and torch.all(torch.isneginf(lse[0]))


def test_bounded_wait_times_out_and_context_survives(cuda_device):
    w = _custom("wait", 8, 2, [64])
    pool = H.make_pool(w)
    kvd.kvd_selftest_wait_timeout(pool.handle, 2_000_000)      # 2 ms
    assert kvd.kvd_get_device_error(pool.handle) == kvd.KVD_ERR_TIMEOUT
    res = _run(w, cuda_device, pool=pool)                      # the context still works
    assert res["err"] == 0


def test_empty_batch_is_a_no_op(cuda_device):
    w = _custom("empty", 8, 2, [64])
    pool = H.make_pool(w)
    ws = torch.empty(256, dtype=torch.uint8, device=cuda_device)
    q = torch.empty(0, 8, 128, dtype=torch.bfloat16, device=cuda_device)
    out = torch.empty(0, 8, 128, dtype=torch.bfloat16, device=cuda_device)
    kvd.kvd_decode_attn(pool.handle, 0, q, torch.zeros(0, 4, dtype=torch.int32, device=cuda_device),
                        torch.zeros(0, dtype=torch.int32, device=cuda_device), 1, ws, out)
    kvd.kvd_append_kv(pool.handle, 0, None, None, None)
    assert kvd.kvd_get_device_error(pool.handle) == 0


def test_cuda_graph_replay_matches_eager(cuda_device):
    w = _custom("graph", 32, 8, [1000, 3000])
    eager = _run(w, cuda_device, out_f32=True)
    pool = eager["pool"]
    bt, bt_d, seq, seq_d, _ = H.device_inputs(w, cuda_device)
    S, ws = H.workspace(pool, w.n_q, w.batch, 3000)
    q = w.q(0, 0, cuda_device)
    out = torch.zeros(w.batch, w.n_q, 128, dtype=torch.float32, device=cuda_device)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        kvd.kvd_decode_attn(pool.handle, 0, q, bt_d, seq_d, 3000, ws, out)   # warm (sets attributes)
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        kvd.kvd_decode_attn(pool.handle, 0, q, bt_d, seq_d, 3000, ws, out)
    out.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), eager["out"])


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
def test_fused_append_equals_separate_append(cuda_device, kv_dtype):
    """k_new/v_new passed to kvd_decode_attn write the same pool bytes and give the same output
    as kvd_append_kv followed by kvd_decode_attn."""
    lens = [300, 17, 1, 4096, 16, 33]
    w = _custom(f"fused_{kv_dtype}", 16, 4, lens, kv_dtype=kv_dtype, seed=5)
    dev = cuda_device
    bt, bt_d, seq, seq_d, _ = H.device_inputs(w, dev)
    prefix = [c - 1 for c in lens]
    pos = w.append_pos(0)
    ks, vs = zip(*[w.kv(0, b, pos[b], pos[b] + 1, dev) for b in range(w.batch)])
    k_new, v_new = torch.cat(ks).contiguous(), torch.cat(vs).contiguous()
    slots = torch.cat([w.slot_mapping(b, pos[b], pos[b] + 1, bt) for b in range(w.batch)]).to(dev)
    q = w.q(0, 0, dev)
    outs = []
    pools = []
    for fused in (False, True):
        pool = H.make_pool(w)
        H.fill_layer(pool, w, 0, bt, prefix, dev)
        if not fused:
            kvd.kvd_append_kv(pool.handle, 0, k_new, v_new, slots)
        S, ws = H.workspace(pool, w.n_q, w.batch, max(lens), 7, dev)
        out = torch.empty(w.batch, w.n_q, 128, dtype=torch.float32, device=dev)
        kvd.kvd_decode_attn(pool.handle, 0, q, bt_d, seq_d, max(lens), ws, out, num_splits=7,
                            k_new=k_new if fused else None, v_new=v_new if fused else None)
        assert kvd.kvd_get_device_error(pool.handle) == 0
        outs.append(out.cpu())
        pools.append(pool)
    assert torch.equal(outs[0], outs[1])
    assert torch.equal(pools[0].mem, pools[1].mem)
    ref = H.oracle_layer(w, 0, bt, lens)
    H.assert_out_close(outs[1].numpy(), ref["out"])


def test_fused_combine_matches_standalone_combine(cuda_device):
    """kvd_decode_attn's own merge launch equals kvd_combine_splits run on the partials of a call
    without output (out = NULL)."""
    w = _custom("fusedcomb", 32, 8, [5000, 77, 2048, 700])
    dev = cuda_device
    bt, bt_d, seq, seq_d, _ = H.device_inputs(w, dev)
    pool = H.make_pool(w)
    H.fill_layer(pool, w, 0, bt, w.seq_lens(), dev)
    q = w.q(0, 0, dev)
    for splits in (5, 0, 300):
        S, ws = H.workspace(pool, w.n_q, w.batch, 5000, splits, dev)
        fused = torch.empty(w.batch, w.n_q, 128, dtype=torch.float32, device=dev)
        flse = torch.empty(w.batch, w.n_q, dtype=torch.float32, device=dev)
        kvd.kvd_decode_attn(pool.handle, 0, q, bt_d, seq_d, 5000, ws, fused, num_splits=splits, lse_out=flse)
        kvd.kvd_decode_attn(pool.handle, 0, q, bt_d, seq_d, 5000, ws, None, num_splits=splits)
        U, g = w.batch * w.n_kv, w.g
        slots = U + S   # workspace layout of an unplanned call (kvd.h): a partial slot per unit and per split
        a256 = lambda x: (x + 255) // 256 * 256
        o_po, o_pl = 0, a256(slots * g * 128 * 4)
        o_uf = o_pl + a256(slots * g * 4)
        o_uc = o_uf + a256(U * 4)
        po = ws[o_po:o_pl].view(torch.float32)
        pl = ws[o_pl:o_pl + slots * g * 4].view(torch.float32)
        uf = ws[o_uf:o_uf + U * 4].view(torch.int32)
        uc = ws[o_uc:o_uc + U * 4].view(torch.int32)
        sep = torch.empty_like(fused)
        slse = torch.empty_like(flse)
        kvd.kvd_combine_splits(po, pl, uf, uc, w.batch, w.n_q, w.n_kv, sep, slse)
        assert kvd.kvd_get_device_error(pool.handle) == 0
        np.testing.assert_allclose(fused.cpu().numpy(), sep.cpu().numpy(), rtol=1e-5, atol=1e-6)
        np.testing.assert_allclose(flse.cpu().numpy(), slse.cpu().numpy(), rtol=1e-6, atol=1e-5)


@pytest.mark.parametrize("shape", ["mixed", "many_partials", "odd_stride"])
def test_fused_score_epilogue_matches_accum_scores(cuda_device, shape):
    """The score update fused into kvd_decode_attn's merge launch equals kvd_accum_scores
    applied to the same call's logits and LSE, and both match the oracle's α sum.  The
    "many_partials" shape (64 heads, 200 splits of one context) needs more partial LSEs per
    request than a score CTA stages in shared memory, so it takes the per-warp path; the
    "odd_stride" shape gives the logits rows an odd stride, so the score CTAs prefetch them
    with 4-byte copies instead of 16-byte ones."""
    extra_cols = 1 if shape == "odd_stride" else 0
    if shape in ("mixed", "odd_stride"):
        w = _custom("fusedscore", 28, 4, [3000, 700, 16, 4100], evict_frac=0.05, protect_prompt=64,
                    protect_recent=32, scores=True)
        split_list = (0, 3, 1)
    else:
        w = _custom("fusedscore_many", 64, 8, [8000], evict_frac=0.05, protect_prompt=64, protect_recent=32,
                    scores=True)
        split_list = (200, 0)
    dev = cuda_device
    bt, bt_d, seq, seq_d, ret_d = H.device_inputs(w, dev)
    pool = H.make_pool(w)
    H.fill_layer(pool, w, 0, bt, w.seq_lens(), dev)
    q = w.q(0, 0, dev)
    S = max(w.seq_lens())
    inv = 1.0 / (3 * w.n_q)
    for splits in split_list:
        _, ws = H.workspace(pool, w.n_q, w.batch, S, splits, dev)
        out = torch.empty(w.batch, w.n_q, 128, dtype=torch.float32, device=dev)
        lse = torch.empty(w.batch, w.n_q, dtype=torch.float32, device=dev)
        logits = torch.full((w.batch, w.n_q, S + extra_cols), float("nan"), dtype=torch.float32, device=dev)
        base = torch.rand(w.batch, S + 3, dtype=torch.float32, device=dev)
        fused = base.clone()
        kvd.kvd_decode_attn(pool.handle, 0, q, bt_d, seq_d, S, ws, out, num_splits=splits, retain_mask=ret_d,
                            lse_out=lse, logits_out=logits, scores=fused, inv_LH=inv)
        sep = base.clone()
        kvd.kvd_accum_scores(logits, lse, seq_d, inv, sep)
        assert kvd.kvd_get_device_error(pool.handle) == 0
        np.testing.assert_allclose(fused.cpu().numpy(), sep.cpu().numpy(), rtol=2e-6, atol=1e-9)
    ref = H.oracle_layer(w, 0, bt, w.seq_lens(), retain=w.retain_mask(bt), want_alpha=True)
    got = (fused - base).double().cpu().numpy()
    for b, n in enumerate(w.seq_lens()):
        want = ref["alpha"][b, :, :n].sum(0) * inv
        assert np.all(np.abs(got[b, :n] - want) <= H.SCORE_RTOL * want + 2 ** -22 * base[b, :n].double().cpu().numpy())


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
def test_early_start_is_bitwise_identical(cuda_device, kv_dtype):
    """KVD_EARLY_START (plan and K/V copies before the grid-dependency wait) changes no bit, also
    for back-to-back calls of two layers captured in one CUDA graph, where the overlap happens."""
    w = _custom(f"early_{kv_dtype}", 32, 8, [3000, 17, 1200, 640], kv_dtype=kv_dtype, L=2, seed=8)
    dev = cuda_device
    bt, bt_d, seq, seq_d, _ = H.device_inputs(w, dev)
    prefix = [c - 1 for c in w.seq_lens()]
    pos = w.append_pos(0)
    S = max(w.seq_lens())
    results = []
    for early in (False, True):
        pool = H.make_pool(w, layers=2)
        kn, vn, qs = [], [], []
        for layer in range(2):
            H.fill_layer(pool, w, layer, bt, prefix, dev)
            ks, vs = zip(*[w.kv(layer, b, pos[b], pos[b] + 1, dev) for b in range(w.batch)])
            kn.append(torch.cat(ks).contiguous())
            vn.append(torch.cat(vs).contiguous())
            qs.append(w.q(layer, 0, dev))
        _, ws = H.workspace(pool, w.n_q, w.batch, S, 0, dev)
        outs = [torch.empty(w.batch, w.n_q, 128, dtype=torch.float32, device=dev) for _ in range(2)]

        def step():
            for layer in range(2):
                kvd.kvd_decode_attn(pool.handle, layer, qs[layer], bt_d, seq_d, S, ws, outs[layer],
                                    k_new=kn[layer], v_new=vn[layer], early_start=early)
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            step()
        torch.cuda.current_stream().wait_stream(s)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        assert kvd.kvd_get_device_error(pool.handle) == 0
        results.append([o.cpu() for o in outs] + [pool.mem.cpu()])
    for a, b in zip(*results):
        assert torch.equal(a, b)

