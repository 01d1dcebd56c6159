"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: values the
pages print (tests/golden), library routines (torch's float8_e4m3fn cast,
scaled_dot_product_attention, scipy's logsumexp), closed forms and invariants.
"""

import os

import numpy as np
import pytest
import torch
from scipy.special import logsumexp

import oracle
from kvd_inputs import gen

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _bf16(x):
    """float32 values rounded to bf16 and widened back (inputs are bf16 tensors)."""
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16).float().numpy()


# ------------------------------------------------------------------ e4m3 codec

def test_e4m3_page_vectors():
    for line in open(os.path.join(GOLDEN, "e4m3_page_vectors.txt")):
        if line.startswith("#") or not line.strip():
            continue
        kind, x, y = line.split()
        x, y = float(x), float(y)
        if kind in ("round", "max"):
            assert oracle.e4m3_decode(oracle.e4m3_encode(np.float32(x))) == y
        elif kind == "spacing":
            c = int(oracle.e4m3_encode(np.float32(x)))
            assert oracle.e4m3_decode(np.uint8(c + 1)) - oracle.e4m3_decode(np.uint8(c)) == y
    # nothing above the largest finite value
    assert oracle.e4m3_decode(np.uint8(0x7E)) == 448.0
    assert np.isnan(oracle.e4m3_decode(np.uint8(0x7F)))


def test_e4m3_decode_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(ours[ok], ref[ok])
    assert np.array_equal(np.signbit(ours[ok]), np.signbit(ref[ok]))


def test_e4m3_decode_format_closed_forms():
    d = oracle.e4m3_decode(np.arange(127, dtype=np.uint8))
    assert np.all(np.diff(d) > 0)                 # monotone over non-negative codes
    assert d[1] == 2.0 ** -9                      # smallest subnormal m·2^-9
    assert d[8] == 2.0 ** -6                      # smallest normal 2^(1-7)
    assert d[0x38] == 1.0                         # exponent field 7 = bias
    assert d[0x7E] == 448.0


def _e4m3_test_values():
    r = _rng(1)
    mag = np.exp2(r.uniform(-12, 10, 200000)).astype(np.float32)
    sgn = np.where(r.random(mag.size) < 0.5, -1, 1).astype(np.float32)
    vals = [mag * sgn]
    # exact midpoints between neighbouring codes (ties) and the codes themselves
    d = oracle.e4m3_decode(np.arange(127, dtype=np.uint8))
    mids = ((d[1:] + d[:-1]) / 2).astype(np.float32)
    vals += [mids, -mids, d.astype(np.float32), np.array([0.0, -0.0, 448, 449, 464, 465, 1e6, -1e6,
                                                           np.inf, -np.inf], np.float32)]
    return np.concatenate(vals)


def test_e4m3_encode_matches_torch_cast():
    y = _e4m3_test_values()
    ours = oracle.e4m3_encode(y)
    ref = torch.from_numpy(np.clip(y, -448, 448)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_e4m3_encode_is_nearest_within_half_spacing():
    y = _e4m3_test_values()
    y = y[np.isfinite(y) & (np.abs(y) <= 448)]
    back = oracle.e4m3_decode(oracle.e4m3_encode(y))
    a = np.abs(y.astype(np.float64))
    # spacing of e4m3 around a: 2^-9 below 2^-6, else 2^(floor(log2 a) - 3)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -6)))
    spacing = np.exp2(e - 3)
    assert np.all(np.abs(back - y) <= spacing / 2)


def test_quantize_rows_properties():
    r = _rng(2)
    x = _bf16(r.standard_normal((400, 128)).astype(np.float32) * np.exp2(r.uniform(-8, 8, (400, 1))))
    x[3] = 0.0
    codes, scales = oracle.quantize_rows(x)
    assert scales[3] == 1.0 and not codes[3].any()
    amax = np.abs(x).max(axis=1)
    nz = amax > 0
    # scale is the fp32 value nearest absmax/448, so absmax/scale lands on the largest code
    assert np.allclose(scales[nz], amax[nz] / 448.0, rtol=2 ** -23, atol=0)
    rows_max = np.abs(oracle.e4m3_decode(codes)).max(axis=1)
    assert np.all(rows_max[nz] == 448.0)
    # read-back error within half an e4m3 spacing of x/scale, times the scale
    back = oracle.e4m3_decode(codes) * scales[:, None].astype(np.float64)
    y = np.abs(x / scales[:, None])
    e = np.floor(np.log2(np.maximum(y, 2.0 ** -6)))
    bound = np.exp2(e - 3) / 2 * scales[:, None] * (1 + 2 ** -20)
    assert np.all(np.abs(back - x) <= bound + 1e-300)
    # the code step itself is torch's float8 cast of the fp32 quotient
    qt = (torch.from_numpy(x) / torch.from_numpy(scales)[:, None]).clamp(-448, 448)
    assert np.array_equal(codes, qt.to(torch.float8_e4m3fn).view(torch.uint8).numpy())


# ------------------------------------------------------------ paged attention

def _dense_sdpa(q, k, v, scale, keep=None):
    """torch fp64 scaled_dot_product_attention over one request's logical K/V.

    q [n_q][d], k/v [ctx][n_kv][d]; query heads map to KV heads in consecutive groups."""
    n_q, n_kv = q.shape[0], k.shape[1]
    g = n_q // n_kv
    qt = torch.from_numpy(np.asarray(q, np.float64))[None, :, None, :]          # [1, n_q, 1, d]
    kt = torch.from_numpy(np.asarray(k, np.float64)).permute(1, 0, 2).repeat_interleave(g, 0)[None]
    vt = torch.from_numpy(np.asarray(v, np.float64)).permute(1, 0, 2).repeat_interleave(g, 0)[None]
    mask = None
    if keep is not None:
        mask = torch.from_numpy(np.asarray(keep, bool))[None, None, None, :].expand(1, n_q, 1, -1)
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=scale)
    return o[0, :, 0, :].numpy()


def _page_example():
    tables = {}
    for line in open(os.path.join(GOLDEN, "block_table_example.txt")):
        if line.startswith("#") or not line.strip():
            continue
        name, rest = line.split(":")
        pairs = [tuple(map(int, p.split("->"))) for p in rest.split()]
        assert [j for j, _ in pairs] == list(range(len(pairs)))
        tables[name] = [p for _, p in pairs]
    return tables


def _make_requests(seed, lens, n_kv, d_h, n_q):
    r = _rng(seed)
    ks = [_bf16(r.standard_normal((c, n_kv, d_h))) for c in lens]
    vs = [_bf16(r.standard_normal((c, n_kv, d_h))) for c in lens]
    q = _bf16(r.standard_normal((len(lens), n_q, d_h)))
    return q, ks, vs


def _paged(tables, lens, ks, vs, num_blocks, n_kv, d_h, fp8=False):
    pool = oracle.OraclePool(num_blocks, n_kv, d_h, 16, fp8)
    bt = np.full((len(tables), max(len(t) for t in tables)), -1, np.int32)
    for b, t in enumerate(tables):
        bt[b, :len(t)] = t
        pos = np.arange(lens[b])
        slots = np.asarray(t, np.int64)[pos // 16] * 16 + pos % 16
        assert pool.append(ks[b], vs[b], slots) == 0
    return pool, bt


def test_page_block_table_example_matches_dense_attention():
    tabs = _page_example()
    tables = [tabs["A"], tabs["B"], tabs["C"]]
    lens = [20, 90, 33]                       # last blocks partly filled
    n_q, n_kv, d_h = 8, 2, 32
    q, ks, vs = _make_requests(3, lens, n_kv, d_h, n_q)
    pool, bt = _paged(tables, lens, ks, vs, 11, n_kv, d_h)
    scale = 1 / np.sqrt(d_h)
    res = oracle.decode(pool, q, n_q, bt, lens, softmax_scale=scale, want_alpha=True)
    assert res["status"] == 0
    for b in range(3):
        ref = _dense_sdpa(q[b], ks[b], vs[b], scale)
        np.testing.assert_allclose(res["out"][b], ref, rtol=1e-12, atol=1e-13)
        assert np.allclose(res["alpha"][b, :, :lens[b]].sum(-1), 1.0, atol=1e-13)


def test_lse_matches_logsumexp_and_alpha_is_softmax():
    lens = [37, 64, 1]
    n_q, n_kv, d_h = 4, 4, 16
    q, ks, vs = _make_requests(4, lens, n_kv, d_h, n_q)
    tables = [[0, 1, 2], [3, 4, 5, 6], [7]]
    pool, bt = _paged(tables, lens, ks, vs, 8, n_kv, d_h)
    res = oracle.decode(pool, q, n_q, bt, lens, want_alpha=True, want_logits=True)
    for b, c in enumerate(lens):
        lg = np.einsum("hd,thd->ht", q[b].astype(np.float64), ks[b].astype(np.float64)) / np.sqrt(d_h)
        np.testing.assert_allclose(res["logits"][b, :, :c], lg, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(res["lse"][b], logsumexp(lg, axis=-1), rtol=1e-13)
        np.testing.assert_allclose(res["alpha"][b, :, :c],
                                   torch.softmax(torch.from_numpy(lg), -1).numpy(), rtol=1e-12, atol=1e-15)


def test_permuting_physical_blocks_is_bitwise_invariant():
    lens = [100, 250]
    n_q, n_kv, d_h = 8, 2, 64
    q, ks, vs = _make_requests(5, lens, n_kv, d_h, n_q)
    nblk = [7, 16]
    nb = 40
    base = [list(range(0, 7)), list(range(7, 23))]
    pool, bt = _paged(base, lens, ks, vs, nb, n_kv, d_h)
    ref = oracle.decode(pool, q, n_q, bt, lens)
    for seed in range(3):
        perm = gen.permutation(gen.stream_key(seed, "relabel"), nb).numpy()
        tables = [[int(perm[p]) for p in t] for t in base]
        pool2, bt2 = _paged(tables, lens, ks, vs, nb, n_kv, d_h)
        res = oracle.decode(pool2, q, n_q, bt2, lens)
        assert np.array_equal(res["out"], ref["out"]) and np.array_equal(res["lse"], ref["lse"])
    assert sum(nblk) == 23


def test_shared_blocks_serve_two_requests():
    # request 1 reuses request 0's first three physical blocks (a shared prefix)
    n_q, n_kv, d_h = 4, 1, 32
    r = _rng(6)
    prefix_k = _bf16(r.standard_normal((48, n_kv, d_h)))
    prefix_v = _bf16(r.standard_normal((48, n_kv, d_h)))
    tail = [_bf16(r.standard_normal((10, n_kv, d_h))) for _ in range(4)]
    ks = [np.concatenate([prefix_k, tail[0]]), np.concatenate([prefix_k, tail[1]])]
    vs = [np.concatenate([prefix_v, tail[2]]), np.concatenate([prefix_v, tail[3]])]
    q = _bf16(r.standard_normal((2, n_q, d_h)))
    pool = oracle.OraclePool(6, n_kv, d_h)
    pos = np.arange(58)
    pool.append(ks[0], vs[0], np.array([2, 0, 4, 5])[pos // 16] * 16 + pos % 16)
    pool.append(tail[1], tail[3], 1 * 16 + np.arange(10))
    bt = np.array([[2, 0, 4, 5], [2, 0, 4, 1]], np.int32)
    res = oracle.decode(pool, q, n_q, bt, [58, 58])
    for b in range(2):
        np.testing.assert_allclose(res["out"][b], _dense_sdpa(q[b], ks[b], vs[b], 1 / np.sqrt(d_h)),
                                   rtol=1e-12, atol=1e-13)


def test_identical_keys_give_mean_of_values():
    n_q, n_kv, d_h, c = 4, 2, 16, 45
    r = _rng(7)
    k1 = _bf16(r.standard_normal((1, n_kv, d_h)))
    ks = [np.repeat(k1, c, axis=0)]
    vs = [_bf16(r.standard_normal((c, n_kv, d_h)))]
    q = _bf16(r.standard_normal((1, n_q, d_h)))
    pool, bt = _paged([[3, 1, 0]], [c], ks, vs, 4, n_kv, d_h)
    res = oracle.decode(pool, q, n_q, bt, [c])
    for h in range(n_q):
        np.testing.assert_allclose(res["out"][0, h], vs[0][:, h // 2].astype(np.float64).mean(0), rtol=1e-12,
                                   atol=1e-14)


def test_one_dominant_logit_selects_its_value():
    n_q, n_kv, d_h, c = 2, 1, 16, 40
    r = _rng(8)
    ks = [np.zeros((c, n_kv, d_h), np.float32)]
    ks[0][17, 0, :] = 64.0                    # q·k = 64·64·d/√d  ≫ every other logit (0)
    vs = [_bf16(r.standard_normal((c, n_kv, d_h)))]
    q = np.full((1, n_q, d_h), 64.0, np.float32)
    pool, bt = _paged([[0, 1, 2]], [c], ks, vs, 3, n_kv, d_h)
    res = oracle.decode(pool, q, n_q, bt, [c])
    for h in range(n_q):
        assert np.array_equal(res["out"][0, h], vs[0][17, 0].astype(np.float64))


def test_masked_attention_equals_compacted_table():
    """Only evicted slots change the result: masking them equals dropping them (offloading Prop. 1)."""
    n_q, n_kv, d_h, c = 4, 2, 32, 150
    q, ks, vs = _make_requests(9, [c], n_kv, d_h, n_q)
    evict = np.array([5, 17, 18, 40, 41, 42, 99, 130])
    keep = np.setdiff1d(np.arange(c), evict)
    tables = [list(range(10))]
    pool, bt = _paged(tables, [c], ks, vs, 10, n_kv, d_h)
    retain = np.full(10, 0xFFFF, np.int64)
    for p in evict:
        retain[p // 16] &= ~(1 << (p % 16))
    res = oracle.decode(pool, q, n_q, bt, [c], retain=retain, want_alpha=True)
    assert np.all(res["alpha"][0][:, evict] == 0)
    ck = [ks[0][keep]]
    cv = [vs[0][keep]]
    pool2, bt2 = _paged([list(range(9))], [keep.size], ck, cv, 9, n_kv, d_h)
    res2 = oracle.decode(pool2, q, n_q, bt2, [keep.size])
    assert np.array_equal(res["out"], res2["out"])
    assert np.array_equal(res["lse"], res2["lse"])
    np.testing.assert_allclose(res["out"][0], _dense_sdpa(q[0], ks[0], vs[0], 1 / np.sqrt(d_h),
                                                          keep=np.isin(np.arange(c), keep)), rtol=1e-12, atol=1e-13)


def test_fp8_pool_reads_back_dequantised_values():
    lens = [70, 33]
    n_q, n_kv, d_h = 8, 2, 64
    q, ks, vs = _make_requests(10, lens, n_kv, d_h, n_q)
    ks[0][:, 1, 5] *= 20.0                     # an outlier channel
    tables = [[4, 0, 2, 6, 1], [3, 5, 7]]
    pool, bt = _paged(tables, lens, ks, vs, 8, n_kv, d_h, fp8=True)
    res = oracle.decode(pool, q, n_q, bt, lens)
    for b, c in enumerate(lens):
        # dequantise through torch's float8 type: value(code) × per-(token, head) scale
        kc, kscale = oracle.quantize_rows(ks[b])
        vc, vscale = oracle.quantize_rows(vs[b])
        kd = torch.from_numpy(kc).view(torch.float8_e4m3fn).double().numpy() * kscale[..., None]
        vd = torch.from_numpy(vc).view(torch.float8_e4m3fn).double().numpy() * vscale[..., None]
        np.testing.assert_allclose(res["out"][b], _dense_sdpa(q[b], kd, vd, 1 / np.sqrt(d_h)), rtol=1e-12,
                                   atol=1e-13)
        # and stays within FP8 rounding of the unquantised attention
        np.testing.assert_allclose(res["out"][b], _dense_sdpa(q[b], ks[b], vs[b], 1 / np.sqrt(d_h)), atol=0.1)


def test_bad_block_id_and_empty_attention_are_reported():
    n_q, n_kv, d_h = 2, 1, 16
    q, ks, vs = _make_requests(11, [20], n_kv, d_h, n_q)
    pool, bt = _paged([[0, 1]], [20], ks, vs, 2, n_kv, d_h)
    bad = bt.copy()
    bad[0, 1] = 7
    assert oracle.decode(pool, q, n_q, bad, [20])["status"] == oracle.oracle.ERR_INDEX
    res = oracle.decode(pool, q, n_q, bt, [20], retain=np.array([0, 0]))
    assert res["status"] == oracle.oracle.ERR_EMPTY
    assert np.all(res["out"] == 0) and np.all(np.isneginf(res["lse"]))


# ------------------------------------------------------------- score update

def test_score_update_closed_forms():
    L, B, H, S = 3, 2, 4, 12
    seq = np.array([12, 9], np.int32)
    # one-hot alphas: layer l, head h puts all weight on position l·H + h
    a = np.zeros((L, B, H, S))
    for ly in range(L):
        for h in range(H):
            for b in range(B):
                a[ly, b, h, (ly * H + h) % seq[b]] = 1.0
    s = oracle.score_update(np.zeros((B, S)), a, seq)
    np.testing.assert_allclose(s[0], np.full(12, 1.0 / (L * H)), rtol=1e-15)
    assert np.isclose(s[1].sum(), 1.0, rtol=1e-15)
    assert np.all(s[1, 9:] == 0)               # positions beyond the context are untouched


def test_score_sum_grows_by_one_per_step_and_single_head_is_softmax():
    n_q, n_kv, d_h = 4, 2, 32
    lens = [50, 77]
    s = np.zeros((2, 80))
    L = 2
    for step in range(3):
        alphas = []
        for ly in range(L):
            q, ks, vs = _make_requests(100 + 10 * step + ly, lens, n_kv, d_h, n_q)
            res = oracle.decode_dense_inputs(ks, vs, q, lens, n_q)
            a = np.zeros((2, n_q, 80))
            a[:, :, :res["alpha"].shape[2]] = res["alpha"]
            alphas.append(a)
        s = oracle.score_update(s, np.stack(alphas), lens)
        np.testing.assert_allclose(s.sum(axis=1), step + 1, rtol=1e-13)
    # L = 1, H = 1: the update is the softmax itself
    q, ks, vs = _make_requests(200, [30], 1, 16, 1)
    res = oracle.decode_dense_inputs(ks, vs, q, [30], 1)
    s1 = oracle.score_update(np.zeros((1, 30)), res["alpha"][None], [30])
    lg = (q[0, 0].astype(np.float64) @ ks[0][:, 0].astype(np.float64).T) / 4.0
    np.testing.assert_allclose(s1[0], torch.softmax(torch.from_numpy(lg), 0).numpy(), rtol=1e-12)


# ------------------------------------------------------------------ tier plan
def _tier_of(imp_per_block, length, max_blocks, pp, pr, t1):
    """Scores that put imp_per_block[j] on the first position of block j (the rest 0)."""
    s = np.zeros((1, max_blocks * 16), np.float32)
    for j, x in enumerate(imp_per_block):
        s[0, 16 * j] = x
    return oracle.tier_plan(s, [length], max_blocks, pp, pr, t1)


def test_tier_plan_worked_example():
    # length 100: blocks 0..6, the last holding positions 96..99.  protect_prompt 20 covers
    # blocks 0 and 1 (block 1 holds 16..19); protect_recent 5 covers positions 95..99, i.e.
    # block 5 (80..95) and block 6.  Unprotected: 2, 3, 4 with importances 3, 1, 2.
    imp, tier = _tier_of([9, 9, 3, 1, 2, 9, 9], 100, 8, 20, 5, 2)
    assert tier[0].tolist() == [0, 0, 0, 1, 1, 0, 0, -1]
    assert imp[0].tolist() == [9, 9, 3, 1, 2, 9, 9, 0]
    # protect_recent 4 leaves block 5 free (its last position 95 < 96); importance 0.5 ranks first
    _, tier = _tier_of([9, 9, 3, 1, 2, 0.5, 9], 100, 8, 20, 4, 2)
    assert tier[0].tolist() == [0, 0, 0, 1, 0, 1, 0, -1]
    # no recent window: the partial last block is free too (it holds no position ≥ 100)
    _, tier = _tier_of([9, 9, 3, 1, 2, 9, 0.25], 100, 8, 20, 0, 1)
    assert tier[0].tolist() == [0, 0, 0, 0, 0, 0, 1, -1]
    # t1 above the free count: every free block goes to the host tier
    _, tier = _tier_of([9, 9, 3, 1, 2, 9, 9], 100, 8, 20, 5, 10)
    assert tier[0].tolist() == [0, 0, 1, 1, 1, 0, 0, -1]
    # t1 = 0 keeps everything in HBM; ties go to the lower block index
    _, tier = _tier_of([9, 9, 3, 1, 2, 9, 9], 100, 8, 20, 5, 0)
    assert tier[0].tolist() == [0, 0, 0, 0, 0, 0, 0, -1]
    _, tier = _tier_of([1, 1, 1, 1, 1, 1, 1], 112, 8, 0, 0, 3)
    assert tier[0].tolist() == [1, 1, 1, 0, 0, 0, 0, -1]


def test_tier_plan_importance_closed_forms():
    # unit scores: block j's importance is its number of positions (16, or the tail)
    s = np.ones((3, 64), np.float32)
    imp, tier = oracle.tier_plan(s, [37, 64, 0], 5, 0, 0, 0)
    assert imp[0].tolist() == [16, 16, 5, 0, 0]
    assert imp[1].tolist() == [16, 16, 16, 16, 0]
    assert tier[2].tolist() == [-1] * 5 and imp[2].tolist() == [0] * 5   # empty request
    # positions at or past the score stride count 0
    imp, _ = oracle.tier_plan(np.ones((1, 40), np.float32), [64], 4, 0, 0, 0)
    assert imp[0].tolist() == [16, 16, 8, 0]
    # a length beyond max_blocks·16 is treated as empty
    _, tier = oracle.tier_plan(np.ones((1, 64), np.float32), [49], 3, 0, 0, 1)
    assert tier[0].tolist() == [-1, -1, -1]


def test_tier_plan_matches_sorting_and_fp64_sums():
    rng = _rng(7)
    lens = [1, 16, 17, 300, 1023, 2048]
    mb = 128
    s = rng.exponential(1e-3, size=(len(lens), mb * 16)).astype(np.float32)
    s[:, ::5] = np.round(s[:, ::5], 4)              # some equal values, so ties occur
    s[3, 16:48] = 0.0                               # two all-zero blocks: a tie on importance 0
    for pp, pr, t1 in [(0, 0, 3), (64, 32, 10), (5, 1, 1000), (2048, 0, 4)]:
        imp, tier = oracle.tier_plan(s, lens, mb, pp, pr, t1)
        for b, ln in enumerate(lens):
            nb = (ln + 15) // 16
            assert np.all(tier[b, nb:] == -1) and np.all(imp[b, nb:] == 0)
            exact = np.array([np.sum(s[b, 16 * j:min(16 * j + 16, ln)].astype(np.float64)) for j in range(nb)])
            mag = np.array([np.sum(np.abs(s[b, 16 * j:min(16 * j + 16, ln)].astype(np.float64))) for j in range(nb)])
            assert np.all(np.abs(imp[b, :nb] - exact) <= 16 * 2.0 ** -24 * mag + 1e-30)
            prot = np.array([any(p < pp or p >= ln - pr for p in range(16 * j, min(16 * j + 16, ln)))
                             for j in range(nb)], bool)
            free = np.nonzero(~prot)[0]
            order = free[np.lexsort((free, imp[b, free]))]   # by importance, then block index
            want = np.zeros(nb, np.int8)
            want[order[:t1]] = 1
            assert tier[b, :nb].tolist() == want.tolist()
            assert int((tier[b] == 1).sum()) == min(t1, len(free))


# ------------------------------------------------------------------ e5m2 codec
def test_e5m2_page_facts():
    for line in open(os.path.join(GOLDEN, "e5m2_page_vectors.txt")):
        if line.startswith("#") or not line.strip():
            continue
        kind, *vals = line.split()
        if kind == "bits":
            s_bits, e_bits, m_bits = map(int, vals)
            assert (s_bits, e_bits, m_bits) == (1, 5, 2)
            # largest finite: all-ones exponent is reserved (inf/NaN), bias 2^(e-1)-1
            top = (2 - 2.0 ** -m_bits) * 2.0 ** ((2 ** e_bits - 2) - (2 ** (e_bits - 1) - 1))
            assert oracle.e5m2_decode(np.uint8(0x7B)) == top
        elif kind == "max":
            assert oracle.e5m2_decode(np.uint8(0x7B)) == float(vals[0])
            assert int(oracle.e5m2_encode(np.float32(vals[0]))) == 0x7B
            assert int(oracle.e5m2_encode(np.float32(1e9))) == 0x7B     # saturates


def test_e5m2_decode_all_codes_match_torch_and_f16_high_byte():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e5m2_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e5m2).to(torch.float64).numpy()
    # closed form: an E5M2 code is the high byte of an IEEE half with the low byte zero
    half = (codes.astype(np.uint16) << 8).view(np.float16).astype(np.float64)
    for other in (ref, half):
        assert np.array_equal(np.isnan(ours), np.isnan(other))
        ok = ~np.isnan(other)
        assert np.array_equal(ours[ok], other[ok])
        assert np.array_equal(np.signbit(ours[ok]), np.signbit(other[ok]))


def _e5m2_test_values():
    r = _rng(11)
    mag = np.exp2(r.uniform(-18, 16, 200000)).astype(np.float32)
    sgn = np.where(r.random(mag.size) < 0.5, -1, 1).astype(np.float32)
    d = oracle.e5m2_decode(np.arange(124, dtype=np.uint8))
    mids = ((d[1:] + d[:-1]) / 2).astype(np.float32)
    return np.concatenate([mag * sgn, mids, -mids, d.astype(np.float32),
                           np.array([0.0, -0.0, 57344, 57345, 61439, 61441, 1e9, -1e9], np.float32)])


def test_e5m2_encode_matches_torch_cast_and_half_spacing():
    y = _e5m2_test_values()
    ours = oracle.e5m2_encode(y)
    ref = torch.from_numpy(np.clip(y, -57344, 57344)).to(torch.float8_e5m2).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)
    fin = np.abs(y) <= 57344
    back = oracle.e5m2_decode(ours[fin])
    a = np.abs(y[fin].astype(np.float64))
    spacing = np.exp2(np.floor(np.log2(np.maximum(a, 2.0 ** -14))) - 2)   # 2^-16 below 2^-14
    assert np.all(np.abs(back - y[fin]) <= spacing / 2)


def test_quantize_rows_in_both_formats():
    r = _rng(12)
    x = _bf16(r.standard_normal((300, 128)).astype(np.float32) * np.exp2(r.uniform(-8, 8, (300, 1))))
    x[5] = 0.0
    c4, s4 = oracle.quantize_rows_fmt(x, oracle.FMT_E4M3)
    c_ref, s_ref = oracle.quantize_rows(x)
    assert np.array_equal(c4, c_ref) and np.array_equal(s4.view(np.uint32), s_ref.view(np.uint32))
    c5, s5 = oracle.quantize_rows_fmt(x, oracle.FMT_E5M2)
    amax = np.abs(x).max(axis=1)
    want = np.where(amax == 0, np.float32(1), (amax / np.float32(57344)).astype(np.float32))
    assert np.array_equal(s5.view(np.uint32), want.view(np.uint32))
    # the row's absmax element maps to the largest code, and codes are torch's cast of x/scale
    i = np.abs(x).argmax(axis=1)
    nz = amax > 0
    assert np.all((c5[np.arange(300), i] & 0x7F)[nz] == 0x7B)
    q = torch.from_numpy((x / s5[:, None]).astype(np.float32)).to(torch.float8_e5m2).view(torch.uint8).numpy()
    assert np.array_equal(c5, q)
    assert np.all(c5[5] == 0) and s5[5] == 1.0


def _mixed_pools(seed, fmt):
    """Three single-format pools and one mixed pool fed the same tokens."""
    r = _rng(seed)
    nb, n_kv, d_h, bs = len(fmt), 2, 32, 16
    n = nb * bs - 5
    k = _bf16(r.standard_normal((n, n_kv, d_h)).astype(np.float32))
    v = _bf16(r.standard_normal((n, n_kv, d_h)).astype(np.float32))
    slots = r.permutation(nb * bs)[:n].astype(np.int64)
    pools = {}
    for f in (oracle.FMT_BF16, oracle.FMT_E4M3, oracle.FMT_E5M2):
        p = oracle.OraclePool(nb, n_kv, d_h, bs, block_fmt=np.full(nb, f, np.uint8))
        assert p.append(k, v, slots) == 0
        pools[f] = p
    mixed = oracle.OraclePool(nb, n_kv, d_h, bs, block_fmt=np.array(fmt, np.uint8))
    assert mixed.append(k, v, slots) == 0
    return pools, mixed, k, v, slots


def test_mixed_pool_blocks_match_their_single_format_pools():
    fmt = [0, 1, 2, 2, 1, 0, 1, 2]
    pools, mixed, k, v, slots = _mixed_pools(13, fmt)
    km, vm = mixed.values()
    for p, f in enumerate(fmt):
        kf, vf = pools[f].values()
        assert np.array_equal(km[p], kf[p]) and np.array_equal(vm[p], vf[p])
        if f:
            assert np.array_equal(mixed.k_codes[p], pools[f].k_codes[p])
    # an all-BF16 mixed pool is the plain BF16 pool; an all-E4M3 one the FP8 pool, bit for bit
    plain = oracle.OraclePool(len(fmt), 2, 32, 16)
    fp8 = oracle.OraclePool(len(fmt), 2, 32, 16, fp8=True)
    assert plain.append(k, v, slots) == 0 and fp8.append(k, v, slots) == 0
    assert np.array_equal(pools[0].values()[0], plain.values()[0])
    assert np.array_equal(pools[1].values()[1], fp8.values()[1])
    assert np.array_equal(pools[1].v_codes, fp8.v_codes)


def test_mixed_pool_attention_matches_torch_casts_and_sdpa():
    fmt = [2, 0, 1, 2, 0, 1, 1, 2]
    nb, n_kv, d_h, bs, n_q = len(fmt), 2, 32, 16, 4
    pools, mixed, k, v, slots = _mixed_pools(14, fmt)
    # expected values from torch's float8 casts of x/scale, block by block
    def via_torch(x, f):
        if f == oracle.FMT_BF16:
            return x.astype(np.float64)
        top, dt = (448.0, torch.float8_e4m3fn) if f == oracle.FMT_E4M3 else (57344.0, torch.float8_e5m2)
        amax = np.abs(x).max(axis=-1, keepdims=True)
        sc = np.where(amax == 0, np.float32(1), (amax / np.float32(top)).astype(np.float32))
        c = torch.from_numpy((x / sc).astype(np.float32)).to(dt).to(torch.float64).numpy()
        return c * sc.astype(np.float64)
    km, vm = mixed.values()
    for t, s in enumerate(slots):
        p, o = divmod(int(s), bs)
        for h in range(n_kv):
            assert np.array_equal(km[p, h, o], via_torch(k[t, h], fmt[p]))
            assert np.array_equal(vm[p, h, o], via_torch(v[t, h], fmt[p]))
    # attention over the mixed pool: one request whose table walks every block
    r = _rng(15)
    q = _bf16(r.standard_normal((1, n_q, d_h)).astype(np.float32))
    table = np.array([r.permutation(nb)], np.int32)
    ln = nb * bs
    res = oracle.decode(mixed, q, n_q, table, np.array([ln], np.int32))
    kl = np.stack([km[table[0, t // bs], :, t % bs] for t in range(ln)])   # [ln][n_kv][d_h]
    vl = np.stack([vm[table[0, t // bs], :, t % bs] for t in range(ln)])
    # the 5 slots never written hold zeros in every format and are attended like any other
    ref = _dense_sdpa(q[0].astype(np.float64), kl, vl, 1 / np.sqrt(d_h))
    np.testing.assert_allclose(res["out"][0], ref, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------------ low-bit KV (INT4 / 2-bit)
def test_round_half_matches_numpy_float16_with_saturation():
    """Half-precision rounding against numpy's IEEE float16 cast: random values over every
    exponent, exact ties, subnormals and the overflow edge (saturated at 65,504 here)."""
    r = _rng(40)
    x = np.concatenate([
        r.standard_normal(20000) * np.exp2(r.integers(-30, 20, 20000)),
        (np.arange(1, 4000) + 0.5) * 2.0 ** -24,              # ties between subnormals
        (1 + (2 * np.arange(1, 1024) + 1) / 2048.0) * 4.0,    # ties between normals
        [0.0, -0.0, 65504.0, 65519.9, 65520.0, 1e6, -1e6, 2.0 ** -25, 3 * 2.0 ** -26],
    ])
    got = oracle.round_half_sat(x)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).astype(np.float64)
    ref = np.where(np.isinf(ref), np.sign(ref) * 65504.0, ref)
    assert np.array_equal(got, ref)


def _lowbit_case(seed, rows=400, d=128):
    r = _rng(seed)
    x = r.standard_normal((rows, d)).astype(np.float32)
    x[5] = 0.0                                     # a zero row
    x[6, :32] = 1.25                               # a constant group
    x[7] *= 1000.0                                 # a wide row
    x[8, 40] = 300.0                               # one outlier in group 1
    x[9] = np.linspace(-3, 3, d, dtype=np.float32)
    return _bf16(x)


@pytest.mark.parametrize("bits", [4, 2])
@pytest.mark.parametrize("G", [32, 64, 128])
def test_lowbit_quantise_closed_forms(bits, G):
    """Per group of G values: the scale is the group's span / (2^bits - 1) to half precision, the zero
    point its minimum to half precision, codes span [0, 2^bits - 1] and reconstruct every value
    to within half a scale (plus the half-precision rounding of the scale and zero)."""
    top = (1 << bits) - 1
    x = _lowbit_case(41)
    codes, scales, zeros = oracle.quantize_rows_lowbit(x, bits, G)
    xg = x.reshape(x.shape[0], -1, G).astype(np.float64)
    mn, mx = xg.min(-1), xg.max(-1)
    span = (mx - mn) / top
    assert codes.max() <= top and codes.dtype == np.uint8
    # scale: the half-precision value nearest span (relative half-ulp 2^-11), 1 for a zero span
    nz = span > 0
    assert np.all(np.abs(scales[nz] - span[nz]) <= 2.0 ** -11 * span[nz] * (1 + 1e-6))
    assert np.all(scales[~nz] == 1.0)
    assert np.all(np.abs(zeros - mn) <= 2.0 ** -11 * np.abs(mn) + 2.0 ** -25)
    # every scale and zero is a half-precision number
    assert np.array_equal(scales.astype(np.float16).astype(np.float32), scales)
    assert np.array_equal(zeros.astype(np.float16).astype(np.float32), zeros)
    # reconstruction bound
    rec = codes.reshape(xg.shape) * scales[..., None].astype(np.float64) + zeros[..., None].astype(np.float64)
    slack = 2.0 ** -11 * (np.abs(mn) + top * span) + 1e-6 * np.abs(xg).max(-1)
    err = np.abs(rec - xg)
    assert np.all(err <= 0.5 * scales[..., None] + slack[..., None]), err.max()
    # the minimum of a group lands on code 0 and its maximum on the top code (up to rounding)
    cg = codes.reshape(xg.shape)
    assert np.all(cg[np.arange(xg.shape[0])[:, None], np.arange(xg.shape[1]), xg.argmin(-1)][nz] == 0)
    assert np.all(cg[np.arange(xg.shape[0])[:, None], np.arange(xg.shape[1]), xg.argmax(-1)][nz] >= top - 1)
    # constant group (the first 32 values of row 6): scale 1, code 0, value = the half-precision zero point
    if G == 32:
        assert scales[6, 0] == 1.0 and np.all(codes[6, :32] == 0) and zeros[6, 0] == np.float32(1.25)


@pytest.mark.parametrize("bits", [4, 2])
@pytest.mark.parametrize("G", [32, 128])
def test_lowbit_codes_are_the_nearest_level(bits, G):
    """Brute force: given the group's scale and zero, the stored code is the level c·scale + zero
    nearest to x among all 2^bits levels (x below the lowest level takes code 0, above the highest
    the top code); an exact tie may go either way only if the single-precision quotient rounded."""
    top = (1 << bits) - 1
    x = _lowbit_case(42, rows=200)
    codes, scales, zeros = oracle.quantize_rows_lowbit(x, bits, G)
    lv = np.arange(top + 1, dtype=np.float64)
    xs = x.reshape(x.shape[0], -1, G).astype(np.float64)
    levels = lv[None, None, None, :] * scales[..., None, None] + zeros[..., None, None]   # [r][g][1][L]
    dist = np.abs(xs[..., None] - levels)
    best = dist.min(-1)
    chosen = np.take_along_axis(dist, codes.reshape(xs.shape)[..., None].astype(np.int64), -1)[..., 0]
    assert np.all(chosen <= best + 1e-6 * scales[..., None] + 1e-30)


def test_lowbit_pool_attention_matches_sdpa_on_read_back_values():
    """A low-bit pool reads back code·scale + zero for every (token, head) row, and decode over it
    equals dense SDPA (fp64, torch) over those read-back values through the block table."""
    bits, G = 4, 32
    r = _rng(43)
    nb, n_kv, d_h, bs, n_q = 9, 2, 128, 16, 8
    n = nb * bs - 7
    k = _bf16(r.standard_normal((n, n_kv, d_h)).astype(np.float32))
    v = _bf16(r.standard_normal((n, n_kv, d_h)).astype(np.float32))
    slots = r.permutation(nb * bs)[:n].astype(np.int64)
    pool = oracle.OraclePool(nb, n_kv, d_h, bs, lowbit=(bits, G))
    assert pool.append(k, v, slots) == 0
    kc, ks, kz = oracle.quantize_rows_lowbit(k, bits, G)
    for t, s in enumerate(slots):
        p, o = divmod(int(s), bs)
        assert np.array_equal(pool.k_codes[p, :, o], kc[t]) and np.array_equal(pool.k_scales[p, :, o], ks[t])
        want = kc[t].reshape(n_kv, -1, G) * ks[t][..., None].astype(np.float64) + kz[t][..., None].astype(np.float64)
        assert np.array_equal(pool.k[p, :, o], want.reshape(n_kv, d_h))
    q = _bf16(r.standard_normal((1, n_q, d_h)).astype(np.float32))
    table = np.array([r.permutation(nb)], np.int32)
    ln = n - 3
    res = oracle.decode(pool, q, n_q, table, np.array([ln], np.int32))
    kv, vv = pool.values()
    kl = np.stack([kv[table[0, t // bs], :, t % bs] for t in range(ln)])
    vl = np.stack([vv[table[0, t // bs], :, t % bs] for t in range(ln)])
    ref = _dense_sdpa(q[0].astype(np.float64), kl, vl, 1 / np.sqrt(d_h))
    np.testing.assert_allclose(res["out"][0], ref, rtol=1e-12, atol=1e-12)


def test_lowbit_bytes_and_intensity_closed_forms():
    """Bytes per (token, KV head) row: d_h·bits/8 of codes plus two half-precision numbers per
    group; with the codes alone, 2-bit storage at g = 8 gives the page's 64 FLOP/B floor."""
    import bench

    for bits, row in ((4, 64 + 16), (2, 32 + 16)):
        assert 128 * bits // 8 + (128 // 32) * 4 == row
    assert bench.decode_intensity(8, 0.25) == 64 and bench.decode_intensity(8, 0.5) == 32


# ------------------------------------------------------------- angle-domain keys
def _angle_case(seed, rows=300, d=128):
    r = _rng(seed)
    x = r.standard_normal((rows, d)).astype(np.float32)
    x[3] = 0.0                                     # a zero row
    x[4] *= 1000.0                                 # a wide row
    x[5, 7] = 250.0                                # one outlier
    x[6] *= 1e-3                                   # a small row (subnormal codes)
    return _bf16(x)


def _torch_e4m3_codes(x):
    """Codes of each row at its absmax scale through torch's float8_e4m3fn cast (fp32 quotient)."""
    amax = np.abs(x).max(-1).astype(np.float32)
    scale = np.where(amax == 0, np.float32(1), (amax / np.float32(448)).astype(np.float32)).astype(np.float32)
    y = torch.from_numpy((x / scale[:, None]).astype(np.float32)).clamp(-448, 448)
    c = y.to(torch.float8_e4m3fn)
    return c.view(torch.uint8).numpy(), c.to(torch.float64).numpy()


def test_angle_key_rows_radius_code_and_factor():
    """Angle-domain keys ("기술 요약: Spherical KV", §2.1: radius r = ||k|| kept quantised, direction kept
    as a code): r̃ is numpy's float16 of the fp64 norm; the direction code is torch's E4M3 cast of the
    row at its absmax scale; the key attention sees, w·d, has the stored radius as its norm (to the fp32
    rounding of w) and points within the E4M3 direction error of k (3 mantissa bits: cos >= 1 - 2^-7)."""
    x = _angle_case(60)
    codes, w, rad = oracle.angle_key_rows(x)
    xd = x.astype(np.float64)
    norm = np.linalg.norm(xd, axis=1)
    assert np.array_equal(rad, norm.astype(np.float16).astype(np.float32))
    tc, tv = _torch_e4m3_codes(x)
    assert np.array_equal(codes, tc)
    keff = w[:, None].astype(np.float64) * tv
    nz = norm > 0
    assert np.all(np.abs(np.linalg.norm(keff, axis=1)[nz] - rad[nz]) <= 2.0 ** -23 * rad[nz])
    cos = (keff * xd).sum(1)[nz] / (np.linalg.norm(keff, axis=1)[nz] * norm[nz])
    assert cos.min() >= 1 - 2.0 ** -7, cos.min()
    assert w[3] == 0 and rad[3] == 0 and np.all(codes[3] == 0)


def test_angle_direction_code_ignores_the_radius():
    """Scaling a key by 2^j leaves its direction code unchanged and scales r̃ and w by 2^j."""
    x = _angle_case(61, rows=50)
    x = x[np.abs(x).max(1) < 100]
    c0, w0, r0 = oracle.angle_key_rows(x)
    for j in (-3, 2, 5):
        c, w, r = oracle.angle_key_rows((x * np.float32(2.0 ** j)).astype(np.float32))
        assert np.array_equal(c, c0)
        assert np.array_equal(r, (r0 * np.float32(2.0 ** j)).astype(np.float32))
        assert np.array_equal(w, (w0 * np.float32(2.0 ** j)).astype(np.float32))


def test_angle_logit_is_the_cosine_form():
    """<angle_query(q), w·d_k> = ||q||·r̃·<d_q, d_k>/(||d_q||·||d_k||), the page's ℓ̂ = ||q||·r̃·f_b(c_q, c_k)
    with f_b the cosine of the two codes (codes decoded through torch, norms by numpy); for rows already on
    the E4M3 grid at their absmax scale it is (r̃/||k||)·<q, k>."""
    q = _angle_case(62, rows=40)
    k = _angle_case(63, rows=40)
    qe = oracle.angle_query(q)
    kc, w, rad = oracle.angle_key_rows(k)
    _, dq = _torch_e4m3_codes(q)
    _, dk = _torch_e4m3_codes(k)
    got = (qe * (w[:, None].astype(np.float64) * dk)).sum(1)
    nq = np.linalg.norm(q.astype(np.float64), axis=1)
    with np.errstate(invalid="ignore", divide="ignore"):
        cosf = (dq * dk).sum(1) / (np.linalg.norm(dq, axis=1) * np.linalg.norm(dk, axis=1))
    want = np.where(np.isfinite(cosf), nq * rad * cosf, 0.0)
    np.testing.assert_allclose(got, want, rtol=1e-6, atol=1e-12)
    # on-grid rows: values e4m3 numbers times 2^j with absmax exactly 448·2^j
    r = _rng(64)
    grid = np.array([oracle.e4m3_decode(np.array([c], np.uint8))[0] for c in range(0, 127)])
    for j in (-4, 0, 3):
        qv = (r.choice(np.concatenate([grid, -grid]), size=128) * 2.0 ** j).astype(np.float32)
        kv = (r.choice(np.concatenate([grid, -grid]), size=128) * 2.0 ** j).astype(np.float32)
        qv[0], kv[5] = np.float32(448 * 2.0 ** j), np.float32(-448 * 2.0 ** j)
        qa = oracle.angle_query(qv[None])[0]
        _, wk, rk = oracle.angle_key_rows(kv[None])
        np.testing.assert_array_equal(qa, qv.astype(np.float64))
        lhs = float(qa @ (wk[0] * oracle.e4m3_decode(oracle.angle_key_rows(kv[None])[0][0]).astype(np.float64)))
        rhs = float(rk[0]) / np.linalg.norm(kv.astype(np.float64)) * float(qv.astype(np.float64) @ kv.astype(np.float64))
        assert abs(lhs - rhs) <= 1e-6 * abs(rhs) + 1e-9


def test_angle_pool_attention_matches_sdpa():
    """Decode over an angle-domain pool, with the query passed through angle_query, equals dense SDPA
    (fp64, torch) over keys w·d_k and values v_scale·d_v decoded through torch's float8 cast."""
    r = _rng(65)
    nb, n_kv, d_h, bs, n_q = 7, 2, 128, 16, 8
    n = nb * bs - 5
    k = _bf16(r.standard_normal((n, n_kv, d_h)).astype(np.float32))
    v = _bf16(r.standard_normal((n, n_kv, d_h)).astype(np.float32))
    slots = r.permutation(nb * bs)[:n].astype(np.int64)
    pool = oracle.OraclePool(nb, n_kv, d_h, bs, angle=True)
    assert pool.append(k, v, slots) == 0
    q = _bf16(r.standard_normal((1, n_q, d_h)).astype(np.float32))
    table = np.array([r.permutation(nb)], np.int32)
    res = oracle.decode(pool, oracle.angle_query(q), n_q, table, np.array([n], np.int32))
    _, kw, _ = oracle.angle_key_rows(k.reshape(-1, d_h))
    _, kd = _torch_e4m3_codes(k.reshape(-1, d_h))
    vsc = np.where(np.abs(v).max(-1) == 0, 1, (np.abs(v).max(-1) / np.float32(448)).astype(np.float32))
    _, vd = _torch_e4m3_codes(v.reshape(-1, d_h))
    # per physical slot: token t was written at slot slots[t]; the 5 slots never written read as 0
    kslot = np.zeros((nb * bs, n_kv, d_h))
    vslot = np.zeros((nb * bs, n_kv, d_h))
    kslot[slots] = (kw[:, None] * kd).reshape(n, n_kv, d_h)
    vslot[slots] = (vsc.reshape(-1)[:, None].astype(np.float64) * vd).reshape(n, n_kv, d_h)
    kl = np.stack([kslot[int(table[0, t // bs]) * bs + t % bs] for t in range(n)])
    vl = np.stack([vslot[int(table[0, t // bs]) * bs + t % bs] for t in range(n)])
    qa = oracle.angle_query(q)[0]
    ref = _dense_sdpa(qa, kl, vl, 1 / np.sqrt(d_h))
    np.testing.assert_allclose(res["out"][0], ref, rtol=1e-12, atol=1e-12)
