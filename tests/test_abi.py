"""The C-ABI library on the host: it loads, exports what include/kvd.h declares, sizes
pools by the closed form, and rejects bad arguments before touching a GPU."""

import ctypes
import os
import re

import pytest

import paged_gqa_decode_kvd_gb300 as kvd

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden")


def _declared():
    text = open(os.path.join(ROOT, "include", "kvd.h")).read()
    return sorted(set(re.findall(r"KVD_API\s+[\w\s\*]*?\b(kvd_\w+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    lib = kvd.load()
    names = _declared()
    assert len(names) >= 11
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(kvd.SYMBOLS) == names


def test_pool_bytes_closed_form_matches_pages():
    rows = [ln.split() for ln in open(os.path.join(GOLDEN, "kv_bytes.txt")) if ln.strip() and not ln.startswith("#")]
    models = {"8B": (32, 8, 128), "70B": (80, 8, 128)}
    for r in rows:
        if r[0] == "per_token":
            _, model, layers, kvh, dh, w, want = r
            dtype = kvd.KVD_BF16 if w == "2" else kvd.KVD_FP8_E4M3
            _, kv = kvd.kvd_pool_bytes(int(layers), int(kvh), 1, dtype)   # one block = 16 tokens
            assert kv // 16 == int(want)
        else:
            _, tokens, gib8, gib70 = r
            for model, want in (("8B", gib8), ("70B", gib70)):
                L, nkv, dh = models[model]
                _, kv = kvd.kvd_pool_bytes(L, nkv, int(tokens) // 16, kvd.KVD_BF16)
                assert abs(kv / 2 ** 30 - float(want)) <= 0.005 + 1e-12   # the page prints two decimals


def test_fp8_scale_bytes():
    pool, kv = kvd.kvd_pool_bytes(80, 8, 8192, kvd.KVD_FP8_E4M3)
    assert kv == 80 * 8192 * 16 * 8 * 128 * 2                  # 1 byte per element, K and V
    assert pool - kv == 80 * 8192 * 8 * 2 * 16 * 4             # one fp32 per (token, head) for K and V
    pool, kv = kvd.kvd_pool_bytes(32, 8, 16384, kvd.KVD_BF16)
    assert pool == kv == 32 * 8192 * 131072 // 8192 * 8192     # 32 GiB: 128 KiB per token


def test_lowbit_pool_bytes():
    """Low-bit pools: codes at w_kv = bits/8 (the closed form 2·L·n_kv·d_h·w_kv per token), plus a
    32-bit (scale, zero point) entry per (token, KV head, group) for K and for V."""
    for dtype, bits in ((kvd.KVD_INT4, 4), (kvd.KVD_INT2, 2)):
        for group in (32, 64, 128):
            pool, kv = kvd.kvd_pool_bytes(80, 8, 8192, dtype, group_size=group)
            tokens = 8192 * 16
            assert kv == 2 * 80 * 8 * 128 * bits * tokens // 8
            assert pool - kv == 2 * 80 * 8 * (128 // group) * 4 * tokens
    # angle-domain pools: FP8-sized records (codes, then one fp32 word per row for K and for V)
    assert kvd.kvd_pool_bytes(80, 8, 8192, kvd.KVD_ANGLE) == kvd.kvd_pool_bytes(80, 8, 8192, kvd.KVD_FP8_E4M3)
    # 70B shape, 128k context: 2-bit codes are an eighth of the BF16 bytes (the page's c = 8)
    _, bf16 = kvd.kvd_pool_bytes(80, 8, 8192, kvd.KVD_BF16)
    _, int2 = kvd.kvd_pool_bytes(80, 8, 8192, kvd.KVD_INT2, group_size=128)
    assert bf16 == 8 * int2


def test_host_tier_bytes():
    """A host tier of hb blocks holds every layer's records of those blocks in host memory;
    its HBM staging area holds two layers' worth (the prefetch of the next layer overlaps the
    attention of this one)."""
    for dtype, rec in ((kvd.KVD_BF16, 8192), (kvd.KVD_FP8_E4M3, 4224)):
        for hb in (0, 1, 37):
            host, staging = kvd.kvd_tier_bytes(28, 4, 1000, dtype, hb)
            assert host == 28 * hb * 4 * rec
            assert staging == 2 * hb * 4 * rec
    with pytest.raises(kvd.KvdError):
        kvd.kvd_tier_bytes(28, 4, 1000, kvd.KVD_BF16, -1)


def test_bad_descriptors_are_rejected():
    with pytest.raises(kvd.KvdError) as e:
        kvd.kvd_pool_bytes(32, 8, 16, kvd.KVD_BF16, d_h=64)
    assert e.value.status == kvd.KVD_ERR_UNSUPPORTED
    with pytest.raises(kvd.KvdError) as e:
        kvd.kvd_pool_bytes(32, 8, 16, kvd.KVD_BF16, block_size=32)
    assert e.value.status == kvd.KVD_ERR_UNSUPPORTED
    for bad in [dict(num_layers=0), dict(n_kv=0), dict(num_blocks=0), dict(kv_dtype=99)]:
        args = dict(num_layers=2, n_kv=8, num_blocks=16, kv_dtype=kvd.KVD_BF16)
        args.update(bad)
        with pytest.raises(kvd.KvdError) as e:
            kvd.kvd_pool_bytes(**args)
        assert e.value.status == kvd.KVD_ERR_INVALID


def test_null_arguments_fail_before_any_launch():
    lib = kvd.load()
    P = ctypes.c_void_p
    d = kvd._lib.PoolDesc(2, 8, 128, 16, 64, kvd.KVD_BF16)
    h = P()
    assert lib.kvd_pool_create(ctypes.byref(d), None, 1 << 20, ctypes.byref(h)) == kvd.KVD_ERR_INVALID
    assert lib.kvd_pool_create(ctypes.byref(d), P(16), 10, ctypes.byref(h)) == kvd.KVD_ERR_NOMEM
    assert lib.kvd_pool_create(ctypes.byref(d), P(8), 1 << 30, ctypes.byref(h)) == kvd.KVD_ERR_INVALID
    assert lib.kvd_decode_attn(None, 0, None, 32, None, None, None, 1, None, 1, 1, 0, None, 0.1, None, 0, None, 0,
                               None, None, 0, None, 0, None) == kvd.KVD_ERR_INVALID
    assert lib.kvd_decode_attn_noalloc(None, 0, None, 32, None, None, None, 1, None, 1, 1, 0, None, 0.1, None, 0,
                                       None, None, 0, None, 0, None) == kvd.KVD_ERR_INVALID
    assert lib.kvd_append_kv(None, 0, None, None, None, 1, None) == kvd.KVD_ERR_INVALID
    assert lib.kvd_combine_splits(None, None, None, None, 1, 32, 8, 64, None, 0, None, None) == \
        kvd.KVD_ERR_UNSUPPORTED
    assert lib.kvd_combine_splits(None, None, None, None, 1, 72, 8, 128, None, 0, None, None) == \
        kvd.KVD_ERR_UNSUPPORTED                      # g = 9 > 8
    assert lib.kvd_combine_splits(None, None, None, None, 0, 32, 8, 128, None, 0, None, None) == kvd.KVD_OK
    assert lib.kvd_accum_scores(None, 16, None, None, 1, 4, 1.0, None, 16, None) == kvd.KVD_ERR_INVALID
    assert lib.kvd_get_device_error(None, None, None) == kvd.KVD_ERR_INVALID
    assert lib.kvd_selftest_wait_timeout(None, 1000, None) == kvd.KVD_ERR_INVALID
    assert kvd.status_string(kvd.KVD_ERR_OOB) == "device-detected index out of range"
