"""Host-side tier reassignment (kvd_tier_reassign): only blocks whose planned tier differs from
their current one move (page "기술 요약: 모든 사고가 HBM 을 필요로 하는 것은 아님", section
"4. 시스템 구현"), destinations come from the planned tier's free list, sources go back to
their own tier's list, and the tables stay consistent.  Pure host code: no GPU needed."""

import numpy as np
import pytest

import paged_gqa_decode_kvd_gb300 as kvd


def _state(nb, nh, tables, free_hbm, free_host):
    hf = np.zeros(nb, np.int32)
    hf[:len(free_hbm)] = free_hbm
    tf = np.zeros(max(1, nh), np.int32)
    tf[:len(free_host)] = free_host
    return np.array(tables, np.int32), hf, len(free_hbm), tf, len(free_host)


def _check_consistent(nb, nh, bt, tier, hf, hn, tf, tn):
    """Every planned entry sits in its tier; referenced and free ids are disjoint and in range."""
    used = set(int(x) for x, t in zip(bt.ravel(), tier.ravel()) if t >= 0)
    free_h, free_t = set(hf[:hn].tolist()), set(tf[:tn].tolist())
    assert len(free_h) == hn and len(free_t) == tn            # no id twice in a list
    assert all(0 <= x < nb for x in free_h) and all(nb <= x < nb + nh for x in free_t)
    assert not (used & free_h) and not (used & free_t)


def test_reassign_worked_example():
    nb, nh = 8, 4
    # two requests of 3 blocks; request 1's block 2 is unused (tier -1)
    bt, hf, hn, tf, tn = _state(nb, nh, [[0, 1, 2], [3, 4, 7]], [5, 6], [8, 9, 10, 11])
    tier = np.array([[0, 1, 1], [1, 0, -1]], np.int8)
    retain = np.arange(nb + nh, dtype=np.uint16) * 3
    st, frm, to, hn, tn = kvd.kvd_tier_reassign(nb, nh, tier, bt, hf, hn, tf, tn, retain)
    assert st == kvd.KVD_OK
    # destinations are popped from the end of the host list: 11, 10, 9 in entry order
    assert frm.tolist() == [1, 2, 3] and to.tolist() == [11, 10, 9]
    assert bt.tolist() == [[0, 11, 10], [9, 4, 7]]
    assert retain[11] == 3 and retain[10] == 6 and retain[9] == 9
    assert hf[:hn].tolist() == [5, 6, 1, 2, 3] and tf[:tn].tolist() == [8]
    _check_consistent(nb, nh, bt, tier, hf, hn, tf, tn)
    # the next reassignment promotes request 0's block 1 back and demotes request 1's block 1
    tier2 = np.array([[0, 0, 1], [1, 1, -1]], np.int8)
    st, frm, to, hn, tn = kvd.kvd_tier_reassign(nb, nh, tier2, bt, hf, hn, tf, tn, retain)
    assert st == kvd.KVD_OK
    assert frm.tolist() == [11, 4] and to.tolist() == [3, 8]
    assert bt.tolist() == [[0, 3, 10], [9, 8, 7]]
    assert retain[3] == 3 and retain[8] == 12     # block 11 carried block 1's bits (3)
    _check_consistent(nb, nh, bt, tier2, hf, hn, tf, tn)


def test_reassign_moves_a_shared_block_once():
    nb, nh = 6, 2
    bt, hf, hn, tf, tn = _state(nb, nh, [[0, 1], [0, 2]], [3], [6, 7])
    tier = np.array([[1, 0], [0, 0]], np.int8)   # the first entry's plan decides for block 0
    st, frm, to, hn, tn = kvd.kvd_tier_reassign(nb, nh, tier, bt, hf, hn, tf, tn)
    assert st == kvd.KVD_OK and frm.tolist() == [0] and to.tolist() == [7]
    assert bt.tolist() == [[7, 1], [7, 2]]


def test_reassign_out_of_free_blocks_and_bad_ids():
    nb, nh = 6, 1
    bt, hf, hn, tf, tn = _state(nb, nh, [[0, 1, 2]], [], [6])
    tier = np.array([[1, 1, 0]], np.int8)
    st, frm, to, hn, tn = kvd.kvd_tier_reassign(nb, nh, tier, bt, hf, hn, tf, tn)
    assert st == kvd.KVD_ERR_NOMEM                 # one host block for two demotions
    assert frm.tolist() == [0] and bt.tolist() == [[6, 1, 2]]
    _check_consistent(nb, nh, bt, np.array([[1, 0, 0]], np.int8), hf, hn, tf, tn)
    bt2, hf2, hn2, tf2, tn2 = _state(nb, nh, [[0, 9]], [], [6])
    st, frm, _, _, _ = kvd.kvd_tier_reassign(nb, nh, np.array([[1, 1]], np.int8), bt2, hf2, hn2, tf2, tn2)
    assert st == kvd.KVD_ERR_OOB and frm.tolist() == [0] and bt2.tolist() == [[6, 9]]
    bt3, hf3, hn3, tf3, tn3 = _state(nb, nh, [[0]], [], [2])   # an HBM id on the host free list
    with pytest.raises(kvd.KvdError):
        kvd.kvd_tier_reassign(nb, nh, np.array([[1]], np.int8), bt3, hf3, hn3, tf3, tn3)


def test_reassign_random_rounds_keep_every_invariant():
    rng = np.random.default_rng(8)
    for trial in range(40):
        nb, nh = int(rng.integers(4, 60)), int(rng.integers(0, 40))
        batch, mb = int(rng.integers(1, 5)), int(rng.integers(1, 12))
        ids = rng.permutation(nb + nh).astype(np.int32)
        n_used = min(batch * mb, nb + nh)
        bt = np.full((batch, mb), -1, np.int32)
        bt.ravel()[:n_used] = ids[:n_used]
        rest = ids[n_used:]
        hf = np.zeros(nb, np.int32)
        tf = np.zeros(max(1, nh), np.int32)
        fh, ft = rest[rest < nb], rest[rest >= nb]
        hf[:len(fh)], tf[:len(ft)] = fh, ft
        hn, tn = len(fh), len(ft)
        retain = rng.integers(0, 65536, nb + nh).astype(np.uint16)
        for rnd in range(3):
            tier = rng.integers(0, 2, (batch, mb)).astype(np.int8)
            tier[bt < 0] = -1
            before = bt.copy()
            payload = {int(x): int(retain[x]) for x in before.ravel() if x >= 0}
            st, frm, to, hn, tn = kvd.kvd_tier_reassign(nb, nh, tier, bt, hf, hn, tf, tn, retain)
            assert st in (kvd.KVD_OK, kvd.KVD_ERR_NOMEM)
            moved = dict(zip(frm.tolist(), to.tolist()))
            for e in range(batch * mb):
                if tier.ravel()[e] < 0:
                    continue
                p, q = int(before.ravel()[e]), int(bt.ravel()[e])
                assert q == moved.get(p, p)                          # follows its block
                assert retain[q] == payload[p]                       # with its retain bits
                if p in moved:
                    assert (q >= nb) == (tier.ravel()[e] == 1)       # into the planned tier
                elif st == kvd.KVD_OK:
                    assert (p >= nb) == (tier.ravel()[e] == 1)
            assert len(set(to.tolist())) == len(to) and not (set(to.tolist()) & set(frm.tolist()))
            _check_consistent(nb, nh, bt, np.where(bt >= 0, 0, -1).astype(np.int8), hf, hn, tf, tn)
