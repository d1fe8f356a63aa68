"""Pins of the oracle's routing index ("routing and index build", HPC-Ops ×
SGLang, section MoE): a worked example derived by hand, a naive rescan on
random inputs, invariants, and degenerate cases."""
import numpy as np
import pytest

import oracle


def test_hand_worked_example():
    # T=3, k=2, E=4, bm=2.  Flat assignments a = t*k + j:
    #   a:  0  1  2  3  4  5
    #   e:  2  0  2  3  0  2
    # counts = [2, 0, 3, 1] -> padded [2, 0, 4, 2] -> offsets [0, 2, 2, 6, 8]
    # expert 0 rows 0..1: a = 1, 4; expert 2 rows 2..5: a = 0, 2, 5, pad;
    # expert 3 rows 6..7: a = 3, pad.  Sentinel = T*k = 6.
    # tiles_cap = ceil(6/2) + min(4, 6) = 7, rows_cap = 14, num_tiles = 4.
    r = oracle.align(np.array([[2, 0], [2, 3], [0, 2]], np.int32), E=4, bm=2)
    assert r["counts"].tolist() == [2, 0, 3, 1]
    assert r["offsets"].tolist() == [0, 2, 2, 6, 8]
    assert r["sorted_ids"].tolist() == [1, 4, 0, 2, 5, 6, 3, 6, 6, 6, 6, 6, 6, 6]
    assert r["inv_pos"].tolist() == [2, 0, 3, 6, 1, 4]
    assert r["num_tiles"][0] == 4
    assert r["tile_expert"].tolist() == [0, 2, 2, 3, -1, -1, -1]
    assert r["tiles"].tolist() == [[0, 0, 2, 0], [2, 2, 2, 0], [2, 4, 1, 0], [3, 6, 1, 0],
                                   [-1, 8, 0, 0], [-1, 10, 0, 0], [-1, 12, 0, 0]]
    assert r["invalid"] == 0


def naive_index(ids, E, bm):
    """Independent rescan: for each expert, walk every assignment in order."""
    T, k = ids.shape
    flat = ids.reshape(-1)
    tk = T * k
    rows, inv, offs = [], [-1] * tk, [0]
    for e in range(E):
        mine = [a for a in range(tk) if flat[a] == e]
        for a in mine:
            inv[a] = len(rows)
            rows.append(a)
        while len(rows) % bm:
            rows.append(tk)
        offs.append(len(rows))
    return rows, inv, offs


@pytest.mark.parametrize("seed", range(12))
def test_random_matches_naive_rescan_and_invariants(seed):
    rng = np.random.default_rng(seed)
    T = int(rng.integers(1, 60))
    E = int(rng.integers(1, 40))
    k = int(rng.integers(1, min(E, 8) + 1))
    bm = int(rng.choice([1, 2, 4, 16, 32]))
    # k distinct experts per token (top-k never repeats an expert)
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    r = oracle.align(ids, E, bm)
    rows, inv, offs = naive_index(ids, E, bm)
    tk = T * k
    assert r["offsets"].tolist() == offs
    assert r["sorted_ids"][: len(rows)].tolist() == rows
    assert np.all(r["sorted_ids"][len(rows):] == tk)
    assert r["inv_pos"].tolist() == inv
    check_invariants(ids, E, bm, r)


def check_invariants(ids, E, bm, r):
    T, k = ids.shape
    tk = T * k
    s = r["sorted_ids"]
    valid = s[s < tk]
    # every (t, j) exactly once; every token exactly k times
    assert sorted(valid.tolist()) == [a for a in range(tk) if 0 <= ids.reshape(-1)[a] < E]
    assert np.all(np.bincount(valid // k, minlength=T) == (ids < E).sum(1) - (ids < 0).sum(1))
    off, cnt = r["offsets"], r["counts"]
    assert np.all(off % bm == 0)
    pad = np.diff(off) - cnt
    assert np.all((pad >= 0) & (pad < bm))
    assert cnt.sum() == valid.size
    for p in np.flatnonzero(s < tk):
        assert r["inv_pos"][s[p]] == p
    for e in range(E):
        seg = s[off[e]: off[e + 1]]
        v = seg[seg < tk]
        assert np.all(ids.reshape(-1)[v] == e)
        assert np.all(np.diff(v) > 0)                       # ascending a (stable)
        assert np.all(seg[cnt[e]:] == tk)
    nt = r["num_tiles"][0]
    assert nt == off[E] // bm
    for q in range(r["tiles_cap"]):
        e, row0, nv, z = r["tiles"][q]
        assert row0 == q * bm and z == 0
        if q < nt:
            assert off[e] <= row0 < off[e + 1] and r["tile_expert"][q] == e
            assert nv == min(bm, off[e] + cnt[e] - row0) and nv >= 1
        else:
            assert e == -1 and nv == 0 and r["tile_expert"][q] == -1


def test_degenerate_cases():
    # T = 1
    r = oracle.align(np.array([[5, 1]], np.int32), E=8, bm=16)
    assert r["num_tiles"][0] == 2 and r["offsets"][-1] == 32
    check_invariants(np.array([[5, 1]], np.int32), 8, 16, r)
    # every token on one expert
    ids = np.full((40, 1), 3, np.int32)
    r = oracle.align(ids, E=4, bm=16)
    assert r["counts"].tolist() == [0, 0, 0, 40]
    assert r["offsets"].tolist() == [0, 0, 0, 0, 48]
    assert r["sorted_ids"][:40].tolist() == list(range(40))
    check_invariants(ids, 4, 16, r)
    # E > T*k: most experts empty, no tiles for them
    ids = np.array([[200, 7]], np.int32)
    r = oracle.align(ids, E=256, bm=16)
    assert r["num_tiles"][0] == 2 and r["tiles_cap"] == 1 + 2
    check_invariants(ids, 256, 16, r)


def test_invalid_ids_are_dropped():
    ids = np.array([[0, 9], [-1, 1], [1, 0]], np.int32)
    r = oracle.align(ids, E=2, bm=4)
    assert r["invalid"] == 2
    assert r["inv_pos"][1] == -1 and r["inv_pos"][2] == -1
    assert r["counts"].tolist() == [2, 2]
    assert r["sorted_ids"][:8].tolist() == [0, 5, 6, 6, 3, 4, 6, 6]


def test_config_shapes_hold_invariants():
    rng = np.random.default_rng(11)
    for T, E, k, bm in [(8, 8, 2, 16), (64, 8, 2, 32), (64, 128, 8, 16), (512, 256, 8, 64)]:
        ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
        check_invariants(ids, E, bm, oracle.align(ids, E, bm))
