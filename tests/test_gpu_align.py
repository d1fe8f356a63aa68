"""Routing index on the GPU (moe_align through the C ABI) against the oracle:
bit-exact on every field, over the workloads' shapes, random shapes and the
degenerate cases (T = 1, one hot expert, E > T*k, invalid ids)."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

FIELDS = ("counts", "offsets", "sorted_ids", "tile_expert", "tiles", "inv_pos", "num_tiles")


def gpu_align(ids_np, E, bm):
    import moe_expert_layer_align_gb300 as moe
    ids = torch.from_numpy(np.ascontiguousarray(ids_np, np.int32)).cuda()
    T, k = ids.shape
    st = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    idx = moe.alloc_index(T, k, E, bm)
    for v in idx.values():
        v.fill_(-7777)          # poison: every entry must be written
    moe.moe_align(ids, E, bm, idx, dev_status=st)
    torch.cuda.synchronize()
    return {n: idx[n].cpu().numpy() for n in FIELDS}, int(st.item())


def assert_index_equal(ids, E, bm):
    got, status = gpu_align(ids, E, bm)
    ref = oracle.align(ids, E, bm)
    for n in FIELDS:
        np.testing.assert_array_equal(got[n].reshape(-1), ref[n].reshape(-1), err_msg=n)
    return got, status, ref


def topk_ids(T, E, k, seed, zipf=None):
    rng = np.random.default_rng(seed)
    if zipf is None:
        return np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    p = np.arange(1, E + 1, dtype=np.float64) ** -zipf
    p /= p.sum()
    return np.stack([rng.choice(E, k, replace=False, p=p) for _ in range(T)]).astype(np.int32)


@pytest.mark.parametrize("T,E,k", [(8, 8, 2), (1, 8, 2), (64, 8, 2), (2048, 8, 2), (1, 128, 8),
                                   (64, 128, 8), (4096, 128, 8), (16, 256, 8), (4096, 256, 8)])
@pytest.mark.parametrize("bm", [16, 64, 256])
def test_workload_shapes(T, E, k, bm):
    _, status, ref = assert_index_equal(topk_ids(T, E, k, T * 7 + E), E, bm)
    assert status == 0


@pytest.mark.parametrize("seed", range(6))
def test_random_and_skewed(seed):
    rng = np.random.default_rng(100 + seed)
    T = int(rng.integers(1, 3000))
    E = int(rng.integers(1, 513))
    k = int(rng.integers(1, min(E, 8) + 1))
    bm = int(rng.choice([16, 32, 64, 128, 256]))
    assert_index_equal(topk_ids(T, E, k, seed, zipf=1.2 if seed % 2 else None), E, bm)


def test_degenerate():
    assert_index_equal(np.full((300, 1), 5, np.int32), 8, 16)      # one hot expert
    assert_index_equal(np.array([[200, 7]], np.int32), 256, 16)    # E > T*k
    assert_index_equal(np.array([[0]], np.int32), 1, 16)           # E = 1, T = 1
    big = np.stack([np.arange(8, dtype=np.int32)] * 4096)          # T*k = 32768, balanced
    assert_index_equal(big, 8, 256)


def test_beyond_staged_capacity():
    # more than 32768 assignments: ids are read from global memory
    assert_index_equal(topk_ids(5000, 64, 8, 9), 64, 128)


def test_invalid_ids_flagged_and_dropped():
    ids = topk_ids(50, 16, 4, 3)
    ids[3, 1] = -1
    ids[10, 0] = 16
    ids[49, 3] = 1 << 20
    got, status, ref = assert_index_equal(ids, 16, 16)
    assert ref["invalid"] == 3
    assert status == (1 << 6)                      # bit of MOE_ERR_EXPERT_ID
    assert got["inv_pos"][3 * 4 + 1] == -1


@pytest.mark.parametrize("seed", range(40))
def test_small_batches(seed):
    # at most 32 assignments (and 33, the first batch past the one-warp
    # build): random experts with repeats and invalid ids, every row tile
    rng = np.random.default_rng(500 + seed)
    E = int(rng.choice([1, 2, 7, 64, 128, 256, 512]))
    k = int(rng.integers(1, min(E, 8) + 1))
    T = int(rng.integers(1, 32 // k + 1)) if seed % 5 else (32 // k) + 1
    bm = int(rng.choice([16, 32, 64, 128, 256]))
    if seed % 3 == 0:
        ids = topk_ids(T, E, k, seed)
    else:
        ids = rng.integers(-2, E + 2, size=(T, k)).astype(np.int32)
    got, status, ref = assert_index_equal(ids, E, bm)
    assert status == (1 << 6 if ref["invalid"] else 0)


def test_small_batch_one_expert_and_boundaries():
    assert_index_equal(np.full((32, 1), 3, np.int32), 4, 16)       # 32 rows of one expert
    assert_index_equal(np.full((4, 8), 511, np.int32), 512, 256)   # the last expert
    assert_index_equal(np.arange(32, dtype=np.int32).reshape(4, 8), 32, 16)   # 32 experts
