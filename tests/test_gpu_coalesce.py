"""Coalesced token tiles (moe_forward_opts.coalesce_rows) on the GPU.

The index pads each expert to block_m = 16 rows; the GEMMs walk a work list
of tiles of up to C consecutive rows of one expert.  Routing here is skewed
(Zipf-shaped expert popularity, as in the Zipf-routed workload), so some
experts hold more than C rows (several work tiles, the last one ragged) and
others a handful.  Checked: the layer against the oracle, bit-equality with
the same call on the task map (each output element is the same sequence of
MMAs and promotions), the index metadata bit-exact against the oracle's, and
the work list against its definition from the oracle's counts and offsets."""
import numpy as np
import pytest
import torch

import oracle
from moe_expert_layer_align_gb300 import workloads
from helpers import assert_layer_close, oracle_layer, run_layer

pytestmark = pytest.mark.gpu

INDEX_FIELDS = ("counts", "offsets", "sorted_ids", "tile_expert", "tiles", "inv_pos", "num_tiles")


def skewed_routing(T, k, E, seed, s=1.2):
    """Top-k ids drawn without replacement with Zipf(s) expert popularity
    (hot experts at random ids) and renormalised random weights."""
    rng = np.random.default_rng(seed)
    p = 1.0 / np.arange(1, E + 1) ** s
    p /= p.sum()
    perm = rng.permutation(E)
    ids = np.stack([perm[rng.choice(E, k, replace=False, p=p)] for _ in range(T)])
    w = rng.random((T, k)) + 0.1
    w /= w.sum(1, keepdims=True)
    return (torch.from_numpy(ids.astype(np.int32)).cuda(),
            torch.from_numpy(w.astype(np.float32)).cuda())


def expected_work_list(counts, offsets, C, tiles_cap):
    """Tiles of up to C rows of each expert with rows, in expert order, padded
    with {-1, 0, 0, 0} to tiles_cap."""
    tiles = []
    for e, c in enumerate(counts):
        for j in range(0, int(c), C):
            tiles.append((e, int(offsets[e]) + j, min(C, int(c) - j), 0))
    n = len(tiles)
    tiles += [(-1, 0, 0, 0)] * (tiles_cap - n)
    return np.array(tiles, np.int32), n


CASES = [
    # cfg, T, overrides, C, smem_index, opts
    (3, 80, dict(H=256, I=128, E=32), 64, False, {}),
    (3, 80, dict(H=256, I=128, E=32), 32, False, {}),
    (3, 80, dict(H=256, I=256, E=32), 64, False, dict(split_gateup=2)),   # separate SiLU-and-mul
    (3, 80, dict(H=256, I=256, E=32), 64, False, dict(split_down=3, unit_order=1)),
    (1, 40, dict(E=8), 32, True, {}),
    (1, 72, dict(E=8), 64, True, dict(unit_order=2)),
    (4, 80, dict(H=512, I=256, E=32), 64, False, {}),
    (4, 80, dict(H=512, I=256, E=32), 32, False, dict(unit_order=1)),
    (4, 80, dict(H=512, I=256, E=32), 64, False, dict(split_down=2, unit_order=2)),
    (4, 30, dict(H=512, I=256, E=16), 64, True, {}),
]


@pytest.mark.parametrize("cfg,T,kw,C,smem_index,extra", CASES)
def test_coalesced_tiles_match_oracle_and_task_map(cfg, T, kw, C, smem_index, extra):
    import moe_expert_layer_align_gb300 as moe
    wl = workloads.make(cfg, T, "cpu", **kw).to("cuda")
    ids, w = skewed_routing(T, wl.k, wl.E, seed=1000 + T + C)
    w13 = wl.w13 if wl.mode == "bf16" else wl.w13q
    out_dtype = torch.float32 if wl.out == "f32" else torch.bfloat16
    shape = moe.layer_shape(wl.x, w13, ids, 16, out_dtype)
    outs = {}
    for c in (C, -1):
        opts = moe.make_opts(coalesce_rows=c, smem_index=smem_index, **extra)
        ws = torch.zeros(moe.moe_workspace_bytes(shape, opts), dtype=torch.uint8, device="cuda")
        status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        outs[c] = run_layer(wl, topk_ids=ids, topk_w=w, block_m=16, opts=opts,
                            dev_status=status, workspace=ws)
        torch.cuda.synchronize()
        assert status.item() == 0, moe.device_status_bits(status.item())
        v = moe.workspace_views(ws, shape, opts)
        L = v["layout"]
        assert L.block_m == 16 and L.smem_index == int(smem_index)
        assert L.coalesce_rows == (C if c > 0 else 0)
        ref = oracle.align(ids.cpu().numpy(), wl.E, 16)
        for n in INDEX_FIELDS:
            np.testing.assert_array_equal(v[n].cpu().numpy().reshape(-1), ref[n].reshape(-1), n)
        if c > 0 and not smem_index:
            # (with the shared-memory index each CTA keeps its work list on chip)
            exp, n_exp = expected_work_list(ref["counts"], ref["offsets"], C, L.work_cap)
            assert v["num_work_tiles"].item() == n_exp
            np.testing.assert_array_equal(v["work_tiles"].cpu().numpy(), exp)
    counts = np.bincount(ids.cpu().numpy().reshape(-1), minlength=wl.E)
    assert counts.max() > C or smem_index, counts          # a hot expert spans work tiles
    assert ((counts > 16) & (counts % 16 != 0)).any(), counts   # ragged multi-box tiles
    assert torch.equal(outs[C], outs[-1]), (outs[C].float() - outs[-1].float()).abs().max()
    assert_layer_close(outs[C].double().cpu().numpy(),
                       oracle_layer(wl, topk_ids=ids.cpu(), topk_w=w.cpu()), wl.mode,
                       f"cfg{cfg} T={T} C={C}")


DOWN_SPLIT_CASES = [
    # cfg, T, overrides: 150, 175 and 300 rows per expert (256-row index tiles)
    (3, 300, dict(H=256, I=128, E=16)),
    (2, 700, dict(H=256, I=384)),
    (3, 600, dict(H=256, I=128, E=16)),
    (1, 600, dict(E=8)),
]


@pytest.mark.parametrize("cfg,T,kw", DOWN_SPLIT_CASES)
def test_down_tiles_of_128_rows_over_a_256_row_index(cfg, T, kw):
    """down_tile_rows=128: the Gate-Up keeps the 256-row token-major tiles of
    the task map, the Down GEMM takes a work list of tiles of up to 128 rows
    of the same index (more entries than the task map: its own capacity)."""
    import moe_expert_layer_align_gb300 as moe
    wl = workloads.make(cfg, T, "cpu", **kw).to("cuda")
    out_dtype = torch.float32 if wl.out == "f32" else torch.bfloat16
    shape = moe.layer_shape(wl.x, wl.w13, wl.topk_ids, 0, out_dtype)
    opts = moe.make_opts(down_tile_rows=128, smem_index=False)
    ws = torch.zeros(moe.moe_workspace_bytes(shape, opts), dtype=torch.uint8, device="cuda")
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    out = run_layer(wl, opts=opts, dev_status=status, workspace=ws)
    torch.cuda.synchronize()
    assert status.item() == 0, moe.device_status_bits(status.item())
    v = moe.workspace_views(ws, shape, opts)
    L = v["layout"]
    assert L.block_m == 256 and L.down_tile_rows == 128 and L.coalesce_rows == 0
    ref = oracle.align(wl.topk_ids.cpu().numpy(), wl.E, 256)
    for n in INDEX_FIELDS:
        np.testing.assert_array_equal(v[n].cpu().numpy().reshape(-1), ref[n].reshape(-1), n)
    exp, n_exp = expected_work_list(ref["counts"], ref["offsets"], 128, L.work_cap)
    assert v["num_work_tiles"].item() == n_exp > int(v["num_tiles"].item())
    np.testing.assert_array_equal(v["work_tiles"].cpu().numpy(), exp)
    assert_layer_close(out.double().cpu().numpy(), oracle_layer(wl), wl.mode, f"cfg{cfg} T={T}")
