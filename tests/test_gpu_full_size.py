"""Parity at the workloads' full sizes, in the launch configuration the
benchmark times: the Layer of bench.py (router where it is in the path, then
moe_forward with the planner's own choices, captured in a CUDA graph and
replayed).  The routing index is compared whole and bit-exact; the layer
output on sampled tokens (first, last and seeded random ones), which the
oracle computes one by one; the in-path router on the same tokens."""
import numpy as np
import pytest
import torch

import oracle
from moe_expert_layer_align_gb300 import workloads
from helpers import (SCORE_TOL, assert_layer_close, bits16, check_topk, oracle_layer_sampled)

pytestmark = pytest.mark.gpu

# config -> [(T, sampled tokens)]; the largest token count of every sweep, the
# decode sizes the benchmark reports first, and T=1.
CASES = {
    1: [(8, 8)],
    2: [(64, 16), (2048, 6), (1, 1)],
    3: [(1, 1), (64, 16), (4096, 48)],
    4: [(1, 1), (64, 6), (4096, 4)],
    5: [(4, 4), (256, 32)],
}


@pytest.fixture(scope="module")
def bases():
    cache = {}

    def get(cfg):
        if cfg not in cache:
            cache.clear()          # one full-size weight set on the device at a time
            torch.cuda.empty_cache()
            cache[cfg] = workloads.make(cfg, 1, "cuda")
        return cache[cfg]
    return get


def sample(T, n, seed):
    if n >= T:
        return np.arange(T)
    rng = np.random.default_rng(seed)
    mid = rng.choice(np.arange(1, T - 1), size=n - 2, replace=False)
    return np.sort(np.concatenate([[0, T - 1], mid]))


@pytest.mark.parametrize("cfg,T,n", [(c, T, n) for c, v in CASES.items() for T, n in v])
def test_full_size_layer(cfg, T, n, bases):
    import bench
    import moe_expert_layer_align_gb300 as moe
    wl = bench.make_workload(cfg, T, "cuda", base=bases(cfg))
    stream = torch.cuda.Stream()
    layer = bench.Layer(wl, stream)          # graph-captured, planner defaults
    layer.run()
    layer.run()                              # a replay over the same buffers
    stream.synchronize()
    assert layer.status.item() == 0

    ids = layer.ids.cpu().numpy()
    w = layer.w.cpu().numpy()
    sel = sample(T, n, 1000 * cfg + T)
    if wl.wr is not None:
        # router in the path: scores and top-k of the sampled tokens
        ref_s = oracle.router_scores(bits16(wl.x[torch.from_numpy(sel).cuda()]),
                                     wl.wr.cpu().numpy())
        got_s = layer.scores.cpu().numpy()[sel]
        assert np.abs(got_s - ref_s).max() <= SCORE_TOL
        ref_ids, _ = oracle.router_topk(ref_s, wl.k, wl.router_fn, wl.router_scale)
        check_topk(ids[sel], ref_ids, ref_s, wl.k, got_s)
        np.testing.assert_allclose(w[sel].sum(1), wl.router_scale, rtol=1e-5)

    # the whole index, bit-exact
    v = moe.workspace_views(layer.ws, layer.shape, routed=wl.wr is not None)
    L = v["layout"]
    ref = oracle.align(ids, wl.E, L.block_m)
    assert ref["invalid"] == 0
    for name in ("counts", "offsets", "sorted_ids", "tile_expert", "tiles", "inv_pos",
                 "num_tiles"):
        np.testing.assert_array_equal(v[name].cpu().numpy().reshape(-1),
                                      ref[name].reshape(-1), name)

    # the output of the sampled tokens (the oracle fed the routing the path used)
    got = layer.out.float().cpu().numpy()[sel]
    want = oracle_layer_sampled(wl, ids, w, sel)
    assert_layer_close(got, want, wl.mode, f"cfg{cfg} T={T} bm={L.block_m}")


# Prefill sizes: whole token tiles of the Down output (every row of the tile,
# so every TMEM lane quadrant and every epilogue warp of both GEMMs is read),
# for the fullest tile (a full one in the middle of the index where there is
# one) and the most ragged one.
TILE_CASES = [(2, 2048), (3, 4096), (4, 4096), (4, 512)]


def expert_rows_oracle(wl, e, tokens):
    """The expert-e output y = W2[e] (SiLU(x W1[e]^T) * x W3[e]^T) of each token
    (the oracle's layer over expert e alone, k = 1, weight 1; a selection of
    inputs, no arithmetic)."""
    n = len(tokens)
    ids = np.zeros((n, 1), np.int32)
    w = np.ones((n, 1), np.float32)
    rows = torch.from_numpy(np.asarray(tokens)).long().to(wl.x.device)
    x = bits16(wl.x[rows])
    sl = slice(e, e + 1)
    if wl.mode == "bf16":
        return oracle.moe_bf16(x, bits16(wl.w13[sl]), bits16(wl.w2[sl]), ids, w)
    from helpers import u8
    xq, xs = oracle.quant_x(x)
    return oracle.moe_fp8(xq, xs, u8(wl.w13q[sl]), wl.w13s[sl].cpu().numpy(), u8(wl.w2q[sl]),
                          wl.w2s[sl].cpu().numpy(), ids, w)


@pytest.mark.parametrize("cfg,T", TILE_CASES)
def test_full_size_whole_tiles(cfg, T, bases):
    import bench
    import moe_expert_layer_align_gb300 as moe
    wl = bench.make_workload(cfg, T, "cuda", base=bases(cfg))
    stream = torch.cuda.Stream()
    layer = bench.Layer(wl, stream)
    layer.run()
    stream.synchronize()
    assert layer.status.item() == 0
    v = moe.workspace_views(layer.ws, layer.shape, routed=wl.wr is not None)
    L = v["layout"]
    tiles = v["tiles"].cpu().numpy()
    nt = int(v["num_tiles"].item())
    sorted_ids = v["sorted_ids"].cpu().numpy()
    valid = tiles[:nt, 2]
    full = np.nonzero(valid == L.block_m)[0]
    fullest = int(full[len(full) // 2]) if len(full) else int(np.argmax(valid))
    picks = {fullest, int(np.argmin(np.where(valid > 0, valid, 1 << 30)))}
    Y = v["Y"]
    for q in sorted(picks):
        e, r0, nv = int(tiles[q, 0]), int(tiles[q, 1]), int(tiles[q, 2])
        a = sorted_ids[r0:r0 + nv]
        assert np.all(a < T * wl.k)
        got = Y[:, r0:r0 + nv, :].double().sum(0).cpu().numpy()
        want = expert_rows_oracle(wl, e, a // wl.k)
        assert_layer_close(got, want, wl.mode,
                           f"cfg{cfg} T={T} tile {q} (expert {e}, {nv} rows, bm={L.block_m})")
