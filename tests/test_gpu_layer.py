"""The whole layer on the GPU (moe_forward through the C ABI) against the
oracle, on small cases that span several tiles and ragged tails, and on the
intermediates the path leaves in its workspace (bit-exact where integer or
quantised)."""
import numpy as np
import pytest
import torch

import oracle
from moe_expert_layer_align_gb300 import workloads
from helpers import assert_layer_close, bits16, oracle_layer, run_layer, u8

pytestmark = pytest.mark.gpu


def small(cfg, T, **kw):
    return workloads.make(cfg, T, "cpu", **kw).to("cuda")


CASES = [
    # cfg, T, overrides
    (1, 8, {}),
    (1, 37, {}),
    (2, 5, dict(H=512, I=1024)),
    (2, 100, dict(H=512, I=448)),
    (3, 1, dict(H=256, I=192, E=32)),
    (3, 40, dict(H=384, I=192, E=32)),
    (3, 300, dict(H=256, I=128, E=16)),
    (4, 3, dict(H=512, I=256, E=16)),
    (4, 70, dict(H=384, I=384, E=12)),
]


@pytest.mark.parametrize("smem_index", [False, True])
@pytest.mark.parametrize("cfg,T,kw", CASES)
def test_layer_matches_oracle(cfg, T, kw, smem_index):
    import moe_expert_layer_align_gb300 as moe
    wl = small(cfg, T, **kw)
    # the index kernel (default) or every GEMM CTA rebuilding the index
    opts = moe.make_opts(smem_index=smem_index)   # both index paths, explicitly
    got = run_layer(wl, opts=opts).float().cpu().numpy()
    ref = oracle_layer(wl)
    assert_layer_close(got, ref, wl.mode, f"cfg{cfg} T={T}")


@pytest.mark.parametrize("bm", [16, 32, 64, 128, 256])
@pytest.mark.parametrize("mode_cfg", [2, 4])
def test_every_block_m(bm, mode_cfg):
    if mode_cfg == 4 and bm == 256:
        pytest.skip("FP8 tiles stop at 128 rows")
    kw = dict(H=256, I=256, E=6, k=4) if mode_cfg == 4 else dict(H=256, I=192, E=6)
    wl = small(mode_cfg, 150, **kw)
    got = run_layer(wl, block_m=bm).float().cpu().numpy()
    assert_layer_close(got, oracle_layer(wl), wl.mode, f"bm={bm}")


@pytest.mark.parametrize("s1,s2,sep", [(1, 1, False), (1, 2, True), (2, 3, False),
                                        (4, 8, False), (3, 1, False)])
@pytest.mark.parametrize("mode_cfg", [2, 4])
def test_forced_splits_and_no_pdl(s1, s2, sep, mode_cfg):
    import moe_expert_layer_align_gb300 as moe
    kw = dict(H=1024, I=512, E=8) if mode_cfg == 4 else dict(H=1024, I=512, E=8)
    wl = small(mode_cfg, 24, **kw)
    opts = moe.make_opts(disable_pdl=(s1 == 3), split_gateup=s1, split_down=s2,
                         separate_act=sep, smem_index=(s2 == 3))
    got = run_layer(wl, opts=opts).float().cpu().numpy()
    assert_layer_close(got, oracle_layer(wl), wl.mode, f"splits {s1},{s2}")


@pytest.mark.parametrize("fused,smem_index,I", [(True, False, 128), (False, False, 128),
                                               (True, True, 128), (False, False, 2112)])
def test_intermediates_bf16(fused, smem_index, I):
    import moe_expert_layer_align_gb300 as moe
    # I = 2112: activation rows of 264 eight-channel chunks (more than a block's threads)
    wl = small(2, 33, H=256, I=I, E=4)
    # unsplit Gate-Up fuses SiLU-and-mul into its epilogue; a split one
    # leaves fp32 partials for the separate stage.  The index comes from the
    # Gate-Up's CTA 0 (shared-memory mode) or from the index kernel.
    opts = moe.make_opts(split_gateup=1 if fused else 2, smem_index=smem_index)
    shape = moe.layer_shape(wl.x, wl.w13, wl.topk_ids, 0, torch.bfloat16)
    ws = torch.zeros(moe.moe_workspace_bytes(shape, opts), dtype=torch.uint8, device="cuda")
    run_layer(wl, workspace=ws, opts=opts)
    torch.cuda.synchronize()
    v = moe.workspace_views(ws, shape, opts)
    assert v["layout"].fused_act == int(fused)
    assert v["layout"].smem_index == int(smem_index)
    ref = oracle.align(wl.topk_ids.cpu().numpy(), wl.E, v["layout"].block_m)
    for n in ("counts", "offsets", "sorted_ids", "tile_expert", "tiles", "inv_pos", "num_tiles"):
        np.testing.assert_array_equal(v[n].cpu().numpy().reshape(-1), ref[n].reshape(-1), n)
    # Gate-Up sums (split case) and the bf16 activation of every valid row
    # against fp64 products
    sid = ref["sorted_ids"]
    X = wl.x.double().cpu().numpy()
    W13 = wl.w13.double().cpu().numpy()
    A = v["A"].double().cpu().numpy()
    G = None if fused else v["G"].sum(0).double().cpu().numpy()
    rows = np.flatnonzero(sid < wl.T * wl.k)
    I = wl.I
    for p in rows:
        a = sid[p]
        e = wl.topk_ids.reshape(-1)[a].item()
        g_ref = W13[e] @ X[a // wl.k]
        if G is not None:
            np.testing.assert_allclose(G[p], g_ref, rtol=1e-4, atol=1e-4 * np.abs(g_ref).max())
        act = g_ref[:I] / (1 + np.exp(-g_ref[:I])) * g_ref[I:]
        np.testing.assert_allclose(A[p], act, rtol=1e-2, atol=1e-2 * np.abs(act).max())


@pytest.mark.parametrize("smem_index,sepq,H,I", [(False, False, 512, 256), (True, False, 512, 256),
                                                 (False, True, 512, 256),
                                                 (False, False, 384, 256), (False, True, 384, 256),
                                                 (False, True, 2304, 256),
                                                 (False, False, 512, 2304)])
def test_intermediates_fp8_codes(smem_index, sepq, H, I):
    """x codes and scales bit-exact (an odd number of 128-channel groups,
    several blocks of group pairs per token), quantised on the index launch's
    other blocks or by their own kernel (sepq, which also writes the scales
    per index row), the index bit-exact, and the activation codes (rows of
    more than 256 eight-channel chunks) within a few rounding-edge flips of
    the oracle's."""
    import moe_expert_layer_align_gb300 as moe
    wl = small(4, 20, H=H, I=I, E=6, k=3)
    opts = moe.make_opts(smem_index=smem_index, separate_quant=sepq)
    shape = moe.layer_shape(wl.x, wl.w13q, wl.topk_ids, 0, torch.bfloat16)
    ws = torch.zeros(moe.moe_workspace_bytes(shape, opts), dtype=torch.uint8, device="cuda")
    got = run_layer(wl, workspace=ws, opts=opts).float().cpu().numpy()
    torch.cuda.synchronize()
    v = moe.workspace_views(ws, shape, opts)
    ref_idx = oracle.align(wl.topk_ids.cpu().numpy(), wl.E, v["layout"].block_m)
    for n in ("counts", "offsets", "sorted_ids", "tile_expert", "tiles", "inv_pos", "num_tiles"):
        np.testing.assert_array_equal(v[n].cpu().numpy().reshape(-1), ref_idx[n].reshape(-1), n)
    xq, xs = oracle.quant_x(bits16(wl.x))
    np.testing.assert_array_equal(v["xq"].cpu().numpy(), xq)          # bit-exact
    np.testing.assert_array_equal(v["xs"].cpu().numpy(), xs)
    assert v["layout"].xs_by_token == int(smem_index or not sepq)
    if not v["layout"].xs_by_token:
        # the same scales scattered to the index rows that hold each token
        sid = v["sorted_ids"].cpu().numpy()
        rows = np.flatnonzero(sid < wl.T * wl.k)
        np.testing.assert_array_equal(v["xs_rows"].cpu().numpy()[rows], xs[sid[rows] // wl.k])
    ref, aq, as_ = oracle_layer(wl, return_act=True)
    assert_layer_close(got, ref, "fp8", "fp8 layer")
    inv = v["inv_pos"].cpu().numpy()
    A = v["A"].cpu().numpy()
    As = v["As"].cpu().numpy()
    n_diff = 0
    for t in range(wl.T):
        for j in range(wl.k):
            p = inv[t * wl.k + j]
            n_diff += int((A[p] != aq[t, j]).sum())
            np.testing.assert_allclose(As[p], as_[t, j], rtol=1e-5)
    # codes come from fp32 values that differ from the oracle's only by
    # summation order: at most a few land on the other side of a rounding edge
    assert n_diff <= max(2, wl.T * wl.k * wl.I // 2000), n_diff


@pytest.mark.parametrize("cfg,T,kw", [(4, 1, dict(H=512, I=256, E=16)),
                                      (4, 70, dict(H=384, I=384, E=12)),
                                      (5, 40, dict(H=256, I=128, E=64))])
def test_fp8_quant_on_index_launch_equals_separate_kernel(cfg, T, kw):
    """FP8 with a one-CTA index: x quantised on the index launch's other
    blocks (per-token scales, looked up through the index by the Gate-Up)
    gives bitwise the codes, scales and output of the separate x-quant
    kernel with its per-row scales; the routed layer (workload 5) too."""
    import moe_expert_layer_align_gb300 as moe
    wl = small(cfg, T, **kw)
    routed = wl.wr is not None
    hi_lo = moe.moe_router_prepare(wl.wr) if routed else None
    ids = wl.topk_ids if not routed else torch.empty(T, wl.k)   # the shape only
    shape = moe.layer_shape(wl.x, wl.w13q, ids, 0, torch.bfloat16)
    res = {}
    for sepq in (False, True):
        opts = moe.make_opts(separate_quant=sepq)
        if routed:
            ws = torch.zeros(moe.moe_routed_workspace_bytes(shape, opts), dtype=torch.uint8,
                             device="cuda")
            out = moe.moe_forward_routed(wl.x, hi_lo, wl.k, wl.w13q, wl.w2q,
                                         scales=(wl.w13s, wl.w2s), workspace=ws, opts=opts)[0]
        else:
            ws = torch.zeros(moe.moe_workspace_bytes(shape, opts), dtype=torch.uint8,
                             device="cuda")
            out = run_layer(wl, workspace=ws, opts=opts)
        torch.cuda.synchronize()
        res[sepq] = (out, moe.workspace_views(ws, shape, opts, routed=routed))
    (o1, v1), (o0, v0) = res[False], res[True]
    assert (v1["layout"].xs_by_token, v0["layout"].xs_by_token) == (1, 0)
    assert torch.equal(o1, o0)
    for n in ("xq", "xs", "sorted_ids", "inv_pos"):
        assert torch.equal(v1[n], v0[n]), n
    if not routed:
        assert_layer_close(o1.float().cpu().numpy(), oracle_layer(wl), "fp8", "quant on index")


@pytest.mark.parametrize("T,kw", [(300, dict(H=512, I=384, E=4, k=2)),
                                  (150, dict(H=384, I=256, E=3, k=3))])
def test_fp8_gateup_stores_silu_rows(T, kw):
    """FP8 on 128-row token tiles: the unsplit Gate-Up's epilogue stores the
    rows of SiLU(gate)*up and the activation stage only quantises them.  The
    codes, scales and layer output are bitwise those of the path that stores
    the gate and up sums instead (separate_act), the stored rows are SiLU of
    those sums, and the output matches the oracle."""
    import moe_expert_layer_align_gb300 as moe
    wl = small(4, T, **kw)
    shape = moe.layer_shape(wl.x, wl.w13q, wl.topk_ids, 0, torch.bfloat16)
    res = {}
    for sep in (False, True):
        opts = moe.make_opts(separate_act=sep)
        ws = torch.zeros(moe.moe_workspace_bytes(shape, opts), dtype=torch.uint8, device="cuda")
        out = run_layer(wl, workspace=ws, opts=opts)
        torch.cuda.synchronize()
        res[sep] = (out, moe.workspace_views(ws, shape, opts))
    (o1, v1), (o0, v0) = res[False], res[True]
    L = v1["layout"]
    assert (L.block_m, L.split_gateup, L.g_act_rows, v0["layout"].g_act_rows) == (128, 1, 1, 0)
    assert torch.equal(o1, o0)
    sid = v1["sorted_ids"].cpu().numpy()
    rows = np.flatnonzero(sid < wl.T * wl.k)
    for n in ("A", "As"):
        np.testing.assert_array_equal(v1[n].cpu().numpy()[rows], v0[n].cpu().numpy()[rows], n)
    I = wl.I
    G = v0["G"][0].double().cpu().numpy()[rows]
    ref = G[:, :I] / (1 + np.exp(-G[:, :I])) * G[:, I:]
    got = v1["Gact"].double().cpu().numpy()[rows]
    np.testing.assert_allclose(got, ref, rtol=1e-5, atol=1e-6 * np.abs(ref).max())
    assert_layer_close(o1.float().cpu().numpy(), oracle_layer(wl), "fp8", "SiLU rows")


@pytest.mark.parametrize("smem_index", [False, True])
def test_invalid_ids_contribute_zero_and_are_flagged(smem_index):
    import moe_expert_layer_align_gb300 as moe
    wl = small(3, 30, H=256, I=128, E=16)
    ids = wl.topk_ids.clone()
    ids[2, 1] = -3
    ids[7, 0] = 99
    st = torch.full((1,), 12345, dtype=torch.int32, device="cuda")   # cleared by the call
    got = run_layer(wl, topk_ids=ids, dev_status=st,
                    opts=moe.make_opts(smem_index=smem_index)).float().cpu().numpy()
    torch.cuda.synchronize()
    assert st.item() == (1 << 6)
    ref = oracle_layer(wl, topk_ids=ids.cpu())
    assert_layer_close(got, ref, "bf16", "invalid ids")


def test_all_tokens_on_one_expert_and_identical_calls_are_bitwise_equal():
    wl = small(3, 200, H=256, I=192, E=16)
    ids = torch.zeros_like(wl.topk_ids)
    ids[:, 1:] = torch.arange(1, wl.k, device="cuda", dtype=torch.int32)
    a = run_layer(wl, topk_ids=ids)
    b = run_layer(wl, topk_ids=ids)
    torch.cuda.synchronize()
    assert torch.equal(a, b)          # deterministic: no float atomics anywhere
    assert_layer_close(a.float().cpu().numpy(), oracle_layer(wl, topk_ids=ids.cpu()), "bf16")


@pytest.mark.parametrize("H,k,bf16", [(384, 3, False), (388, 5, False), (388, 5, True),
                                      (4, 9, True), (2060, 2, False)])
def test_combine_alone(H, k, bf16):
    """The standalone combine, with row widths that end in a 4-column tail
    (H % 8 == 4) and odd token rows whose bf16 output is only 8-byte aligned."""
    import moe_expert_layer_align_gb300 as moe
    g = torch.Generator().manual_seed(3)
    T, S, rows = 9, 2, 96
    Y = torch.randn(S, rows, H, generator=g).cuda()
    inv = torch.randperm(rows, generator=g)[: T * k].int().cuda()
    inv[4] = -1
    w = torch.rand(T, k, generator=g).cuda()
    out = moe.moe_combine(Y, inv, w, T, H, k, S, rows,
                          out_dtype=torch.bfloat16 if bf16 else torch.float32)
    torch.cuda.synchronize()
    Ys = Y.double().sum(0).cpu().numpy()
    ref = np.zeros((T, H))
    for t in range(T):
        for j in range(k):
            p = inv[t * k + j].item()
            if p >= 0:
                ref[t] += w[t, j].item() * Ys[p]
    tol = 1e-2 if bf16 else 1e-5
    np.testing.assert_allclose(out.float().cpu().numpy(), ref, rtol=tol, atol=tol)


@pytest.mark.parametrize("bm", [128, 256])
@pytest.mark.parametrize("single", [False, True])
def test_two_weight_tiles_per_unit(bm, single):
    # large token tiles pair two 128-row weight tiles per GEMM unit (bf16)
    import moe_expert_layer_align_gb300 as moe
    wl = small(2, 300, H=512, I=256, E=4)
    opts = moe.make_opts(single_weight_tile=single)
    shape = moe.layer_shape(wl.x, wl.w13, wl.topk_ids, bm, torch.bfloat16)
    L = moe.moe_plan(shape, opts)
    assert L.weight_tiles_per_unit == (0x101 if single else 0x202)
    got = run_layer(wl, block_m=bm, opts=opts).float().cpu().numpy()
    assert_layer_close(got, oracle_layer(wl), "bf16", f"bm={bm} single={single}")


@pytest.mark.parametrize("zipf", [None, 1.2])
def test_index_over_chunks_is_bitwise_the_single_block_index(zipf):
    # Above a few thousand assignments the index is built by several CTAs over
    # chunks of the flat assignment list (the last one ragged); the rows must
    # still list each expert's assignments in ascending order, exactly as the
    # oracle's counting sort does, and invalid ids must still be flagged.
    import moe_expert_layer_align_gb300 as moe
    wl = small(3, 700, H=256, I=128, E=64)
    ids = wl.topk_ids.clone()
    if zipf is not None:
        g = torch.Generator().manual_seed(11)
        p = 1.0 / torch.arange(1, 65, dtype=torch.float64) ** zipf
        draw = torch.multinomial(p.expand(700, 64), wl.k, replacement=False, generator=g)
        ids = draw.int().cuda()
    ids[5, 3] = -1
    ids[690, 7] = 64
    shape = moe.layer_shape(wl.x, wl.w13, ids, 0, torch.bfloat16)
    L = moe.moe_plan(shape)
    assert wl.T * wl.k > 2048 and L.off_xq > L.off_index_scratch   # chunked build planned
    ws = torch.zeros(moe.moe_workspace_bytes(shape), dtype=torch.uint8, device="cuda")
    st = torch.full((1,), 777, dtype=torch.int32, device="cuda")
    got = run_layer(wl, topk_ids=ids, workspace=ws, dev_status=st).float().cpu().numpy()
    torch.cuda.synchronize()
    assert st.item() == (1 << 6)
    v = moe.workspace_views(ws, shape)
    ref = oracle.align(ids.cpu().numpy(), wl.E, L.block_m)
    for n in ("counts", "offsets", "sorted_ids", "tile_expert", "tiles", "inv_pos", "num_tiles"):
        np.testing.assert_array_equal(v[n].cpu().numpy().reshape(-1), ref[n].reshape(-1), n)
    assert_layer_close(got, oracle_layer(wl, topk_ids=ids.cpu()), "bf16", "chunked index")


@pytest.mark.parametrize("cfg,T,kw", [
    (3, 40, dict(H=256, I=128, E=512, k=8)),     # the largest expert count
    (2, 30, dict(H=256, I=128, E=8, k=8)),       # every token picks every expert
    (2, 17, dict(H=256, I=128, E=1, k=1)),       # one expert: a dense SwiGLU MLP
    (2, 33, dict(H=128, I=64, E=4, k=2)),        # the smallest H and I of the bf16 layer
    (4, 33, dict(H=128, I=128, E=4, k=2)),       # ... and of the FP8 layer
    (3, 5000, dict(H=128, I=64, E=4, k=2)),      # many tiles per expert, chunked index
])
def test_shape_limits(cfg, T, kw):
    wl = small(cfg, T, **kw)
    got = run_layer(wl).float().cpu().numpy()
    assert_layer_close(got, oracle_layer(wl), wl.mode, f"cfg{cfg} T={T} {kw}")


@pytest.mark.parametrize("cfg,T,bm,s2", [(2, 300, 64, 0), (2, 700, 128, 2), (4, 600, 128, 0),
                                         (4, 200, 16, 3), (3, 900, 32, 0)])
def test_unit_orders_are_bitwise_equal(cfg, T, bm, s2):
    """Both walks over the work units (weight-tile-major, token-tile-major)
    compute every output element in the same unit with the same arithmetic,
    so the layer outputs are bitwise equal, and equal to the oracle's within
    tolerance.  Several token tiles per expert, ragged tails, forced split."""
    import moe_expert_layer_align_gb300 as moe
    kw = dict(H=512, I=256, E=8) if cfg != 3 else dict(H=256, I=128, E=16)
    wl = small(cfg, T, **kw)
    outs = []
    for order in (1, 2):
        opts = moe.make_opts(split_down=s2, unit_order=order)
        outs.append(run_layer(wl, block_m=bm, opts=opts).float().cpu().numpy())
    np.testing.assert_array_equal(outs[0], outs[1])
    assert_layer_close(outs[1], oracle_layer(wl), wl.mode, f"cfg{cfg} T={T} bm={bm}")


@pytest.mark.parametrize("T,E,kw", [
    (300, 4, dict(H=512, I=256)),     # one 256-row tile per expert, its second half ragged
    (700, 3, dict(H=256, I=384)),     # a full 256-row tile and a ragged one per expert
    (100, 4, dict(H=384, I=128)),     # at most 128 valid rows: second half never computed
])
@pytest.mark.parametrize("split", [False, True])
def test_token_major_256_row_tiles(T, E, kw, split):
    """bf16 with 256-row token tiles and two weight tiles per unit: the
    token-major 256 x 256 tile (two M = 128 halves against one N = 256
    weight operand), fused SiLU-and-mul or, with a split Gate-Up, fp32
    partial rows."""
    import moe_expert_layer_align_gb300 as moe
    wl = small(2, T, E=E, **kw)
    opts = moe.make_opts(split_gateup=2, separate_act=True) if split else None
    shape = moe.layer_shape(wl.x, wl.w13, wl.topk_ids, 256, torch.bfloat16)
    L = moe.moe_plan(shape, opts)
    assert L.block_m == 256 and (L.weight_tiles_per_unit & 0xff) == 2
    got = run_layer(wl, block_m=256, opts=opts).float().cpu().numpy()
    assert_layer_close(got, oracle_layer(wl), "bf16", f"T={T} E={E} {kw} split={split}")
