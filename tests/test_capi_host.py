"""Host-side checks of the C ABI, no GPU needed: the library loads, exports
every symbol include/moe.h declares, the planner is self-consistent, and bad
arguments are rejected before anything is launched."""
import ctypes
import os
import re

import pytest

import moe_expert_layer_align_gb300 as moe
from moe_expert_layer_align_gb300 import _binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "moe.h")).read()
    return sorted(set(re.findall(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    names = declared_symbols()
    assert len(names) >= 11
    for n in names:
        assert hasattr(B.lib, n), n
        assert n in B.SYMBOLS, n


def test_status_strings():
    for s in range(9):
        assert moe.moe_status_str(s) and moe.moe_status_str(s) != "unknown status"
    assert moe.moe_status_str(99) == "unknown status"


@pytest.mark.parametrize("T,H,I,E,k,fp8", [
    (8, 256, 512, 8, 2, False), (64, 4096, 14336, 8, 2, False), (1, 2048, 768, 128, 8, False),
    (4096, 2048, 768, 128, 8, False), (64, 7168, 2048, 256, 8, True), (4096, 7168, 2048, 256, 8, True),
])
def test_plan_is_consistent(T, H, I, E, k, fp8):
    s = moe.make_shape(T, H, I, E, k, 0, fp8, True)
    L = moe.moe_plan(s)
    assert L.block_m in (16, 32, 64, 128, 256) and (not fp8 or L.block_m <= 128)
    assert L.tiles_cap == moe.moe_index_tiles_cap(T, k, E, L.block_m)
    assert L.tiles_cap == -(-T * k // L.block_m) + min(E, T * k)
    assert L.rows_cap == L.tiles_cap * L.block_m
    assert L.split_gateup >= 1 and L.split_down >= 1
    offs = [L.off_counts, L.off_offsets, L.off_sorted_ids, L.off_tile_expert, L.off_tiles,
            L.off_inv_pos, L.off_num_tiles, L.off_index_scratch, L.off_xq, L.off_xs, L.off_g, L.off_a, L.off_as,
            L.off_y]
    assert offs == sorted(offs) and all(o % 256 == 0 for o in offs)
    assert L.y_bf16 == (L.split_down == 1)   # an unsplit Down stores bf16 rows
    assert L.off_y + (2 if L.y_bf16 else 4 * L.split_down) * L.rows_cap * H <= L.total_bytes
    assert moe.moe_workspace_bytes(s) == L.total_bytes
    # forced splits are honoured and resize the workspace
    o = moe.make_opts(split_gateup=2, split_down=3)
    L2 = moe.moe_plan(s, o)
    assert L2.split_gateup == 2 and L2.split_down == 3


def test_rejects_bad_shapes_without_launching():
    bad = [
        moe.make_shape(0, 256, 512, 8, 2),      # T
        moe.make_shape(8, 200, 512, 8, 2),      # H % 128
        moe.make_shape(8, 256, 500, 8, 2),      # I % 64
        moe.make_shape(8, 256, 512, 8, 9),      # k > E
        moe.make_shape(8, 256, 512, 600, 2),    # E > 512
        moe.make_shape(8, 256, 576, 8, 2, 0, True),   # FP8 needs I % 128
        moe.make_shape(8, 256, 512, 8, 2, 24),  # block_m
        moe.make_shape(8, 256, 512, 8, 2, 256, True),  # FP8 block_m <= 128
    ]
    for s in bad:
        assert moe.moe_workspace_bytes(s) == 0
        with pytest.raises(moe.MoeError) as ei:
            moe.moe_plan(s)
        assert ei.value.status == moe.MOE_ERR_SHAPE
    s = moe.make_shape(8, 256, 512, 8, 2)
    s.mode = 7
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_plan(s)
    assert ei.value.status == moe.MOE_ERR_DTYPE


def _fwd(shape, ptrs, ws_bytes, scales=None):
    x, w13, w2, ids, w, out, ws = ptrs
    return B.lib.moe_forward(ctypes.byref(shape), x, w13, w2, ids, w,
                             ctypes.byref(scales) if scales else None, out, ws, ws_bytes, None,
                             None)


def test_forward_argument_errors_precede_any_launch():
    # Fake (never dereferenced) addresses: every call below must fail in the
    # host checks, before a CUDA call is made.
    s = moe.make_shape(8, 256, 512, 8, 2)
    need = moe.moe_workspace_bytes(s)
    good = [0x100000 * (i + 1) for i in range(7)]
    assert _fwd(s, [None] + good[1:], need) == moe.MOE_ERR_ARG
    assert _fwd(s, good[:6] + [None], need) == moe.MOE_ERR_ARG
    mis = list(good)
    mis[0] += 8
    assert _fwd(s, mis, need) == moe.MOE_ERR_ALIGN
    mis = list(good)
    mis[6] += 128
    assert _fwd(s, mis, need) == moe.MOE_ERR_ALIGN
    assert _fwd(s, good, need - 1) == moe.MOE_ERR_WORKSPACE
    f = moe.make_shape(8, 256, 512, 8, 2, 0, True)
    assert _fwd(f, good, moe.moe_workspace_bytes(f)) == moe.MOE_ERR_ARG   # FP8 without scales
    assert B.lib.moe_align(None, 8, 2, 8, 16, None, None, None) == moe.MOE_ERR_ARG
    idx = B.moe_index(*good)
    assert B.lib.moe_align(good[0], 8, 2, 8, 24, ctypes.byref(idx), None, None) == moe.MOE_ERR_SHAPE
    idx.tiles = good[4] + 4
    assert B.lib.moe_align(good[0], 8, 2, 8, 16, ctypes.byref(idx), None, None) == moe.MOE_ERR_ALIGN


def test_router_host_checks():
    assert moe.moe_router_workspace_bytes(64, 2048, 128) > 0
    assert moe.moe_router_workspace_bytes(64, 2000, 128) == 0
    assert moe.moe_router_workspace_bytes(64, 2048, 100) == 0
    g = [0x100000 * (i + 1) for i in range(7)]
    assert B.lib.moe_router_topk(g[0], g[1], 64, 2048, 128, 33, 0, 1.0, g[2], g[3], g[4], g[5],
                                 1 << 30, None) == moe.MOE_ERR_SHAPE
    assert B.lib.moe_router_topk(g[0], g[1], 64, 2048, 128, 8, 5, 1.0, g[2], g[3], g[4], g[5],
                                 1 << 30, None) == moe.MOE_ERR_ARG
    assert B.lib.moe_router_topk(g[0], g[1], 64, 2048, 128, 8, 0, 1.0, g[2], g[3], g[4], g[5],
                                 16, None) == moe.MOE_ERR_WORKSPACE


def test_shared_expert_and_ep_options_are_checked_and_planned():
    s = moe.make_shape(64, 2048, 768, 128, 8)
    L0 = moe.moe_plan(s)
    L = moe.moe_plan(s, moe.make_opts(num_shared_experts=1))
    assert L.tiles_cap == moe.moe_index_tiles_cap(64, 9, 129, L.block_m)
    assert L.total_bytes >= L0.total_bytes
    Le = moe.moe_plan(moe.make_shape(64, 2048, 768, 32, 8), moe.make_opts(ep_first_expert=32,
                                                                          ep_num_experts=128))
    assert Le.tiles_cap == moe.moe_index_tiles_cap(64, 8, 32, Le.block_m)
    bad = [moe.make_opts(num_shared_experts=9), moe.make_opts(num_shared_experts=-1),
           moe.make_opts(ep_first_expert=100, ep_num_experts=128),     # 100 + 128 > 128
           moe.make_opts(ep_first_expert=3)]                           # a range without EP
    for o in bad:
        assert moe.moe_workspace_bytes(s, o) == 0
        with pytest.raises(moe.MoeError) as ei:
            moe.moe_plan(s, o)
        assert ei.value.status == moe.MOE_ERR_SHAPE


def test_align_ex_host_checks():
    g = [0x100000 * (i + 1) for i in range(7)]
    idx = B.moe_index(*g)
    o = B.moe_align_opts(1, 0, 0)
    # mapped ids are staged on chip: at most 32768 assignments
    assert B.lib.moe_align_ex(g[0], 8192, 4, 8, 16, ctypes.byref(o), ctypes.byref(idx), None,
                              None) == moe.MOE_ERR_SHAPE
    o = B.moe_align_opts(0, 6, 8)                                    # 6 + 8 > 8
    assert B.lib.moe_align_ex(g[0], 8, 2, 8, 16, ctypes.byref(o), ctypes.byref(idx), None,
                              None) == moe.MOE_ERR_SHAPE
    assert B.lib.moe_align_ex(None, 8, 2, 8, 16, ctypes.byref(o), ctypes.byref(idx), None,
                              None) == moe.MOE_ERR_ARG


def test_routed_plan():
    s = moe.make_shape(64, 2048, 768, 128, 8, 0, True)
    assert moe.moe_plan_routed(s).route_fused == 0          # separate kernels by default
    L = moe.moe_plan_routed(s, moe.make_opts(fuse_routing=True))
    assert L.route_fused == 1 and L.off_router >= L.off_y and L.off_route_counter > L.off_router
    assert L.off_route_hist > L.off_route_counter
    assert L.off_route_hist + 4 * 11 * 128 <= L.total_bytes   # a histogram row per owner CTA (6 tokens each)
    assert moe.moe_routed_workspace_bytes(s, moe.make_opts(fuse_routing=True)) == L.total_bytes
    assert L.total_bytes > moe.moe_workspace_bytes(s)
    L2 = moe.moe_plan_routed(s, moe.make_opts(fuse_routing=False))
    assert L2.route_fused == 0 and L2.total_bytes > moe.moe_workspace_bytes(s)
    # separate kernels: the router GEMM may split further (a block of warps per
    # token sums the partials), the fused front keeps at most four splits
    assert L2.off_route_counter - L2.off_router >= L.off_route_counter - L.off_router
    assert moe.moe_plan_routed(moe.make_shape(4096, 2048, 768, 128, 8, 0, True),
                               moe.make_opts(fuse_routing=True)).route_fused == 1
    o = moe.make_opts()
    o.fuse_routing = 2
    with pytest.raises(moe.MoeError):
        moe.moe_plan_routed(s, o)
    for o in (moe.make_opts(smem_index=True), moe.make_opts(num_shared_experts=1),
              moe.make_opts(ep_first_expert=0, ep_num_experts=256)):
        with pytest.raises(moe.MoeError):
            moe.moe_plan_routed(s, o)
    with pytest.raises(moe.MoeError):           # router E must be a multiple of 64
        moe.moe_plan_routed(moe.make_shape(64, 2048, 768, 100, 8))


def test_split_counts_of_the_measured_decode_shapes():
    """The planner's split-K counts where they were measured against the
    alternatives: the Mixtral-shaped Down 4 ways at T=16..128 and 7 at T=4,
    the Qwen3-shaped Down unsplit at T=1..64 (bf16 units carry a fixed
    per-unit cost), the DeepSeek-shaped FP8 Gate-Up split 4 / 3 / 2 ways at
    T=1 / 4 / 16 (FP8 units do not)."""
    def splits(T, H, I, E, k, fp8):
        L = moe.moe_plan(moe.make_shape(T, H, I, E, k, 0, fp8))
        return L.split_gateup, L.split_down
    for T in (16, 32, 64, 128):
        assert splits(T, 4096, 14336, 8, 2, False) == (1, 4), T
    assert splits(4, 4096, 14336, 8, 2, False) == (1, 7)
    for T in (1, 4, 8, 64):
        assert splits(T, 2048, 768, 128, 8, False) == (1, 1), T
    for T, s1 in ((1, 4), (4, 3), (16, 2), (64, 1)):
        assert splits(T, 7168, 2048, 256, 8, True) == (s1, 1), T


def test_static_scratch_covers_the_documented_token_counts():
    """The header's statement of what MOE_STATIC_SCRATCH_BYTES covers with the
    current plans: every T up to 768 / 912 / 20 for the Mixtral-, Qwen3- and
    DeepSeek-shaped layers, and not the next token count."""
    lim = B.STATIC_SCRATCH_BYTES
    for (H, I, E, k, fp8), tmax in (((4096, 14336, 8, 2, False), 768),
                                    ((2048, 768, 128, 8, False), 912),
                                    ((7168, 2048, 256, 8, True), 20)):
        sizes = [moe.moe_workspace_bytes(moe.make_shape(T, H, I, E, k, 0, fp8))
                 for T in range(1, tmax + 2)]
        assert max(sizes[:-1]) <= lim < sizes[-1], (H, tmax)


def test_fp8_quant_on_index_launch_plan():
    """FP8 layers with a one-CTA index quantise x on the index launch (scales
    per token, no per-row copy); the chunked index, separate_quant, the
    shared-memory index and bf16 layers keep what they had."""
    ds = moe.make_shape(64, 7168, 2048, 256, 8, 0, True)
    L = moe.moe_plan(ds)
    assert L.xs_by_token == 1
    sep = moe.make_opts(separate_quant=True)
    assert moe.moe_plan(ds, sep).xs_by_token == 0
    rows = 4 * L.rows_cap * (7168 // 128)                 # the per-row scales it no longer needs
    assert abs(moe.moe_workspace_bytes(ds, sep) - moe.moe_workspace_bytes(ds) - rows) < 256
    big = moe.make_shape(4096, 7168, 2048, 256, 8, 0, True)   # 32768 assignments: chunked index
    assert moe.moe_plan(big).xs_by_token == 0
    assert moe.moe_plan(ds, moe.make_opts(smem_index=True)).xs_by_token == 1
    assert moe.moe_plan(moe.make_shape(64, 2048, 768, 128, 8, 0)).xs_by_token == 0


def test_fp8_silu_rows_plan():
    """FP8 layers whose Gate-Up runs unsplit on 128-row token tiles store
    SiLU(gate)*up (I fp32 values a row) instead of the gate and up sums (2I);
    separate_act, forced splits, decode tiles and bf16 layers keep the sums."""
    ds = moe.make_shape(4096, 7168, 2048, 256, 8, 0, True)
    L = moe.moe_plan(ds)
    assert (L.block_m, L.split_gateup, L.g_act_rows, L.fused_act) == (128, 1, 1, 0)
    assert L.off_a - L.off_g >= 4 * L.rows_cap * 2048
    sep = moe.make_opts(separate_act=True)
    assert moe.moe_plan(ds, sep).g_act_rows == 0
    grow = moe.moe_workspace_bytes(ds, sep) - moe.moe_workspace_bytes(ds)
    assert abs(grow - 4 * L.rows_cap * 2048) < 256            # the half of G it no longer needs
    assert moe.moe_plan(ds, moe.make_opts(split_gateup=2)).g_act_rows == 0
    assert moe.moe_plan(moe.make_shape(64, 7168, 2048, 256, 8, 0, True)).g_act_rows == 0
    assert moe.moe_plan(moe.make_shape(4096, 2048, 768, 128, 8, 0)).g_act_rows == 0
    w8 = moe.make_shape(4096, 7168, 2048, 256, 8, 0, mode=moe.MOE_W8A16)
    assert moe.moe_plan(w8).g_act_rows == 0


def test_router_plan_keeps_split_k_at_large_token_tiles():
    """The expert GEMMs run 128-row token tiles unsplit; the router GEMM, whose
    output is fp32 partials either way and whose 2E/128 weight tiles alone
    would leave most SMs idle, keeps splitting K (router table shape: K = 4096,
    192 experts)."""
    for T in (96, 512, 2048):
        rows_cap = -(-T // 128) * 128
        one_split = 4 * rows_cap * 2 * 192
        assert moe.moe_router_workspace_bytes(T, 4096, 192) >= 3 * one_split, T


def test_unit_order_plan():
    """Token-tile-major where an expert's token tiles x units per tile fit one
    wave of CTAs; weight-tile-major for the Mixtral-shaped prefill Gate-Up
    (four token tiles per expert, 112 units each); forced orders are kept;
    anything else is rejected."""
    mix = moe.make_shape(2048, 4096, 14336, 8, 2, 0)
    L = moe.moe_plan(mix)
    assert (L.unit_order & 255, L.unit_order >> 8) == (1, 2)
    qwen = moe.make_shape(4096, 2048, 768, 128, 8, 0)
    assert moe.moe_plan(qwen).unit_order == 2 | (2 << 8)
    ds = moe.make_shape(4096, 7168, 2048, 256, 8, 0, True)
    assert moe.moe_plan(ds).unit_order == 2 | (2 << 8)
    for order in (1, 2):
        assert moe.moe_plan(mix, moe.make_opts(unit_order=order)).unit_order == order | (order << 8)
    for bad in (-1, 3):
        with pytest.raises(moe.MoeError):
            moe.moe_plan(mix, moe.make_opts(unit_order=bad))


def test_smem_index_plan():
    """The in-GEMM index is the default for bf16 layers with at most 16
    experts (where it fits), never for FP8 or larger expert counts; it can be
    forced on or off; other values are rejected."""
    tiny = moe.make_shape(8, 256, 512, 8, 2, 0)
    assert moe.moe_plan(tiny).smem_index == 1
    assert moe.moe_plan(tiny, moe.make_opts(smem_index=False)).smem_index == 0
    assert moe.moe_plan(moe.make_shape(1, 2048, 768, 128, 8, 0)).smem_index == 0
    assert moe.moe_plan(moe.make_shape(1, 2048, 768, 128, 8, 0),
                        moe.make_opts(smem_index=True)).smem_index == 1
    assert moe.moe_plan(moe.make_shape(8, 256, 512, 8, 2, 0, True)).smem_index == 0
    assert moe.moe_plan(moe.make_shape(2048, 4096, 14336, 8, 2, 0)).smem_index == 0   # T*k > 4096
    o = moe.make_opts()
    o.smem_index = 2
    with pytest.raises(moe.MoeError):
        moe.moe_plan(tiny, o)


def test_fp8_row_tile_rule():
    """FP8 takes 128-row (token-major) tiles where the mean-rows rule gives
    64; bf16 keeps 64 there; w8a16 follows the bf16 rule."""
    # DeepSeek-shaped at T=1024: 32 rows per active expert -> 64 by the rule
    assert moe.moe_plan(moe.make_shape(1024, 7168, 2048, 256, 8, 0, True)).block_m == 128
    assert moe.moe_plan(moe.make_shape(1024, 7168, 2048, 256, 8, 0)).block_m == 64
    assert moe.moe_plan(moe.make_shape(1024, 7168, 2048, 256, 8, 0,
                                       mode=B.MOE_W8A16)).block_m == 64
    # decode sizes keep their narrow tiles
    assert moe.moe_plan(moe.make_shape(64, 7168, 2048, 256, 8, 0, True)).block_m == 16
    assert moe.moe_plan(moe.make_shape(512, 7168, 2048, 256, 8, 0, True)).block_m == 32


def test_wait_limit_option_changes_no_plan_and_rejects_negatives():
    s = moe.make_shape(8, 256, 512, 8, 2)
    assert moe.moe_workspace_bytes(s, moe.make_opts(pipeline_wait_ns=1)) == moe.moe_workspace_bytes(s)
    with pytest.raises(moe.MoeError):
        moe.moe_plan(s, moe.make_opts(pipeline_wait_ns=-5))


@pytest.mark.parametrize("T,H,I,E,k,fp8,bm", [
    (64, 2048, 768, 128, 8, True, 0), (256, 2048, 768, 128, 8, True, 0),
    (64, 2048, 768, 128, 8, False, 0), (8, 256, 512, 8, 2, False, 16),
])
def test_coalesce_option_plan(T, H, I, E, k, fp8, bm):
    s = moe.make_shape(T, H, I, E, k, bm, fp8, True)
    base = moe.moe_plan(s, moe.make_opts(coalesce_rows=-1))
    assert base.coalesce_rows == 0 and base.work_cap == 0
    assert base.off_work_tiles == base.off_num_work_tiles
    for c in (32, 64):
        L = moe.moe_plan(s, moe.make_opts(coalesce_rows=c))
        # the index is the same (block_m, caps); the work list is used where C > block_m
        assert (L.block_m, L.tiles_cap, L.rows_cap) == (base.block_m, base.tiles_cap, base.rows_cap)
        assert L.coalesce_rows == (c if c > L.block_m else 0)
        if L.coalesce_rows:
            assert L.work_cap == L.tiles_cap        # tiles larger than the index's: no more of them
            assert L.off_work_tiles >= L.off_route_hist
            assert L.off_work_tiles + 16 * L.work_cap <= L.off_num_work_tiles
            assert L.off_num_work_tiles + 4 <= L.total_bytes
            assert L.total_bytes > base.total_bytes
    for bad in (-2, 16, 48, 128):
        with pytest.raises(moe.MoeError) as ei:
            moe.moe_plan(s, moe.make_opts(coalesce_rows=bad))
        assert ei.value.status == moe.MOE_ERR_ARG
    # w8a16 keeps the task map
    if fp8:
        sw = moe.make_shape(T, H, I, E, k, bm, False, True)
        sw.mode = moe.MOE_W8A16
        assert moe.moe_plan(sw, moe.make_opts(coalesce_rows=64)).coalesce_rows == 0


def test_down_tile_rows_option_plan():
    # Qwen3-shaped T=4096: 256 rows per expert, 256-row token tiles
    s = moe.make_shape(4096, 2048, 768, 128, 8, 0, False, True)
    L0 = moe.moe_plan(s, moe.make_opts(down_tile_rows=-1))
    assert L0.block_m == 256 and L0.down_tile_rows == 0 and L0.work_cap == 0
    L = moe.moe_plan(s, moe.make_opts(down_tile_rows=128))
    assert L.block_m == 256 and L.down_tile_rows == 128 and L.coalesce_rows == 0
    # 128-row tiles of an index padded to 256: up to ceil(T*k/128) + E of them
    assert L.work_cap == moe.moe_index_tiles_cap(4096, 8, 128, 128) > L.tiles_cap
    assert L.off_work_tiles + 16 * L.work_cap <= L.off_num_work_tiles < L.total_bytes
    # the planner's choice: 128-row Down tiles from 256 rows per active expert
    assert moe.moe_plan(s).down_tile_rows == 128                        # 256 rows
    assert moe.moe_plan(moe.make_shape(2048, 4096, 14336, 8, 2, 0)).down_tile_rows == 128  # 512
    assert moe.moe_plan(moe.make_shape(2048, 2048, 768, 128, 8, 0)).down_tile_rows == 0   # 128
    assert moe.moe_plan(moe.make_shape(512, 4096, 14336, 8, 2, 0)).down_tile_rows == 0    # 128
    # no effect where the index tiles are not 256 rows
    s2 = moe.make_shape(64, 2048, 768, 128, 8, 0, False, True)
    assert moe.moe_plan(s2, moe.make_opts(down_tile_rows=128)).down_tile_rows == 0
    for bad in (-2, 64, 256):
        with pytest.raises(moe.MoeError) as ei:
            moe.moe_plan(s, moe.make_opts(down_tile_rows=bad))
        assert ei.value.status == moe.MOE_ERR_ARG
