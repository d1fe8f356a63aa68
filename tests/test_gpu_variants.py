"""The two routing variants through the C ABI against the oracle: shared
experts fused as extra experts of the grouped GEMM, and the expert-parallel
local part (a rank holding a range of the experts).  Index bit-exact, outputs
within the layer tolerances, dev_status flags as specified."""
import numpy as np
import pytest
import torch

import oracle
from moe_expert_layer_align_gb300 import workloads
from helpers import assert_layer_close, bits16, u8

pytestmark = pytest.mark.gpu

INDEX_FIELDS = ("counts", "offsets", "sorted_ids", "tile_expert", "tiles", "inv_pos", "num_tiles")


def routed(T, E, k, seed):
    """top-k ids over E routed experts and positive weights (seeded)."""
    g = torch.Generator().manual_seed(seed)
    ids = torch.stack([torch.randperm(E, generator=g)[:k] for _ in range(T)]).int()
    w = torch.rand(T, k, generator=g) + 0.1
    return ids, w / w.sum(1, keepdim=True)


def weights(wl, lo=None, hi=None):
    """(w13, w2, scales) of the workload, optionally experts [lo, hi) only."""
    s = slice(lo, hi)
    if wl.mode == "bf16":
        return wl.w13[s].contiguous(), wl.w2[s].contiguous(), None
    return (wl.w13q[s].contiguous(), wl.w2q[s].contiguous(),
            (wl.w13s[s].contiguous(), wl.w2s[s].contiguous()))


def oracle_out(wl, ids, w, lo=None, hi=None):
    x = bits16(wl.x)
    s = slice(lo, hi)
    if wl.mode == "bf16":
        return oracle.moe_bf16(x, bits16(wl.w13[s]), bits16(wl.w2[s]), ids, w)
    xq, xs = oracle.quant_x(x)
    return oracle.moe_fp8(xq, xs, u8(wl.w13q[s]), wl.w13s[s].cpu().numpy(), u8(wl.w2q[s]),
                          wl.w2s[s].cpu().numpy(), ids, w)


def run(wl, ids, w, opts, lo=None, hi=None, block_m=0):
    import moe_expert_layer_align_gb300 as moe
    w13, w2, sc = weights(wl, lo, hi)
    out_dtype = torch.float32 if wl.out == "f32" else torch.bfloat16
    shape = moe.layer_shape(wl.x, w13, ids, block_m, out_dtype, opts.num_shared_experts)
    ws = torch.zeros(moe.moe_workspace_bytes(shape, opts), dtype=torch.uint8, device="cuda")
    st = torch.full((1,), 99, dtype=torch.int32, device="cuda")
    out = moe.moe_forward(wl.x, w13, w2, ids, w, scales=sc, out_dtype=out_dtype, workspace=ws,
                          block_m=block_m, dev_status=st, opts=opts)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), moe.workspace_views(ws, shape, opts), int(st.item())


def check_index(views, ids_mapped, E_index):
    ref = oracle.align(ids_mapped, E_index, views["layout"].block_m)
    for n in INDEX_FIELDS:
        np.testing.assert_array_equal(views[n].cpu().numpy().reshape(-1), ref[n].reshape(-1), n)


# (workload, T, shape overrides): bf16 and FP8, small and chunked-index sizes
CASES = [
    (3, 40, dict(H=256, I=128)),
    (4, 24, dict(H=256, I=256)),
    (3, 700, dict(H=256, I=128)),     # T*(k+n) > 2048: the chunked index build
]


@pytest.mark.parametrize("n_shared,weight", [(1, 0.0), (2, 0.5)])
@pytest.mark.parametrize("cfg,T,kw", CASES)
def test_shared_experts(cfg, T, kw, n_shared, weight):
    import moe_expert_layer_align_gb300 as moe
    E, k = 12, 4
    wl = workloads.make(cfg, T, "cpu", E=E + n_shared, k=k, **kw).to("cuda")
    ids, w = routed(T, E, k, 100 + T)
    opts = moe.make_opts(num_shared_experts=n_shared, shared_expert_weight=weight)
    got, views, st = run(wl, ids.cuda(), w.cuda(), opts)
    assert st == 0
    sid, sw = oracle.shared_routing(ids.numpy(), w.numpy(), E, n_shared, weight or 1.0)
    check_index(views, sid, E + n_shared)
    assert_layer_close(got, oracle_out(wl, sid, sw), wl.mode, f"shared x{n_shared}")


@pytest.mark.parametrize("cfg,T,kw", CASES)
def test_expert_parallel_parts(cfg, T, kw):
    import moe_expert_layer_align_gb300 as moe
    Eg, k = 12, 4
    wl = workloads.make(cfg, T, "cpu", E=Eg, k=k, **kw).to("cuda")
    ids, w = routed(T, Eg, k, 200 + T)
    total = 0
    for lo, hi in ((0, 5), (5, 12)):
        opts = moe.make_opts(ep_first_expert=lo, ep_num_experts=Eg)
        got, views, st = run(wl, ids.cuda(), w.cuda(), opts, lo, hi)
        assert st == 0                      # other ranks' experts are not errors
        loc = oracle.ep_local_ids(ids.numpy(), lo, hi - lo)
        check_index(views, loc, hi - lo)
        assert_layer_close(got, oracle_out(wl, loc, w.numpy(), lo, hi), wl.mode, f"rank {lo}")
        total = total + got
    # the ranks' partial sums add up to the whole layer
    assert_layer_close(total, oracle_out(wl, ids.numpy(), w.numpy()), wl.mode, "sum of ranks")


def test_expert_parallel_flags_only_invalid_ids():
    import moe_expert_layer_align_gb300 as moe
    Eg, k, T = 10, 3, 30
    wl = workloads.make(3, T, "cpu", H=256, I=128, E=Eg, k=k).to("cuda")
    ids, w = routed(T, Eg, k, 7)
    ids[3, 1] = Eg          # invalid globally
    ids[9, 0] = -4          # invalid
    opts = moe.make_opts(ep_first_expert=4, ep_num_experts=Eg)
    got, views, st = run(wl, ids.cuda(), w.cuda(), opts, 4, 8)
    assert st == (1 << 6)
    loc = oracle.ep_local_ids(ids.numpy(), 4, 4)
    check_index(views, loc, 4)
    assert_layer_close(got, oracle_out(wl, loc, w.numpy(), 4, 8), "bf16", "ep + invalid")


@pytest.mark.parametrize("n_shared,e0,Eg", [(1, 0, 0), (0, 3, 16), (2, 8, 16)])
def test_align_ex_matches_oracle(n_shared, e0, Eg):
    import moe_expert_layer_align_gb300 as moe
    T, k, E = 333, 4, 8
    ids, _ = routed(T, Eg or E, k, 11)
    st = torch.full((1,), 5, dtype=torch.int32, device="cuda")
    idx = moe.moe_align_ex(ids.cuda(), E, 32, num_shared_experts=n_shared, ep_first_expert=e0,
                           ep_num_experts=Eg, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    m = ids.numpy() if Eg == 0 else oracle.ep_local_ids(ids.numpy(), e0, E)
    if n_shared:
        m, _ = oracle.shared_routing(m, np.ones_like(m, np.float32), E, n_shared)
    ref = oracle.align(m, E + n_shared, 32)
    for n in INDEX_FIELDS:
        np.testing.assert_array_equal(idx[n].cpu().numpy().reshape(-1), ref[n].reshape(-1), n)
