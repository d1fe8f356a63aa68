"""The w8a16 layer (e4m3 weights with fp32 128x128 block scales, bf16
activations) through the C ABI against the oracle's exact dequantisation:
small cases over every row tile, split-K with the separate activation
stage, the chunked index, and the DeepSeek-V3-shaped weights at full size on
sampled tokens.  The kernel rounds each dequantised weight to bf16, inside
the bf16 tolerance."""
import numpy as np
import pytest
import torch

from moe_expert_layer_align_gb300 import workloads
from helpers import assert_layer_close, oracle_layer, oracle_layer_sampled

pytestmark = pytest.mark.gpu


def run(wl, block_m=0, opts=None, workspace=None):
    import moe_expert_layer_align_gb300 as moe
    st = torch.full((1,), 3, dtype=torch.int32, device="cuda")
    out = moe.moe_forward(wl.x, wl.w13q, wl.w2q, wl.topk_ids, wl.topk_w,
                          scales=(wl.w13s, wl.w2s), out_dtype=torch.bfloat16, block_m=block_m,
                          dev_status=st, opts=opts, workspace=workspace, w8a16=True)
    torch.cuda.synchronize()
    assert st.item() == 0
    return out.float().cpu().numpy()


@pytest.mark.parametrize("T,kw", [(1, dict(H=256, I=256, E=8, k=2)),
                                  (37, dict(H=512, I=256, E=6, k=3)),
                                  (150, dict(H=256, I=384, E=12, k=4))])
@pytest.mark.parametrize("bm", [0, 16, 32, 64, 128])
def test_w8a16_matches_oracle(T, kw, bm):
    wl = workloads.make(4, T, "cpu", **kw).to("cuda")
    assert_layer_close(run(wl, bm), oracle_layer(wl, w8a16=True), "bf16", f"T={T} bm={bm}")


@pytest.mark.parametrize("s1,s2", [(2, 1), (1, 3), (3, 2)])
def test_w8a16_split_k(s1, s2):
    import moe_expert_layer_align_gb300 as moe
    wl = workloads.make(4, 24, "cpu", H=1024, I=512, E=8, k=2).to("cuda")
    got = run(wl, opts=moe.make_opts(split_gateup=s1, split_down=s2))
    assert_layer_close(got, oracle_layer(wl, w8a16=True), "bf16", f"splits {s1},{s2}")


def test_w8a16_chunked_index_and_determinism():
    wl = workloads.make(4, 600, "cpu", H=256, I=256, E=16, k=4).to("cuda")   # 2400 assignments
    a = run(wl)
    b = run(wl)
    assert np.array_equal(a, b)
    assert_layer_close(a, oracle_layer(wl, w8a16=True), "bf16", "chunked")


@pytest.mark.parametrize("T,n", [(1, 1), (64, 4)])
def test_w8a16_deepseek_shape_full_size(T, n):
    wl = workloads.make(4, T, "cuda")
    got = run(wl)
    sel = np.unique(np.linspace(0, T - 1, n).astype(np.int64))
    want = oracle_layer_sampled(wl, wl.topk_ids.cpu().numpy(), wl.topk_w.cpu().numpy(), sel,
                                w8a16=True)
    assert_layer_close(got[sel], want, "bf16", f"DeepSeek-shaped w8a16 T={T}")
