"""moe_forward_static: the entry point for callers that cannot allocate device
memory (serving engines that reserve all device memory at start-up, plain-C
hosts without a device allocator).

It is called here through the C ABI directly.  Each checked call is preceded
by a static call on a different shape and different data, so the shared
scratch it starts from holds another call's leftovers; its output must then be
bitwise equal to the workspace-taking moe_forward's (the same plan runs the
same deterministic kernels), on two calls in a row, and within the layer
tolerances of the oracle.  This file is collected last so that a run stopping
at its first failure has already run every other test; it also passes alone
in a fresh process."""
import ctypes

import pytest
import torch

from moe_expert_layer_align_gb300 import workloads
from helpers import assert_layer_close, oracle_layer

pytestmark = pytest.mark.gpu


def static_call(wl, out, status):
    import moe_expert_layer_align_gb300 as moe
    from moe_expert_layer_align_gb300 import _binding as B
    fp8 = wl.mode == "fp8"
    w13, w2 = (wl.w13q, wl.w2q) if fp8 else (wl.w13, wl.w2)
    shape = moe.layer_shape(wl.x, w13, wl.topk_ids, 0, out.dtype)
    sc = B.moe_scales(wl.w13s.data_ptr(), wl.w2s.data_ptr()) if fp8 else None
    return B.lib.moe_forward_static(ctypes.byref(shape), wl.x.data_ptr(), w13.data_ptr(),
                                    w2.data_ptr(), wl.topk_ids.data_ptr(), wl.topk_w.data_ptr(),
                                    ctypes.byref(sc) if sc else None, out.data_ptr(),
                                    status.data_ptr(), torch.cuda.current_stream().cuda_stream)


def workspace_call(wl, out_dtype):
    import moe_expert_layer_align_gb300 as moe
    if wl.mode == "fp8":
        return moe.moe_forward(wl.x, wl.w13q, wl.w2q, wl.topk_ids, wl.topk_w,
                               scales=(wl.w13s, wl.w2s), out_dtype=out_dtype)
    return moe.moe_forward(wl.x, wl.w13, wl.w2, wl.topk_ids, wl.topk_w, out_dtype=out_dtype)


def run_static(wl):
    import moe_expert_layer_align_gb300 as moe
    out = torch.full(wl.x.shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    rc = static_call(wl, out, status)
    assert rc == moe.MOE_OK, moe.moe_status_str(rc)
    torch.cuda.synchronize()
    assert status.item() == 0, f"device status {status.item()}"
    return out


# Each case: the checked layer, then another layer (other shape, other data)
# run through the static entry point before every checked call.
CASES = [
    ((3, 40, dict(H=384, I=192, E=32)), (3, 300, dict(H=256, I=128, E=16))),
    ((4, 20, dict(H=512, I=256, E=16)), (4, 70, dict(H=384, I=384, E=12))),
]


@pytest.mark.parametrize("case,other", CASES)
def test_static_entry_equals_workspace_entry_after_other_calls(case, other):
    cfg, T, kw = case
    wl = workloads.make(cfg, T, "cpu", **kw).to("cuda")
    ocfg, oT, okw = other
    wl_other = workloads.make(ocfg, oT, "cpu", weight_seed=77, token_seed=78, **okw).to("cuda")
    ref = workspace_call(wl, torch.bfloat16)
    torch.cuda.synchronize()
    for call in range(2):
        run_static(wl_other)                      # leaves other contents in the scratch
        out = run_static(wl)
        assert torch.equal(out, ref), f"call {call}: differs from moe_forward"
        if call == 0:
            assert_layer_close(out.double().cpu().numpy(), oracle_layer(wl), wl.mode,
                               "static entry vs oracle")


def test_static_entry_rejects_shapes_beyond_its_scratch():
    import moe_expert_layer_align_gb300 as moe
    from moe_expert_layer_align_gb300 import _binding as B
    big = moe.make_shape(4096, 4096, 14336, 8, 2)          # needs ~1 GB of workspace
    assert moe.moe_workspace_bytes(big) > B.STATIC_SCRATCH_BYTES
    fake = [0x100000 * (i + 1) for i in range(7)]         # never dereferenced
    rc = B.lib.moe_forward_static(ctypes.byref(big), *fake[:5], None, fake[5], None, None)
    assert rc == moe.MOE_ERR_WORKSPACE
