"""moe_forward_static: the entry point for callers that cannot allocate device
memory (code running under global-mode CUDA-graph capture, engines that
reserve all device memory at start-up, plain-C hosts without an allocator).

It is called here through the C ABI directly and must give the output of the
workspace-taking moe_forward, within the layer tolerances, on two calls in a
row (the second call reuses the static scratch the first one left behind).
This file is collected last so that a run stopping at its first failure has
already run every other test; it also passes alone in a fresh process."""
import ctypes

import numpy as np
import pytest
import torch

from moe_expert_layer_align_gb300 import workloads
from helpers import assert_layer_close

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


def reference_call(wl, out_dtype):
    import moe_expert_layer_align_gb300 as moe
    if wl.mode == "fp8":
        return moe.moe_forward(wl.x, wl.w13q, wl.w2q, wl.topk_ids, wl.topk_w,
                               scales=(wl.w13s, wl.w2s), out_dtype=out_dtype)
    return moe.moe_forward(wl.x, wl.w13, wl.w2, wl.topk_ids, wl.topk_w, out_dtype=out_dtype)


@pytest.mark.parametrize("cfg,T,kw", [
    (3, 40, dict(H=384, I=192, E=32)),
    (4, 20, dict(H=512, I=256, E=16)),
])
def test_static_entry_matches_workspace_entry_twice(cfg, T, kw):
    import moe_expert_layer_align_gb300 as moe
    wl = workloads.make(cfg, T, "cpu", **kw).to("cuda")
    ref = reference_call(wl, torch.bfloat16)
    torch.cuda.synchronize()
    for call in range(2):
        out = torch.full(wl.x.shape, float("nan"), dtype=torch.bfloat16, device="cuda")
        status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        rc = static_call(wl, out, status)
        assert rc == moe.MOE_OK, moe.moe_status_str(rc)
        torch.cuda.synchronize()
        assert status.item() == 0, f"call {call}: device status {status.item()}"
        assert_layer_close(out.double().cpu().numpy(), ref.double().cpu().numpy(), wl.mode,
                           f"static entry, call {call}")


def test_static_entry_rejects_shapes_beyond_its_scratch():
    import moe_expert_layer_align_gb300 as moe
    from moe_expert_layer_align_gb300 import _binding as B
    big = moe.make_shape(4096, 4096, 14336, 8, 2)          # needs ~1 GB of workspace
    assert moe.moe_workspace_bytes(big) > B.STATIC_SCRATCH_BYTES
    fake = [0x100000 * (i + 1) for i in range(7)]         # never dereferenced
    rc = B.lib.moe_forward_static(ctypes.byref(big), *fake[:5], None, fake[5], None, None)
    assert rc == moe.MOE_ERR_WORKSPACE
