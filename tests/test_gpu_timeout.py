"""The bounded-wait timeout path of the expert GEMMs, run on the GPU.

Every on-chip wait of the GEMM kernels is bounded; when one gives up, the
kernel flags MOE_ERR_TIMEOUT in dev_status, raises its CTA-wide abort flag so
that every role leaves its loop, lets its own copies and MMAs finish, frees
its tensor memory and returns.  moe_forward_opts.pipeline_wait_ns shortens the
pipeline waits (not the final waits for the kernel's own copies and MMAs) so
that a test can make them give up: nothing faults, hangs or traps here — the
waits simply run out of time.  The call must come back with the timeout bit
set and the CUDA context usable, and the next normal call on the same buffers
must give the oracle's result."""
import pytest
import torch

from moe_expert_layer_align_gb300 import workloads
from helpers import assert_layer_close, oracle_layer

pytestmark = pytest.mark.gpu

CASES = [
    # cfg, T, overrides, w8a16: long K so that the pipelines have waits to give up on
    (2, 24, dict(H=2048, I=512), False),                # bf16, gathered rows, fused SiLU-and-mul
    (2, 300, dict(H=1024, I=256, E=4), False),          # bf16, 128-row tiles (TMA + cp.async gather)
    (4, 20, dict(H=1024, I=512, E=16), False),          # FP8 swap-AB tiles
    (4, 300, dict(H=1024, I=256, E=4, k=2), False),     # FP8 token-major 128-row tiles
    (4, 20, dict(H=1024, I=512, E=16), True),           # w8a16
]


def call(wl, w8a16, opts, status, ws):
    import moe_expert_layer_align_gb300 as moe
    out_dtype = torch.bfloat16
    if wl.mode == "bf16":
        return moe.moe_forward(wl.x, wl.w13, wl.w2, wl.topk_ids, wl.topk_w, out_dtype=out_dtype,
                               opts=opts, dev_status=status, workspace=ws)
    return moe.moe_forward(wl.x, wl.w13q, wl.w2q, wl.topk_ids, wl.topk_w,
                           scales=(wl.w13s, wl.w2s), out_dtype=out_dtype, opts=opts,
                           dev_status=status, workspace=ws, w8a16=w8a16)


@pytest.mark.parametrize("cfg,T,kw,w8a16", CASES)
def test_short_wait_limit_flags_timeout_then_normal_call_is_correct(cfg, T, kw, w8a16):
    import moe_expert_layer_align_gb300 as moe
    wl = workloads.make(cfg, T, "cpu", **kw).to("cuda")
    w13 = wl.w13q if wl.mode == "fp8" else wl.w13
    shape = moe.layer_shape(wl.x, w13, wl.topk_ids, 0, torch.bfloat16, 0, w8a16)
    short = moe.make_opts(pipeline_wait_ns=1)
    ws = torch.empty(moe.moe_workspace_bytes(shape, short), dtype=torch.uint8, device="cuda")
    assert moe.moe_workspace_bytes(shape) == ws.numel()      # the option changes no plan
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    call(wl, w8a16, short, status, ws)
    torch.cuda.synchronize()                                  # returns: nothing hung or faulted
    assert status.item() & (1 << moe.MOE_ERR_TIMEOUT), f"status {status.item()}"
    for _ in range(2):                                        # the next normal calls
        status.fill_(-1)
        out = call(wl, w8a16, None, status, ws)
        torch.cuda.synchronize()
        assert status.item() == 0, moe.device_status_bits(status.item())
        assert_layer_close(out.double().cpu().numpy(), oracle_layer(wl, w8a16=w8a16), wl.mode,
                           f"cfg{cfg} T={T} after a timed-out call")

