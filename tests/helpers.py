"""Shared test helpers: tolerances and conversions between torch tensors and
the oracle's numpy inputs."""
import numpy as np
import torch

# Tolerances of the layer output against the oracle (fp64):
#   bf16: relative L2 <= 1e-2 and max-abs <= 3e-2 * max|ref|
#   fp8:  relative L2 <= 5e-3 against the oracle fed the same quantised operands
BF16_REL_L2 = 1e-2
BF16_MAX_ABS_FRAC = 3e-2
FP8_REL_L2 = 5e-3


def bits16(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def u8(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.uint8).numpy()


def errors(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    rel_l2 = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300)
    max_abs = np.abs(got - ref).max()
    return rel_l2, max_abs, np.abs(ref).max()


def assert_layer_close(got, ref, mode: str, what: str = ""):
    rel_l2, max_abs, ref_max = errors(got, ref)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    if mode == "bf16":
        assert rel_l2 <= BF16_REL_L2, f"{what}: rel L2 {rel_l2:.3e} > {BF16_REL_L2}"
        assert max_abs <= BF16_MAX_ABS_FRAC * ref_max, (
            f"{what}: max abs {max_abs:.3e} > {BF16_MAX_ABS_FRAC} * {ref_max:.3e}")
    else:
        assert rel_l2 <= FP8_REL_L2, f"{what}: rel L2 {rel_l2:.3e} > {FP8_REL_L2}"
    return rel_l2, max_abs


def oracle_layer(wl, sel=None, topk_ids=None, topk_w=None, return_act=False):
    """Oracle output rows for a workloads.Workload (inputs copied to the host)."""
    import oracle
    ids = (wl.topk_ids if topk_ids is None else topk_ids).cpu().numpy()
    w = (wl.topk_w if topk_w is None else topk_w).cpu().numpy()
    if wl.mode == "bf16":
        return oracle.moe_bf16(bits16(wl.x), bits16(wl.w13), bits16(wl.w2), ids, w, sel)
    xq, xs = oracle.quant_x(bits16(wl.x))
    return oracle.moe_fp8(xq, xs, u8(wl.w13q), wl.w13s.cpu().numpy(), u8(wl.w2q),
                          wl.w2s.cpu().numpy(), ids, w, sel, return_act=return_act)


def run_layer(wl, topk_ids=None, topk_w=None, block_m=0, opts=None, dev_status=None,
              workspace=None):
    """The CUDA path through the C ABI for a workload already on the GPU."""
    import moe_expert_layer_align_gb300 as moe
    ids = wl.topk_ids if topk_ids is None else topk_ids
    w = wl.topk_w if topk_w is None else topk_w
    out_dtype = torch.float32 if wl.out == "f32" else torch.bfloat16
    if wl.mode == "bf16":
        return moe.moe_forward(wl.x, wl.w13, wl.w2, ids, w, out_dtype=out_dtype, block_m=block_m,
                               opts=opts, dev_status=dev_status, workspace=workspace)
    return moe.moe_forward(wl.x, wl.w13q, wl.w2q, ids, w, scales=(wl.w13s, wl.w2s),
                           out_dtype=out_dtype, block_m=block_m, opts=opts,
                           dev_status=dev_status, workspace=workspace)
