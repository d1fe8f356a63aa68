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
# Router: scores within SCORE_TOL of the fp64 oracle; top-k ids equal except
# where the oracle's k-th and (k+1)-th scores lie within TIE_GAP.
SCORE_TOL = 2e-3
TIE_GAP = 1e-5


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


def oracle_layer(wl, sel=None, topk_ids=None, topk_w=None, return_act=False, w8a16=False):
    """Oracle output rows for a workloads.Workload (inputs copied to the host).
    w8a16: the FP8 workload's weights with bf16 activations."""
    import oracle
    ids = (wl.topk_ids if topk_ids is None else topk_ids).cpu().numpy()
    w = (wl.topk_w if topk_w is None else topk_w).cpu().numpy()
    if w8a16:
        return oracle.moe_w8a16(bits16(wl.x), u8(wl.w13q), wl.w13s.cpu().numpy(), u8(wl.w2q),
                                wl.w2s.cpu().numpy(), ids, w, sel)
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


def check_topk(ids_gpu, ids_ref, scores_ref, k, scores_gpu=None):
    """The selected id sets must match except where the oracle's k-th and
    (k+1)-th scores lie within TIE_GAP; the GPU's own order must be
    descending in its scores."""
    for t in range(ids_ref.shape[0]):
        if scores_gpu is not None:
            assert np.all(np.diff(scores_gpu[t][ids_gpu[t]]) <= 0), t
        if set(ids_gpu[t]) == set(ids_ref[t]):
            continue
        s = np.sort(scores_ref[t])[::-1]
        assert s[k - 1] - s[k] < TIE_GAP, (t, ids_gpu[t], ids_ref[t])


def oracle_layer_sampled(wl, ids, w, sel, w8a16=False):
    """Oracle rows of the tokens `sel` only.  A token's output depends on its
    own x row, ids, weights and the experts it routes to, so the oracle is
    fed just those: the sampled x rows and the used experts' weights, with
    the ids renumbered into that expert subset (a pure selection of inputs,
    no arithmetic)."""
    import oracle
    sel = np.asarray(sel)
    ids_s = np.asarray(ids)[sel]
    used, inv = np.unique(ids_s, return_inverse=True)
    ids_c = inv.reshape(ids_s.shape).astype(np.int32)
    w_s = np.asarray(w)[sel]
    rows = torch.from_numpy(sel).long().to(wl.x.device)
    ex = torch.from_numpy(used).long().to(wl.x.device)
    x = bits16(wl.x[rows])
    if w8a16:
        return oracle.moe_w8a16(x, u8(wl.w13q[ex]), wl.w13s[ex].cpu().numpy(), u8(wl.w2q[ex]),
                                wl.w2s[ex].cpu().numpy(), ids_c, w_s)
    if wl.mode == "bf16":
        return oracle.moe_bf16(x, bits16(wl.w13[ex]), bits16(wl.w2[ex]), ids_c, w_s)
    xq, xs = oracle.quant_x(x)
    return oracle.moe_fp8(xq, xs, u8(wl.w13q[ex]), wl.w13s[ex].cpu().numpy(), u8(wl.w2q[ex]),
                          wl.w2s[ex].cpu().numpy(), ids_c, w_s)
