"""ctypes binding of the C ABI in ``include/moe.h``.

Argument marshalling only: every step of the layer runs in the CUDA library
``lib/libmoe_gb300.so``.  Importing this module loads that library and raises
if it is missing — there is no fallback path.  PyTorch provides device memory
and streams.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "lib", "libmoe_gb300.so")

MOE_OK, MOE_ERR_ARG, MOE_ERR_SHAPE, MOE_ERR_DTYPE, MOE_ERR_ALIGN = 0, 1, 2, 3, 4
MOE_ERR_WORKSPACE, MOE_ERR_EXPERT_ID, MOE_ERR_TIMEOUT, MOE_ERR_CUDA = 5, 6, 7, 8
MOE_BF16, MOE_FP8_W8A8, MOE_W8A16 = 0, 1, 2
MOE_OUT_F32, MOE_OUT_BF16 = 0, 1
MOE_SCORE_SOFTMAX, MOE_SCORE_SIGMOID = 0, 1
# Stage indices of moe_forward_opts.stage_events.
STAGES = ("align", "quant_x", "gateup", "act", "down", "combine")

_i32 = ctypes.c_int32
_vp = ctypes.c_void_p
_sz = ctypes.c_size_t


class moe_shape(ctypes.Structure):
    _fields_ = [("T", _i32), ("H", _i32), ("I", _i32), ("E", _i32), ("k", _i32),
                ("block_m", _i32), ("mode", _i32), ("out_dtype", _i32)]


class moe_index(ctypes.Structure):
    _fields_ = [(n, _vp) for n in ("counts", "offsets", "sorted_ids", "tile_expert", "tiles",
                                   "inv_pos", "num_tiles")]


class moe_scales(ctypes.Structure):
    _fields_ = [("w13_scale", _vp), ("w2_scale", _vp)]


class moe_forward_opts(ctypes.Structure):
    _fields_ = [("disable_pdl", _i32), ("split_gateup", _i32), ("split_down", _i32),
                ("grid_ctas", _i32), ("stage_events", _vp * 8), ("separate_act", _i32),
                ("smem_index", _i32), ("single_weight_tile", _i32),
                ("num_shared_experts", _i32), ("shared_expert_weight", ctypes.c_float),
                ("ep_first_expert", _i32), ("ep_num_experts", _i32), ("fuse_routing", _i32),
                ("unit_order", _i32), ("pipeline_wait_ns", _i32), ("coalesce_rows", _i32),
                ("down_tile_rows", _i32), ("separate_quant", _i32)]


class moe_align_opts(ctypes.Structure):
    _fields_ = [("num_shared_experts", _i32), ("ep_first_expert", _i32), ("ep_num_experts", _i32)]


class moe_workspace_layout(ctypes.Structure):
    _fields_ = [("block_m", _i32), ("tiles_cap", _i32), ("rows_cap", _i32),
                ("split_gateup", _i32), ("split_down", _i32), ("grid_gateup", _i32),
                ("grid_down", _i32), ("fused_act", _i32), ("smem_index", _i32),
                ("weight_tiles_per_unit", _i32), ("route_fused", _i32), ("unit_order", _i32)] + [
        (n, _sz) for n in ("off_counts", "off_offsets", "off_sorted_ids", "off_tile_expert",
                           "off_tiles", "off_inv_pos", "off_num_tiles", "off_index_scratch", "off_xq", "off_xs",
                           "off_xs_rows", "off_g", "off_a", "off_as", "off_y", "off_router",
                           "off_route_counter", "total_bytes", "off_route_hist")] + [
        ("coalesce_rows", _i32), ("off_work_tiles", _sz), ("off_num_work_tiles", _sz),
        ("y_bf16", _i32), ("down_tile_rows", _i32), ("work_cap", _i32), ("g_act_rows", _i32),
        ("xs_by_token", _i32)]


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"CUDA library {LIB_PATH} is missing; build it first "
            "(python -c 'import __graft_entry__ as g; g.build()')")
    L = ctypes.CDLL(LIB_PATH)
    P = ctypes.POINTER
    sig = {
        "moe_index_tiles_cap": (_sz, [_i32, _i32, _i32, _i32]),
        "moe_plan": (_i32, [P(moe_shape), P(moe_forward_opts), P(moe_workspace_layout)]),
        "moe_workspace_bytes": (_sz, [P(moe_shape), P(moe_forward_opts)]),
        "moe_align": (_i32, [_vp, _i32, _i32, _i32, _i32, P(moe_index), _vp, _vp]),
        "moe_align_ex": (_i32, [_vp, _i32, _i32, _i32, _i32, P(moe_align_opts), P(moe_index),
                                _vp, _vp]),
        "moe_forward": (_i32, [P(moe_shape), _vp, _vp, _vp, _vp, _vp, P(moe_scales), _vp, _vp,
                               _sz, _vp, _vp]),
        "moe_forward_ex": (_i32, [P(moe_shape), _vp, _vp, _vp, _vp, _vp, P(moe_scales), _vp,
                                  _vp, _sz, _vp, _vp, P(moe_forward_opts)]),
        "moe_combine": (_i32, [P(moe_shape), _i32, _i32, _vp, _vp, _vp, _vp, _vp]),
        "moe_router_prepare": (_i32, [_vp, _i32, _i32, _vp, _vp]),
        "moe_router_workspace_bytes": (_sz, [_i32, _i32, _i32]),
        "moe_router_topk": (_i32, [_vp, _vp, _i32, _i32, _i32, _i32, _i32, ctypes.c_float,
                                   _vp, _vp, _vp, _vp, _sz, _vp]),
        "moe_forward_static": (_i32, [P(moe_shape), _vp, _vp, _vp, _vp, _vp, P(moe_scales),
                                      _vp, _vp, _vp]),
        "moe_status_str": (ctypes.c_char_p, [_i32]),
        "moe_plan_routed": (_i32, [P(moe_shape), P(moe_forward_opts), P(moe_workspace_layout)]),
        "moe_routed_workspace_bytes": (_sz, [P(moe_shape), P(moe_forward_opts)]),
        "moe_forward_routed": (_i32, [P(moe_shape), _vp, _vp, _i32, ctypes.c_float, _vp, _vp,
                                      P(moe_scales), _vp, _vp, _vp, _vp, _vp, _sz, _vp, _vp,
                                      P(moe_forward_opts)]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    return L


lib = _load()
SYMBOLS = ("moe_index_tiles_cap", "moe_plan", "moe_workspace_bytes", "moe_align", "moe_forward",
           "moe_forward_ex", "moe_combine", "moe_router_prepare", "moe_router_workspace_bytes",
           "moe_router_topk", "moe_forward_static", "moe_status_str", "moe_align_ex",
           "moe_plan_routed", "moe_routed_workspace_bytes", "moe_forward_routed")
# Largest workspace moe_forward_static can serve (MOE_STATIC_SCRATCH_BYTES).
STATIC_SCRATCH_BYTES = 128 << 20


class MoeError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {moe_status_str(status)} (status {status})")


def moe_status_str(status: int) -> str:
    return lib.moe_status_str(status).decode()


def _check(status: int, what: str):
    if status != MOE_OK:
        raise MoeError(status, what)


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def device_status_bits(word: int) -> list[int]:
    """Decode a dev_status word into the moe_status codes whose bits are set."""
    return [c for c in (MOE_ERR_EXPERT_ID, MOE_ERR_TIMEOUT) if word & (1 << c)]


# ---------------------------------------------------------------- shapes

def make_shape(T, H, I, E, k, block_m=0, fp8=False, out_bf16=True, mode=None) -> moe_shape:
    """mode: MOE_BF16 / MOE_FP8_W8A8 / MOE_W8A16 (default from `fp8`)."""
    m = mode if mode is not None else (MOE_FP8_W8A8 if fp8 else MOE_BF16)
    return moe_shape(T, H, I, E, k, block_m, m, MOE_OUT_BF16 if out_bf16 else MOE_OUT_F32)


def moe_index_tiles_cap(T, k, E, block_m) -> int:
    return int(lib.moe_index_tiles_cap(T, k, E, block_m))


def make_opts(disable_pdl=False, split_gateup=0, split_down=0, grid_ctas=0,
              stage_events=None, separate_act=False, smem_index=None,
              single_weight_tile=False, num_shared_experts=0, shared_expert_weight=0.0,
              ep_first_expert=0, ep_num_experts=0, fuse_routing=None,
              unit_order=0, pipeline_wait_ns=0, coalesce_rows=0,
              down_tile_rows=0, separate_quant=False) -> moe_forward_opts:
    o = moe_forward_opts()
    o.separate_quant = int(separate_quant)
    o.down_tile_rows = down_tile_rows   # 0 planner, -1 off, 128
    o.coalesce_rows = coalesce_rows   # 0 planner, -1 off, 32 / 64
    o.pipeline_wait_ns = pipeline_wait_ns
    o.unit_order = unit_order
    # None: planner (separate kernels); True / False: one cooperative launch / separate
    o.fuse_routing = 0 if fuse_routing is None else (1 if fuse_routing else -1)
    o.num_shared_experts = num_shared_experts
    o.shared_expert_weight = shared_expert_weight
    o.ep_first_expert = ep_first_expert
    o.ep_num_experts = ep_num_experts
    o.disable_pdl = int(disable_pdl)
    o.separate_act = int(separate_act)
    # None: planner; True / False: on / off
    o.smem_index = 0 if smem_index is None else (1 if smem_index else -1)
    o.single_weight_tile = int(single_weight_tile)
    o.split_gateup = split_gateup
    o.split_down = split_down
    o.grid_ctas = grid_ctas
    for i, ev in enumerate(stage_events or []):
        o.stage_events[i] = None if ev is None else ev.cuda_event
    return o


def moe_plan(shape: moe_shape, opts: moe_forward_opts | None = None) -> moe_workspace_layout:
    L = moe_workspace_layout()
    _check(lib.moe_plan(ctypes.byref(shape), ctypes.byref(opts) if opts else None,
                        ctypes.byref(L)), "moe_plan")
    return L


def moe_workspace_bytes(shape: moe_shape, opts: moe_forward_opts | None = None) -> int:
    return int(lib.moe_workspace_bytes(ctypes.byref(shape), ctypes.byref(opts) if opts else None))


# ---------------------------------------------------------------- calls

def alloc_index(T, k, E, block_m, device="cuda") -> dict:
    tc = moe_index_tiles_cap(T, k, E, block_m)
    z = lambda n: torch.empty(n, dtype=torch.int32, device=device)  # noqa: E731
    return dict(counts=z(E), offsets=z(E + 1), sorted_ids=z(tc * block_m), tile_expert=z(tc),
                tiles=z(tc * 4).view(tc, 4), inv_pos=z(T * k), num_tiles=z(1))


def moe_align(topk_ids: torch.Tensor, E: int, block_m: int, index: dict | None = None,
              dev_status: torch.Tensor | None = None, stream=None) -> dict:
    T, k = topk_ids.shape
    idx = index if index is not None else alloc_index(T, k, E, block_m, topk_ids.device)
    ci = moe_index(*[_ptr(idx[n]) for n in ("counts", "offsets", "sorted_ids", "tile_expert",
                                            "tiles", "inv_pos", "num_tiles")])
    _check(lib.moe_align(_ptr(topk_ids), T, k, E, block_m, ctypes.byref(ci), _ptr(dev_status),
                         _stream(stream)), "moe_align")
    return idx


def moe_align_ex(topk_ids: torch.Tensor, E: int, block_m: int, num_shared_experts=0,
                 ep_first_expert=0, ep_num_experts=0, index: dict | None = None,
                 dev_status: torch.Tensor | None = None, stream=None) -> dict:
    """moe_align with shared experts and / or the expert-parallel local range:
    the index covers T*(k + n_shared) assignments over E + n_shared experts."""
    T, k = topk_ids.shape
    kk, Ei = k + num_shared_experts, E + num_shared_experts
    idx = index if index is not None else alloc_index(T, kk, Ei, block_m, topk_ids.device)
    ci = moe_index(*[_ptr(idx[n]) for n in ("counts", "offsets", "sorted_ids", "tile_expert",
                                            "tiles", "inv_pos", "num_tiles")])
    o = moe_align_opts(num_shared_experts, ep_first_expert, ep_num_experts)
    _check(lib.moe_align_ex(_ptr(topk_ids), T, k, E, block_m, ctypes.byref(o), ctypes.byref(ci),
                            _ptr(dev_status), _stream(stream)), "moe_align_ex")
    return idx


def layer_shape(x, w13, topk_ids, block_m=0, out_dtype=None, n_shared=0,
                w8a16=False) -> moe_shape:
    """Shape of a layer call; w13 holds the routed experts and then `n_shared`
    shared ones, so the shape's E (routed) is w13's first extent - n_shared.
    e4m3 weights mean the FP8 layer, or with w8a16 the bf16-activation one."""
    T, H = x.shape
    E, I2, _ = w13.shape
    E -= n_shared
    fp8 = w13.dtype in (torch.uint8, torch.float8_e4m3fn)
    out_bf16 = (out_dtype or torch.bfloat16) == torch.bfloat16
    return make_shape(T, H, I2 // 2, E, topk_ids.shape[1], block_m, fp8, out_bf16,
                      MOE_W8A16 if (fp8 and w8a16) else None)


def moe_forward(x, w13, w2, topk_ids, topk_w, *, scales=None, out=None, out_dtype=None,
                workspace=None, block_m=0, dev_status=None, stream=None, opts=None,
                w8a16=False):
    """The whole layer.  BF16: w13/w2 bf16.  FP8: w13/w2 uint8 e4m3 codes and
    scales = (w13_scale, w2_scale); w8a16=True keeps the activations bf16
    (MOE_W8A16).  Returns `out` [T, H] (bf16 or fp32)."""
    shape = layer_shape(x, w13, topk_ids, block_m,
                        out.dtype if out is not None else out_dtype,
                        opts.num_shared_experts if opts is not None else 0, w8a16)
    if out is None:
        out = torch.empty(x.shape, dtype=torch.bfloat16 if shape.out_dtype else torch.float32,
                          device=x.device)
    need = moe_workspace_bytes(shape, opts)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    sc = moe_scales(_ptr(scales[0]), _ptr(scales[1])) if scales is not None else None
    args = (ctypes.byref(shape), _ptr(x), _ptr(w13), _ptr(w2), _ptr(topk_ids), _ptr(topk_w),
            ctypes.byref(sc) if sc else None, _ptr(out), _ptr(workspace), workspace.numel(),
            _ptr(dev_status), _stream(stream))
    if opts is None:
        _check(lib.moe_forward(*args), "moe_forward")
    else:
        _check(lib.moe_forward_ex(*args, ctypes.byref(opts)), "moe_forward_ex")
    return out


def moe_forward_static(x, w13, w2, topk_ids, topk_w, *, scales=None, out=None, out_dtype=None,
                       dev_status=None, stream=None):
    """moe_forward for callers that cannot allocate device memory: the
    intermediates live in the library's own static device scratch
    (STATIC_SCRATCH_BYTES, shared by all calls, so calls must not overlap on
    the GPU).  Only `out` is allocated here when not given."""
    shape = layer_shape(x, w13, topk_ids, 0, out.dtype if out is not None else out_dtype)
    if out is None:
        out = torch.empty(x.shape, dtype=torch.bfloat16 if shape.out_dtype else torch.float32,
                          device=x.device)
    sc = moe_scales(_ptr(scales[0]), _ptr(scales[1])) if scales is not None else None
    _check(lib.moe_forward_static(ctypes.byref(shape), _ptr(x), _ptr(w13), _ptr(w2),
                                  _ptr(topk_ids), _ptr(topk_w), ctypes.byref(sc) if sc else None,
                                  _ptr(out), _ptr(dev_status), _stream(stream)),
           "moe_forward_static")
    return out


def moe_combine(y, inv_pos, topk_w, T, H, k, splits, rows_cap, out=None, out_dtype=None,
                stream=None):
    out_dtype = out.dtype if out is not None else (out_dtype or torch.float32)
    if out is None:
        out = torch.empty((T, H), dtype=out_dtype, device=y.device)
    shape = make_shape(T, H, 64, 1, k, 0, False, out_dtype == torch.bfloat16)
    _check(lib.moe_combine(ctypes.byref(shape), splits, rows_cap, _ptr(y), _ptr(inv_pos),
                           _ptr(topk_w), _ptr(out), _stream(stream)), "moe_combine")
    return out


def moe_router_prepare(wr: torch.Tensor, stream=None) -> torch.Tensor:
    E, H = wr.shape
    hi_lo = torch.empty((2 * E, H), dtype=torch.bfloat16, device=wr.device)
    _check(lib.moe_router_prepare(_ptr(wr), E, H, _ptr(hi_lo), _stream(stream)),
           "moe_router_prepare")
    return hi_lo


def moe_router_workspace_bytes(T, H, E) -> int:
    return int(lib.moe_router_workspace_bytes(T, H, E))


def moe_router_topk(x, hi_lo, k, score_fn=MOE_SCORE_SOFTMAX, scale=1.0, *, scores=None,
                    topk_ids=None, topk_w=None, workspace=None, stream=None):
    T, H = x.shape
    E = hi_lo.shape[0] // 2
    dev = x.device
    scores = scores if scores is not None else torch.empty((T, E), dtype=torch.float32, device=dev)
    topk_ids = topk_ids if topk_ids is not None else torch.empty((T, k), dtype=torch.int32, device=dev)
    topk_w = topk_w if topk_w is not None else torch.empty((T, k), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = torch.empty(max(16, moe_router_workspace_bytes(T, H, E)), dtype=torch.uint8,
                                device=dev)
    _check(lib.moe_router_topk(_ptr(x), _ptr(hi_lo), T, H, E, k, score_fn, scale, _ptr(scores),
                               _ptr(topk_ids), _ptr(topk_w), _ptr(workspace), workspace.numel(),
                               _stream(stream)), "moe_router_topk")
    return scores, topk_ids, topk_w


def moe_plan_routed(shape: moe_shape, opts: moe_forward_opts | None = None) -> moe_workspace_layout:
    L = moe_workspace_layout()
    _check(lib.moe_plan_routed(ctypes.byref(shape), ctypes.byref(opts) if opts else None,
                               ctypes.byref(L)), "moe_plan_routed")
    return L


def moe_routed_workspace_bytes(shape: moe_shape, opts: moe_forward_opts | None = None) -> int:
    return int(lib.moe_routed_workspace_bytes(ctypes.byref(shape),
                                              ctypes.byref(opts) if opts else None))


def moe_forward_routed(x, hi_lo, k, w13, w2, *, score_fn=MOE_SCORE_SOFTMAX, scale=1.0,
                       scales=None, out=None, out_dtype=None, scores=None, topk_ids=None,
                       topk_w=None, workspace=None, block_m=0, dev_status=None, stream=None,
                       opts=None):
    """The layer with its router in the path: returns (out, scores, topk_ids,
    topk_w); the routing outputs are written by the call."""
    T, H = x.shape
    E = hi_lo.shape[0] // 2
    dev = x.device
    scores = scores if scores is not None else torch.empty((T, E), dtype=torch.float32, device=dev)
    topk_ids = topk_ids if topk_ids is not None else torch.empty((T, k), dtype=torch.int32, device=dev)
    topk_w = topk_w if topk_w is not None else torch.empty((T, k), dtype=torch.float32, device=dev)
    shape = layer_shape(x, w13, topk_ids, block_m, out.dtype if out is not None else out_dtype)
    if out is None:
        out = torch.empty(x.shape, dtype=torch.bfloat16 if shape.out_dtype else torch.float32,
                          device=dev)
    need = moe_routed_workspace_bytes(shape, opts)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    sc = moe_scales(_ptr(scales[0]), _ptr(scales[1])) if scales is not None else None
    _check(lib.moe_forward_routed(ctypes.byref(shape), _ptr(x), _ptr(hi_lo), score_fn, scale,
                                  _ptr(w13), _ptr(w2), ctypes.byref(sc) if sc else None,
                                  _ptr(scores), _ptr(topk_ids), _ptr(topk_w), _ptr(out),
                                  _ptr(workspace), workspace.numel(), _ptr(dev_status),
                                  _stream(stream), ctypes.byref(opts) if opts else None),
           "moe_forward_routed")
    return out, scores, topk_ids, topk_w


def workspace_views(workspace: torch.Tensor, shape: moe_shape, opts=None, routed=False) -> dict:
    """Views of the intermediates moe_forward (moe_forward_routed with
    routed=True) left in `workspace` (index, quantised x, Gate-Up partials or
    SiLU(gate)*up rows, activation, Down partials)."""
    L = moe_plan_routed(shape, opts) if routed else moe_plan(shape, opts)
    T, H, I, E, k = shape.T, shape.H, shape.I, shape.E, shape.k
    ns = opts.num_shared_experts if opts is not None else 0
    E, k = E + ns, k + ns   # experts and assignments per token of the index
    rc, tc = L.rows_cap, L.tiles_cap
    fp8 = shape.mode == MOE_FP8_W8A8

    def v(off, n, dtype, shp):
        nbytes = n * torch.tensor([], dtype=dtype).element_size()
        return workspace[off: off + nbytes].view(dtype).view(*shp)

    out = dict(
        layout=L,
        counts=v(L.off_counts, E, torch.int32, (E,)),
        offsets=v(L.off_offsets, E + 1, torch.int32, (E + 1,)),
        sorted_ids=v(L.off_sorted_ids, rc, torch.int32, (rc,)),
        tile_expert=v(L.off_tile_expert, tc, torch.int32, (tc,)),
        tiles=v(L.off_tiles, 4 * tc, torch.int32, (tc, 4)),
        inv_pos=v(L.off_inv_pos, T * k, torch.int32, (T * k,)),
        num_tiles=v(L.off_num_tiles, 1, torch.int32, (1,)),
        Y=(v(L.off_y, rc * H, torch.bfloat16, (1, rc, H)) if L.y_bf16 else
           v(L.off_y, L.split_down * rc * H, torch.float32, (L.split_down, rc, H))),
    )
    if L.work_cap:
        wc = L.work_cap
        out["work_tiles"] = v(L.off_work_tiles, 4 * wc, torch.int32, (wc, 4))
        out["num_work_tiles"] = v(L.off_num_work_tiles, 1, torch.int32, (1,))
    if L.g_act_rows:
        out["Gact"] = v(L.off_g, rc * I, torch.float32, (rc, I))   # SiLU(gate) * up
    elif not L.fused_act:
        out["G"] = v(L.off_g, L.split_gateup * rc * 2 * I, torch.float32,
                     (L.split_gateup, rc, 2 * I))
    if fp8:
        out["xq"] = v(L.off_xq, T * H, torch.uint8, (T, H))
        out["xs"] = v(L.off_xs, T * (H // 128), torch.float32, (T, H // 128))
        if not L.xs_by_token:
            out["xs_rows"] = v(L.off_xs_rows, rc * (H // 128), torch.float32, (rc, H // 128))
        out["A"] = v(L.off_a, rc * I, torch.uint8, (rc, I))
        out["As"] = v(L.off_as, rc * (I // 128), torch.float32, (rc, I // 128))
    else:
        out["A"] = v(L.off_a, rc * I, torch.bfloat16, (rc, I))
    return out
