"""CPU oracle of the fused MoE layer — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` may import this package.  The product path (the CUDA
library ``moe_expert_layer_align_gb300`` and its C ABI) never calls it.

The arithmetic lives in ``moe_oracle.c`` (plain C, fp64, OpenMP over output
rows only); this module compiles it with gcc and marshals numpy arrays through
ctypes.  Every function is pinned by ``tests/test_oracle_*.py``.

Passages followed (see the C file for details):
  * routing index — HPC-Ops × SGLang (LMSYS blog), section "MoE", fused
    pipeline, "routing and index build";
  * layer — same section, the conventional path's step order (route, Gate-Up,
    activation + quantisation, Down, top-k weighted reduce);
  * router — same post, section "Router GEMM", "a precision-aware BF16
    formulation";
  * FP8 — OCP E4M3 format; per-128 block scales of the SGLang MoE Triton
    tuning guide, section 4.1 (block_shape [128, 128]);
  * w8a16 — the HPC-Ops post's operator table, row MoE ("BF16 hidden
    states; FP8 E4M3 expert weights").
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle_moe.so")
_lock = threading.Lock()
_lib = None

_i32p = np.ctypeslib.ndpointer(dtype=np.int32, flags="C_CONTIGUOUS")
_u16p = np.ctypeslib.ndpointer(dtype=np.uint16, flags="C_CONTIGUOUS")
_u8p = np.ctypeslib.ndpointer(dtype=np.uint8, flags="C_CONTIGUOUS")
_f32p = np.ctypeslib.ndpointer(dtype=np.float32, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")
_c_int = ctypes.c_int


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/liboracle_moe.so`` (gcc, OpenMP)."""
    if force or not os.path.exists(_LIB_PATH) or (
        os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    ):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB_PATH)
            L.oracle_num_threads.restype = _c_int
            L.oracle_bf16_value.restype = ctypes.c_double
            L.oracle_bf16_value.argtypes = [ctypes.c_uint16]
            L.oracle_bf16_rne.restype = ctypes.c_uint16
            L.oracle_bf16_rne.argtypes = [ctypes.c_float]
            L.oracle_bf16_trunc.restype = ctypes.c_uint16
            L.oracle_bf16_trunc.argtypes = [ctypes.c_float]
            L.oracle_e4m3_decode.restype = ctypes.c_double
            L.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
            L.oracle_e4m3_encode.restype = ctypes.c_uint8
            L.oracle_e4m3_encode.argtypes = [ctypes.c_float]
            for nm, a, b in (("oracle_e4m3_encode_n", _f32p, _u8p),
                             ("oracle_e4m3_decode_n", _u8p, _f64p),
                             ("oracle_bf16_rne_n", _f32p, _u16p),
                             ("oracle_bf16_trunc_n", _f32p, _u16p)):
                f = getattr(L, nm)
                f.restype = None
                f.argtypes = [a, ctypes.c_int64, b]
            L.oracle_quant_group.restype = None
            L.oracle_quant_group.argtypes = [_f32p, _c_int, _u8p, _f32p]
            L.oracle_quant_x.restype = None
            L.oracle_quant_x.argtypes = [_c_int, _c_int, _u16p, _u8p, _f32p]
            L.oracle_tiles_cap.restype = ctypes.c_int64
            L.oracle_tiles_cap.argtypes = [_c_int] * 4
            L.oracle_align.restype = _c_int
            L.oracle_align.argtypes = [_i32p, _c_int, _c_int, _c_int, _c_int,
                                       _i32p, _i32p, _i32p, _i32p, _i32p, _i32p, _i32p]
            L.oracle_moe_bf16.restype = None
            L.oracle_moe_bf16.argtypes = [_c_int] * 5 + [_u16p, _u16p, _u16p, _i32p, _f32p,
                                                         _i32p, _c_int, _f64p]
            L.oracle_moe_fp8.restype = None
            L.oracle_moe_fp8.argtypes = [_c_int] * 5 + [
                _u8p, _f32p, _u8p, _f32p, _u8p, _f32p, _i32p, _f32p, _i32p, _c_int, _f64p,
                ctypes.c_void_p, ctypes.c_void_p]
            L.oracle_moe_w8a16.restype = None
            L.oracle_moe_w8a16.argtypes = [_c_int] * 5 + [
                _u16p, _u8p, _f32p, _u8p, _f32p, _i32p, _f32p, _i32p, _c_int, _f64p]
            L.oracle_router_split.restype = None
            L.oracle_router_split.argtypes = [_f32p, ctypes.c_int64, _u16p, _u16p]
            L.oracle_router_scores.restype = None
            L.oracle_router_scores.argtypes = [_c_int, _c_int, _c_int, _u16p, _f32p, _f64p]
            L.oracle_router_topk.restype = None
            L.oracle_router_topk.argtypes = [_c_int, _c_int, _c_int, _f64p, _c_int,
                                             ctypes.c_double, _i32p, _f64p]
            _lib = L
    return _lib


def num_threads() -> int:
    return int(lib().oracle_num_threads())


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ------------------------------------------------------------------ numbers

def bf16_value(bits) -> np.ndarray:
    b = _c(bits, np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _map(fname, values, in_dtype, out_dtype):
    v = _c(values, in_dtype)
    out = np.zeros(v.shape, out_dtype)
    getattr(lib(), fname)(v.reshape(-1), v.size, out.reshape(-1))
    return out


def bf16_rne(values) -> np.ndarray:
    return _map("oracle_bf16_rne_n", values, np.float32, np.uint16)


def bf16_trunc(values) -> np.ndarray:
    return _map("oracle_bf16_trunc_n", values, np.float32, np.uint16)


def e4m3_decode(codes) -> np.ndarray:
    return _map("oracle_e4m3_decode_n", codes, np.uint8, np.float64)


def e4m3_encode(values) -> np.ndarray:
    return _map("oracle_e4m3_encode_n", values, np.float32, np.uint8)


def quant_group(values):
    v = _c(values, np.float32).ravel()
    q = np.zeros(v.size, np.uint8)
    s = np.zeros(1, np.float32)
    lib().oracle_quant_group(v, v.size, q, s)
    return q, float(s[0])


def quant_x(x_bits):
    """bf16 bits [T, H] -> (e4m3 codes [T, H], fp32 scales [T, H/128])."""
    x = _c(x_bits, np.uint16)
    T, H = x.shape
    assert H % 128 == 0
    xq = np.zeros((T, H), np.uint8)
    xs = np.zeros((T, H // 128), np.float32)
    lib().oracle_quant_x(T, H, x, xq, xs)
    return xq, xs


# ------------------------------------------------------------------ index

def tiles_cap(T: int, k: int, E: int, bm: int) -> int:
    return int(lib().oracle_tiles_cap(T, k, E, bm))


def align(topk_ids, E: int, bm: int) -> dict:
    ids = _c(topk_ids, np.int32)
    T, k = ids.shape
    tc = tiles_cap(T, k, E, bm)
    out = dict(
        counts=np.zeros(E, np.int32),
        offsets=np.zeros(E + 1, np.int32),
        sorted_ids=np.zeros(tc * bm, np.int32),
        tile_expert=np.zeros(tc, np.int32),
        tiles=np.zeros((tc, 4), np.int32),
        inv_pos=np.zeros(T * k, np.int32),
        num_tiles=np.zeros(1, np.int32),
    )
    out["invalid"] = int(lib().oracle_align(
        ids.ravel(), T, k, E, bm, out["counts"], out["offsets"], out["sorted_ids"],
        out["tile_expert"], out["tiles"].reshape(-1), out["inv_pos"], out["num_tiles"]))
    out["tiles_cap"] = tc
    out["rows_cap"] = tc * bm
    return out


# ------------------------------------------------------------------ layer

def _sel(sel, T):
    return _c(np.arange(T) if sel is None else sel, np.int32)


def moe_bf16(x_bits, w13_bits, w2_bits, topk_ids, topk_w, sel=None) -> np.ndarray:
    """fp64 output rows [len(sel), H] of the BF16 layer for the tokens `sel`."""
    x = _c(x_bits, np.uint16)
    w13 = _c(w13_bits, np.uint16)
    w2 = _c(w2_bits, np.uint16)
    ids = _c(topk_ids, np.int32)
    w = _c(topk_w, np.float32)
    T, H = x.shape
    E, I2, _ = w13.shape
    k = ids.shape[1]
    s = _sel(sel, T)
    out = np.zeros((s.size, H), np.float64)
    lib().oracle_moe_bf16(T, H, I2 // 2, E, k, x.ravel(), w13.ravel(), w2.ravel(),
                          ids.ravel(), w.ravel(), s, s.size, out)
    return out


def moe_fp8(xq, xs, w13q, w13s, w2q, w2s, topk_ids, topk_w, sel=None, return_act=False):
    """fp64 output rows of the FP8 w8a8 layer.  With return_act, also the
    activation codes [n_sel, k, I] and scales [n_sel, k, I/128]."""
    xq = _c(xq, np.uint8)
    xs = _c(xs, np.float32)
    w13q = _c(w13q, np.uint8)
    w13s = _c(w13s, np.float32)
    w2q = _c(w2q, np.uint8)
    w2s = _c(w2s, np.float32)
    ids = _c(topk_ids, np.int32)
    w = _c(topk_w, np.float32)
    T, H = xq.shape
    E, I2, _ = w13q.shape
    I = I2 // 2
    k = ids.shape[1]
    s = _sel(sel, T)
    out = np.zeros((s.size, H), np.float64)
    aq = np.zeros((s.size, k, I), np.uint8) if return_act else None
    as_ = np.zeros((s.size, k, I // 128), np.float32) if return_act else None
    lib().oracle_moe_fp8(T, H, I, E, k, xq.ravel(), xs.ravel(), w13q.ravel(), w13s.ravel(),
                         w2q.ravel(), w2s.ravel(), ids.ravel(), w.ravel(), s, s.size, out,
                         aq.ctypes.data if return_act else None,
                         as_.ctypes.data if return_act else None)
    if return_act:
        return out, aq, as_
    return out


def moe_w8a16(x_bits, w13q, w13s, w2q, w2s, topk_ids, topk_w, sel=None) -> np.ndarray:
    """fp64 output rows of the w8a16 layer: bf16 x, e4m3 weights with fp32
    128x128 block scales dequantised exactly, no activation quantisation."""
    x = _c(x_bits, np.uint16)
    w13q = _c(w13q, np.uint8)
    w13s = _c(w13s, np.float32)
    w2q = _c(w2q, np.uint8)
    w2s = _c(w2s, np.float32)
    ids = _c(topk_ids, np.int32)
    w = _c(topk_w, np.float32)
    T, H = x.shape
    E, I2, _ = w13q.shape
    k = ids.shape[1]
    s = _sel(sel, T)
    out = np.zeros((s.size, H), np.float64)
    lib().oracle_moe_w8a16(T, H, I2 // 2, E, k, x.ravel(), w13q.ravel(), w13s.ravel(),
                           w2q.ravel(), w2s.ravel(), ids.ravel(), w.ravel(), s, s.size, out)
    return out


# ------------------------------------------------------------------ variants
# Two variants of the layer that the pages' serving stack uses, written as
# what they are: the plain layer applied to re-mapped routing.

def shared_routing(topk_ids, topk_w, E: int, n_shared: int, weight: float = 1.0):
    """Shared-expert fusion (SGLang's MoE kernels for DeepSeek-V3 / GLM4-MoE /
    Llama 4): the shared experts E..E+n_shared-1 are extra experts that every
    token selects with `weight`.  Returns the routing of the plain layer over
    E + n_shared experts: topk_ids[T][k + n_shared], topk_w likewise."""
    ids = _c(topk_ids, np.int32)
    w = _c(topk_w, np.float32)
    T = ids.shape[0]
    sid = np.broadcast_to(np.arange(E, E + n_shared, dtype=np.int32), (T, n_shared))
    sw = np.full((T, n_shared), weight, np.float32)
    return np.concatenate([ids, sid], 1), np.concatenate([w, sw], 1)


def ep_local_ids(topk_ids, e0: int, E_local: int):
    """Expert parallelism, one rank's part (SGLang MoE tuning guide, section 1:
    EP places whole experts on ranks): the rank holds the global experts
    [e0, e0 + E_local) as its local 0..E_local-1; an assignment to any other
    expert is not this rank's (-1: dropped, contributes 0).  The rank's output
    is its partial sum; the ranks' outputs add up to the full layer."""
    ids = _c(topk_ids, np.int32)
    loc = ids - e0
    return np.where((ids >= e0) & (ids < e0 + E_local), loc, -1).astype(np.int32)


# ------------------------------------------------------------------ router

def router_split(wr):
    w = _c(wr, np.float32)
    hi = np.zeros(w.shape, np.uint16)
    lo = np.zeros(w.shape, np.uint16)
    lib().oracle_router_split(w.ravel(), w.size, hi.reshape(-1), lo.reshape(-1))
    return hi, lo


def router_scores(x_bits, wr) -> np.ndarray:
    x = _c(x_bits, np.uint16)
    w = _c(wr, np.float32)
    T, H = x.shape
    E = w.shape[0]
    out = np.zeros((T, E), np.float64)
    lib().oracle_router_scores(T, H, E, x.ravel(), w.ravel(), out)
    return out


def router_topk(scores, k: int, score_fn: int = 0, scale: float = 1.0):
    s = _c(scores, np.float64)
    T, E = s.shape
    ids = np.zeros((T, k), np.int32)
    w = np.zeros((T, k), np.float64)
    lib().oracle_router_topk(T, E, k, s, score_fn, scale, ids, w)
    return ids, w
