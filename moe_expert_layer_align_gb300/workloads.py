"""Seeded synthetic workloads of the fused MoE layer.

This module only draws inputs: hidden states, expert weights (and, for the
FP8 layers, their 128x128 block quantisation), top-k routing for the layers
whose router is outside the path, and router weights for the layer whose
router is in the path.  It holds none of the layer's own arithmetic; both
the CUDA path and the CPU oracle consume what it returns.

The five workloads follow the shapes on which the "HPC-Ops × SGLang" post and
the SGLang MoE Triton tuning guide measure MoE layers (Mixtral-, Qwen3- and
DeepSeek-V3-shaped experts), with random weights and routing in place of the
served models and captured routing traces, which are not available:

  1 tiny-bf16           T=8, H=256, I=512, E=8, k=2, softmax top-2, fp32 out
  2 mixtral-8x7b-bf16   H=4096, I=14336, E=8, k=2, softmax top-2, bf16 out
  3 qwen3-30b-a3b-bf16  H=2048, I=768, E=128, k=8, softmax top-8, bf16 out
  4 deepseek-v3-fp8     H=7168, I=2048, E=256, k=8, sigmoid top-8 renormalised
                        and scaled by 2.5, e4m3 weights with fp32 128x128 block
                        scales, bf16 out
  5 zipf-router-fp8     the FP8 layer with config-3 shapes whose routing comes
                        from an in-path router GEMM over fp32 router weights
                        biased so that expert popularity follows Zipf(1.2)

Recipe: x ~ N(0, 1) rounded to bf16; W13 ~ N(0, 1) / sqrt(H) and
W2 ~ N(0, 1) / sqrt(I) (the std is 1/sqrt(fan-in)); routing logits ~ N(0, 1).
Weights are drawn from a torch.Generator seeded 1000*config on the generating
device; x and the routing from one seeded 1000*config + T.  The values
therefore depend on the generating device (CPU and CUDA generators differ);
whatever is drawn is handed to both sides unchanged.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

CONFIGS = {
    1: dict(name="tiny-bf16", H=256, I=512, E=8, k=2, mode="bf16", out="f32",
            routing="softmax", scale=1.0, sweep=(8,)),
    2: dict(name="mixtral-8x7b-bf16", H=4096, I=14336, E=8, k=2, mode="bf16", out="bf16",
            routing="softmax", scale=1.0, sweep=(1, 2, 4, 8, 16, 32, 64, 128, 512, 2048)),
    3: dict(name="qwen3-30b-a3b-bf16", H=2048, I=768, E=128, k=8, mode="bf16", out="bf16",
            routing="softmax", scale=1.0, sweep=(1, 8, 16, 32, 64, 256, 1024, 4096)),
    4: dict(name="deepseek-v3-fp8", H=7168, I=2048, E=256, k=8, mode="fp8", out="bf16",
            routing="sigmoid", scale=2.5, sweep=(1, 16, 64, 512, 4096)),
    5: dict(name="zipf-router-fp8", H=2048, I=768, E=128, k=8, mode="fp8", out="bf16",
            routing="router", scale=1.0, zipf_s=1.2, sweep=(4, 16, 64, 256)),
}


@dataclass
class Workload:
    """Inputs of one layer invocation (torch tensors on one device)."""
    name: str
    T: int
    H: int
    I: int
    E: int
    k: int
    mode: str                      # "bf16" | "fp8"
    out: str                       # "f32" | "bf16"
    x: torch.Tensor                # bf16 [T, H]
    w13: torch.Tensor | None = None    # bf16 [E, 2I, H]
    w2: torch.Tensor | None = None     # bf16 [E, H, I]
    w13q: torch.Tensor | None = None   # uint8 (e4m3 codes) [E, 2I, H]
    w13s: torch.Tensor | None = None   # fp32 [E, 2I/128, H/128]
    w2q: torch.Tensor | None = None    # uint8 [E, H, I]
    w2s: torch.Tensor | None = None    # fp32 [E, H/128, I/128]
    topk_ids: torch.Tensor | None = None   # int32 [T, k]
    topk_w: torch.Tensor | None = None     # fp32 [T, k]
    wr: torch.Tensor | None = None         # fp32 [E, H] router weights (in-path router)
    router_fn: int = 0                     # 0 softmax, 1 sigmoid
    router_scale: float = 1.0
    meta: dict = field(default_factory=dict)

    def to(self, device) -> "Workload":
        kw = {}
        for f in self.__dataclass_fields__:
            v = getattr(self, f)
            kw[f] = v.to(device) if isinstance(v, torch.Tensor) else v
        return Workload(**kw)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _quant_blocks(w: torch.Tensor):
    """Weight block quantisation for input synthesis: per 128x128 block,
    s = amax/448 (1 if the block is 0), codes = torch's e4m3 cast of w/s."""
    R, C = w.shape
    b = w.reshape(R // 128, 128, C // 128, 128)
    amax = b.abs().amax(dim=(1, 3))
    s = torch.where(amax == 0, torch.ones_like(amax), amax / 448.0)
    q = (b / s[:, None, :, None]).clamp(-448.0, 448.0).to(torch.float8_e4m3fn)
    return q.reshape(R, C).view(torch.uint8), s.float()


def expert_weights(H, I, E, mode, seed, device="cpu"):
    """W13 [E, 2I, H] and W2 [E, H, I], bf16 or e4m3 + block scales."""
    g = _gen(seed, device)
    if mode == "bf16":
        w13 = torch.empty((E, 2 * I, H), dtype=torch.bfloat16, device=device)
        w2 = torch.empty((E, H, I), dtype=torch.bfloat16, device=device)
        for e in range(E):
            w13[e] = (torch.randn((2 * I, H), generator=g, device=device) / math.sqrt(H)).bfloat16()
            w2[e] = (torch.randn((H, I), generator=g, device=device) / math.sqrt(I)).bfloat16()
        return dict(w13=w13, w2=w2)
    w13q = torch.empty((E, 2 * I, H), dtype=torch.uint8, device=device)
    w2q = torch.empty((E, H, I), dtype=torch.uint8, device=device)
    w13s = torch.empty((E, 2 * I // 128, H // 128), dtype=torch.float32, device=device)
    w2s = torch.empty((E, H // 128, I // 128), dtype=torch.float32, device=device)
    for e in range(E):
        w13q[e], w13s[e] = _quant_blocks(torch.randn((2 * I, H), generator=g, device=device) / math.sqrt(H))
        w2q[e], w2s[e] = _quant_blocks(torch.randn((H, I), generator=g, device=device) / math.sqrt(I))
    return dict(w13q=w13q, w13s=w13s, w2q=w2q, w2s=w2s)


def synth_routing(T, E, k, kind, scale, g, device="cpu"):
    """Top-k routing for layers whose router is outside the path: N(0,1)
    logits; softmax (or sigmoid) probabilities; the k largest; weights
    renormalised to sum 1, times `scale`."""
    logits = torch.randn((T, E), generator=g, device=device, dtype=torch.float64)
    probs = torch.softmax(logits, dim=-1) if kind == "softmax" else torch.sigmoid(logits)
    _, ids = torch.topk(logits, k, dim=-1)
    sel = torch.gather(probs, 1, ids)
    w = sel / sel.sum(dim=-1, keepdim=True) * scale
    return ids.to(torch.int32), w.to(torch.float32)


def zipf_router_weights(H, E, s, seed, device="cpu"):
    """fp32 router weights [E, H] ~ N(0, 1)/sqrt(H) with channel 0 biased by
    ln p_e, p_e proportional to rank_e^-s over a seeded permutation of ranks;
    paired with x[:, 0] = 1 this makes expert popularity Zipf(s)-shaped."""
    g = _gen(seed, device)
    wr = torch.randn((E, H), generator=g, device=device) / math.sqrt(H)
    rank = torch.randperm(E, generator=g, device=device).to(torch.float64) + 1.0
    p = rank.pow(-s)
    p = p / p.sum()
    wr[:, 0] += torch.log(p).to(wr.dtype)
    return wr


def make_tokens(cfg: int, T: int, H: int, E: int, k: int, device="cpu", token_seed=None):
    """Hidden states and (for layers whose router is outside the path) top-k
    routing of workload `cfg` at T tokens: x first, then the routing, both
    from one generator seeded 1000*cfg + T."""
    c = CONFIGS[cfg]
    gt = _gen(1000 * cfg + T if token_seed is None else token_seed, device)
    x = torch.randn((T, H), generator=gt, device=device).bfloat16()
    if c["routing"] == "router":
        x[:, 0] = 1.0            # carries the Zipf bias of the router weights
        return x, None, None
    ids, w = synth_routing(T, E, k, c["routing"], c["scale"], gt, device)
    return x, ids, w


def make(cfg: int, T: int | None = None, device="cpu", *, H=None, I=None, E=None, k=None,
         weight_seed: int | None = None, token_seed: int | None = None,
         base: "Workload | None" = None) -> Workload:
    """Workload `cfg` (1..5) at T tokens.  Shape fields may be overridden to
    draw smaller cases of the same recipe (tests).  With `base`, its weights
    are reused and only the tokens are drawn (a sweep over T)."""
    c = dict(CONFIGS[cfg])
    T = c["sweep"][0] if T is None else T
    if base is not None:
        H, I, E, k = base.H, base.I, base.E, base.k
    H = c["H"] if H is None else H
    I = c["I"] if I is None else I
    E = c["E"] if E is None else E
    k = c["k"] if k is None else k
    wseed = 1000 * cfg if weight_seed is None else weight_seed
    x, ids, w = make_tokens(cfg, T, H, E, k, device, token_seed)
    wl = Workload(name=c["name"], T=T, H=H, I=I, E=E, k=k, mode=c["mode"], out=c["out"], x=x,
                  topk_ids=ids, topk_w=w,
                  meta=dict(config=cfg, weight_seed=wseed,
                            token_seed=1000 * cfg + T if token_seed is None else token_seed))
    if base is not None:
        for key in ("w13", "w2", "w13q", "w13s", "w2q", "w2s", "wr"):
            setattr(wl, key, getattr(base, key))
    else:
        for key, v in expert_weights(H, I, E, c["mode"], wseed, device).items():
            setattr(wl, key, v)
        if c["routing"] == "router":
            wl.wr = zipf_router_weights(H, E, c["zipf_s"], wseed + 1, device)
    if c["routing"] == "router":
        wl.router_fn, wl.router_scale = 0, 1.0
    return wl


# The router on its own at the "HPC-Ops × SGLang" post's router-GEMM table
# shape (section "Router GEMM", Table 2: K = 4096, N = 192, BF16 activations
# times FP32 router weights), over the table's token counts M.
ROUTER_SHAPE = dict(H=4096, E=192, k=8, sweep=(1, 16, 48, 96, 208, 512, 1024, 2048, 4096))


def router_inputs(M: int, device="cpu", H: int = ROUTER_SHAPE["H"], E: int = ROUTER_SHAPE["E"],
                  seed: int = 6000):
    """x [M, H] ~ N(0, 1) rounded to bf16 and fp32 router weights [E, H] ~
    N(0, 1/sqrt(H)) (weights from `seed`, x from seed + M)."""
    wr = torch.randn((E, H), generator=_gen(seed, device), device=device) / math.sqrt(H)
    x = torch.randn((M, H), generator=_gen(seed + M, device), device=device).bfloat16()
    return x, wr


def bf16_bits(t: torch.Tensor):
    """numpy uint16 view of a bf16 tensor (bit patterns), on the host."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view("uint16")
