"""Pins of the two routing variants of the oracle (shared-expert fusion and
the expert-parallel local part) against facts that hold whatever the oracle
computes: a shared expert adds a dense SwiGLU MLP of every token (numpy), and
the expert-parallel parts of a partition of the experts add up to the full
layer."""
import math

import numpy as np
import torch

import oracle


def bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def val(t):
    return t.float().double().numpy()


def case(T, H, I, E, k, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(T, H, generator=g).bfloat16()
    w13 = (torch.randn(E, 2 * I, H, generator=g) / math.sqrt(H)).bfloat16()
    w2 = (torch.randn(E, H, I, generator=g) / math.sqrt(I)).bfloat16()
    ids = torch.stack([torch.randperm(E, generator=g)[:k] for _ in range(T)]).int()
    w = torch.rand(T, k, generator=g) + 0.1
    return x, w13, w2, ids, w


def dense_swiglu(x, w13, w2):
    """x [T,H] @ one expert, in fp64 numpy: W2 (SiLU(x W_gate^T) * x W_up^T)."""
    I = w13.shape[0] // 2
    g = x @ w13[:I].T
    u = x @ w13[I:].T
    return (g / (1.0 + np.exp(-g)) * u) @ w2.T


def test_shared_expert_adds_a_dense_mlp():
    T, H, I, E, k = 6, 48, 32, 5, 2
    x, w13, w2, ids, w = case(T, H, I, E + 2, k, 3)   # experts E, E+1 are the shared ones
    ids = ids % E                                      # routed ids stay below E
    for n_shared, weight in ((1, 1.0), (2, 0.5)):
        sid, sw = oracle.shared_routing(ids.numpy(), w.numpy(), E, n_shared, weight)
        assert sid.shape == (T, k + n_shared) and (sid[:, k:] == np.arange(E, E + n_shared)).all()
        got = oracle.moe_bf16(bits(x), bits(w13), bits(w2), sid, sw)
        routed = oracle.moe_bf16(bits(x), bits(w13), bits(w2), ids.numpy(), w.numpy())
        extra = sum(weight * dense_swiglu(val(x), val(w13[e]), val(w2[e]))
                    for e in range(E, E + n_shared))
        np.testing.assert_allclose(got, routed + extra, rtol=1e-9, atol=1e-12)


def test_expert_parallel_parts_add_up_to_the_layer():
    T, H, I, E, k = 7, 32, 16, 8, 3
    x, w13, w2, ids, w = case(T, H, I, E, k, 5)
    full = oracle.moe_bf16(bits(x), bits(w13), bits(w2), ids.numpy(), w.numpy())
    for bounds in ((0, 3, 8), (0, 1, 2, 5, 8), (0, 8)):
        parts = []
        for e0, e1 in zip(bounds[:-1], bounds[1:]):
            loc = oracle.ep_local_ids(ids.numpy(), e0, e1 - e0)
            assert ((loc >= 0) == ((ids.numpy() >= e0) & (ids.numpy() < e1))).all()
            parts.append(oracle.moe_bf16(bits(x), bits(w13[e0:e1]), bits(w2[e0:e1]), loc,
                                         w.numpy()))
        np.testing.assert_allclose(sum(parts), full, rtol=1e-9, atol=1e-12)


def test_ep_part_of_an_expert_nobody_selected_is_zero():
    x, w13, w2, ids, w = case(4, 32, 16, 6, 2, 7)
    ids = ids % 5                                      # expert 5 never selected
    loc = oracle.ep_local_ids(ids.numpy(), 5, 1)
    assert (loc == -1).all()
    assert not oracle.moe_bf16(bits(x), bits(w13[5:]), bits(w2[5:]), loc, w.numpy()).any()


def test_shared_expert_index_holds_every_token_in_order():
    T, E, k, bm = 37, 6, 2, 16
    g = np.random.default_rng(0)
    ids = np.stack([g.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    sid, _ = oracle.shared_routing(ids, np.ones((T, k), np.float32), E, 1)
    idx = oracle.align(sid, E + 1, bm)
    o = idx["offsets"]
    rows = idx["sorted_ids"][o[E]: o[E] + T]
    np.testing.assert_array_equal(rows, np.arange(T) * (k + 1) + k)   # slot k of every token
    assert idx["counts"][E] == T


# ---------------------------------------------------------------- w8a16

def w8_case(T, H, I, E, k, seed, pow2_scales=False):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(T, H, generator=g).bfloat16()
    q13 = torch.randint(0, 256, (E, 2 * I, H), generator=g, dtype=torch.uint8)
    q2 = torch.randint(0, 256, (E, H, I), generator=g, dtype=torch.uint8)
    q13[(q13 & 0x7F) == 0x7F] = 0          # no NaN codes
    q2[(q2 & 0x7F) == 0x7F] = 0
    if pow2_scales:
        s13 = 2.0 ** torch.randint(-12, -4, (E, 2 * I // 128, H // 128), generator=g).float()
        s2 = 2.0 ** torch.randint(-12, -4, (E, H // 128, I // 128), generator=g).float()
    else:
        s13 = torch.rand(E, 2 * I // 128, H // 128, generator=g) * 1e-3 + 1e-4
        s2 = torch.rand(E, H // 128, I // 128, generator=g) * 1e-3 + 1e-4
    ids = torch.stack([torch.randperm(E, generator=g)[:k] for _ in range(T)]).int()
    w = torch.rand(T, k, generator=g) + 0.1
    return x, q13, s13, q2, s2, ids, w


def test_w8a16_with_power_of_two_scales_is_the_bf16_layer():
    # e4m3 values times 2^n are exact in bf16: the w8a16 oracle must then equal
    # the bf16 oracle fed those dequantised weights
    x, q13, s13, q2, s2, ids, w = w8_case(5, 256, 128, 3, 2, 1, pow2_scales=True)
    deq13 = torch.from_numpy(oracle.e4m3_decode(q13.numpy())).float() * \
        s13.repeat_interleave(128, 1).repeat_interleave(128, 2)
    deq2 = torch.from_numpy(oracle.e4m3_decode(q2.numpy())).float() * \
        s2.repeat_interleave(128, 1).repeat_interleave(128, 2)
    assert torch.equal(deq13.bfloat16().float(), deq13) and torch.equal(deq2.bfloat16().float(), deq2)
    got = oracle.moe_w8a16(bits(x), q13.numpy(), s13.numpy(), q2.numpy(), s2.numpy(),
                           ids.numpy(), w.numpy())
    ref = oracle.moe_bf16(bits(x), bits(deq13.bfloat16()), bits(deq2.bfloat16()), ids.numpy(),
                          w.numpy())
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-15)


def test_w8a16_brute_force_and_block_scales():
    # each scale acts on its own 128x128 block only: a numpy restatement with
    # the scales expanded per element, per token and slot
    x, q13, s13, q2, s2, ids, w = w8_case(3, 256, 256, 2, 2, 2)
    got = oracle.moe_w8a16(bits(x), q13.numpy(), s13.numpy(), q2.numpy(), s2.numpy(),
                           ids.numpy(), w.numpy())
    dq = lambda q, s: oracle.e4m3_decode(q.numpy()) * np.repeat(np.repeat(  # noqa: E731
        s.numpy().astype(np.float64), 128, 1), 128, 2)
    W13, W2 = dq(q13, s13), dq(q2, s2)
    X = val(x)
    I = 256
    ref = np.zeros((3, 256))
    for t in range(3):
        for j in range(2):
            e = ids[t, j].item()
            g = W13[e, :I] @ X[t]
            u = W13[e, I:] @ X[t]
            ref[t] += w[t, j].item() * (W2[e] @ (g / (1 + np.exp(-g)) * u))
    np.testing.assert_allclose(got, ref, rtol=1e-9, atol=1e-12)
