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
