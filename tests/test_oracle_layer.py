"""Pins of the oracle's layer: closed forms, a textbook special case, brute
force on tiny inputs, linearity and relabelling symmetry.

Each case is built so that a plausible slip in the oracle — gate and up
swapped, a transposed weight, the wrong expert or slot weight, a dropped term,
a sign — changes the result."""
import math

import numpy as np
import pytest
import torch

import oracle


def bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def silu(z):
    return z / (1.0 + math.exp(-z))


def rand_case(T, H, I, E, k, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(T, H, generator=g).bfloat16()
    w13 = (torch.randn(E, 2 * I, H, generator=g) / math.sqrt(H)).bfloat16()
    w2 = (torch.randn(E, H, I, generator=g) / math.sqrt(I)).bfloat16()
    ids = torch.stack([torch.randperm(E, generator=g)[:k] for _ in range(T)]).int()
    w = torch.rand(T, k, generator=g) + 0.1
    return x, w13, w2, ids, w


def run(x, w13, w2, ids, w, sel=None):
    return oracle.moe_bf16(bits(x), bits(w13), bits(w2), ids.numpy(), w.numpy(), sel)


def test_zero_weights_give_zero():
    x, w13, w2, ids, w = rand_case(5, 32, 16, 4, 2, 1)
    assert not run(x, torch.zeros_like(w13), w2, ids, w).any()
    assert not run(x, w13, torch.zeros_like(w2), ids, w).any()


def test_permutation_experts_closed_form():
    # I = H.  gate[e] = a_e P(sig_e), up[e] = b_e P(tau_e), W2[e] = d_e P(pi_e):
    # g_i = a_e x[sig_e(i)], u_i = b_e x[tau_e(i)], act_i = SiLU(g_i) u_i,
    # y_h = d_e act[pi_e(h)], out[t, h] = sum_j w_tj y_h.  Non-involutive
    # permutations make a transposed operand visible; distinct a, b make a
    # gate/up swap visible.
    T, H, E, k = 4, 16, 3, 2
    I = H
    rng = np.random.default_rng(0)
    coef = [(0.5 + e, -1.25 + 0.5 * e, 2.0 - 0.75 * e) for e in range(E)]   # exact in bf16
    perms = [[rng.permutation(H) for _ in range(3)] for _ in range(E)]
    w13 = torch.zeros(E, 2 * I, H)
    w2 = torch.zeros(E, H, I)
    for e in range(E):
        a, b, d = coef[e]
        sig, tau, pi = perms[e]
        for i in range(I):
            w13[e, i, sig[i]] = a
            w13[e, I + i, tau[i]] = b
        for h in range(H):
            w2[e, h, pi[h]] = d
    x = torch.randn(T, H, generator=torch.Generator().manual_seed(2)).bfloat16()
    ids = torch.tensor([[0, 2], [1, 0], [2, 1], [1, 2]], dtype=torch.int32)
    w = torch.tensor([[0.75, 0.25], [0.5, 0.5], [0.125, 0.875], [1.0, 0.375]])
    got = run(x, w13.bfloat16(), w2.bfloat16(), ids, w)
    xf = x.double().numpy()
    ref = np.zeros((T, H))
    for t in range(T):
        for j in range(k):
            e = int(ids[t, j])
            a, b, d = coef[e]
            sig, tau, pi = perms[e]
            act = [silu(a * xf[t, sig[i]]) * b * xf[t, tau[i]] for i in range(I)]
            for h in range(H):
                ref[t, h] += float(w[t, j]) * d * act[pi[h]]
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_diagonal_experts_closed_form():
    T, H, E = 3, 8, 2
    al, be, de = [1.5, -0.5], [0.25, 2.0], [-1.0, 0.75]
    w13 = torch.zeros(E, 2 * H, H)
    w2 = torch.zeros(E, H, H)
    for e in range(E):
        w13[e, :H] = torch.eye(H) * al[e]
        w13[e, H:] = torch.eye(H) * be[e]
        w2[e] = torch.eye(H) * de[e]
    x = torch.randn(T, H, generator=torch.Generator().manual_seed(3)).bfloat16()
    ids = torch.tensor([[1, 0], [0, 1], [1, 0]], dtype=torch.int32)
    w = torch.tensor([[0.6, 0.4], [0.3, 0.7], [0.9, 0.1]])
    got = run(x, w13.bfloat16(), w2.bfloat16(), ids, w)
    xf = x.double().numpy()
    ref = np.zeros((T, H))
    for t in range(T):
        for j in range(2):
            e = int(ids[t, j])
            for h in range(H):
                ref[t, h] += float(w[t, j]) * de[e] * silu(al[e] * xf[t, h]) * be[e] * xf[t, h]
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-14)


def test_single_expert_is_dense_swiglu_mlp():
    # k = 1, E = 1, weight 1: the textbook SwiGLU MLP W2 (SiLU(Wg x) * (Wu x)),
    # evaluated with numpy's fp64 matmul.
    T, H, I = 6, 64, 96
    x, w13, w2, _, _ = rand_case(T, H, I, 1, 1, 4)
    ids = torch.zeros(T, 1, dtype=torch.int32)
    w = torch.ones(T, 1)
    got = run(x, w13, w2, ids, w)
    X = x.double().numpy()
    Wg, Wu = w13[0, :I].double().numpy(), w13[0, I:].double().numpy()
    W2 = w2[0].double().numpy()
    G, U = X @ Wg.T, X @ Wu.T
    ref = (G / (1 + np.exp(-G)) * U) @ W2.T
    np.testing.assert_allclose(got, ref, rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("seed", range(4))
def test_brute_force_tiny(seed):
    # independent pure-Python loop over (t, j, i, h) in fp64
    rng = np.random.default_rng(seed)
    T, E = int(rng.integers(1, 5)), int(rng.integers(1, 5))
    k = int(rng.integers(1, min(E, 2) + 1))
    H, I = int(rng.integers(1, 17)), int(rng.integers(1, 17))
    x, w13, w2, ids, w = rand_case(T, H, I, E, k, 100 + seed)
    got = run(x, w13, w2, ids, w)
    X, W13, W2 = x.double().tolist(), w13.double().tolist(), w2.double().tolist()
    for t in range(T):
        ref = [0.0] * H
        for j in range(k):
            e = int(ids[t, j])
            act = []
            for i in range(I):
                gsum = sum(X[t][h] * W13[e][i][h] for h in range(H))
                usum = sum(X[t][h] * W13[e][I + i][h] for h in range(H))
                act.append(silu(gsum) * usum)
            for h in range(H):
                ref[h] += float(w[t, j]) * sum(act[i] * W2[e][h][i] for i in range(I))
        np.testing.assert_allclose(got[t], ref, rtol=1e-11, atol=1e-13)


def test_linearity_and_relabelling():
    x, w13, w2, ids, w = rand_case(7, 32, 24, 5, 3, 6)
    base = run(x, w13, w2, ids, w)
    np.testing.assert_array_equal(run(x, w13, (w2.float() * 2).bfloat16(), ids, w), 2 * base)
    np.testing.assert_allclose(run(x, w13, w2, ids, w * 4), 4 * base, rtol=1e-13, atol=0)
    perm = torch.randperm(5, generator=torch.Generator().manual_seed(9))
    inv = torch.argsort(perm)
    # expert e of the permuted set is expert perm[e] of the original
    got = run(x, w13[perm], w2[perm], inv[ids.long()].int(), w)
    np.testing.assert_array_equal(got, base)
    # selecting a subset of tokens returns the same rows
    sel = np.array([5, 0, 3], np.int32)
    np.testing.assert_array_equal(run(x, w13, w2, ids, w, sel), base[sel])


def test_invalid_ids_contribute_zero():
    x, w13, w2, ids, w = rand_case(4, 16, 16, 3, 2, 7)
    base = run(x, w13, w2, ids[:, :1].contiguous(), w[:, :1].contiguous())
    bad = ids.clone()
    bad[:, 1] = torch.tensor([3, -1, 99, 3], dtype=torch.int32)
    np.testing.assert_array_equal(run(x, w13, w2, bad, w), base)


# ------------------------------------------------------------------ FP8

def fp8_case(T, H, I, E, k, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(T, H, generator=g).bfloat16()
    w13q = torch.randint(0, 256, (E, 2 * I, H), generator=g, dtype=torch.uint8)
    w2q = torch.randint(0, 256, (E, H, I), generator=g, dtype=torch.uint8)
    w13q[(w13q & 0x7F) == 0x7F] = 0x3A      # no NaN codes in weights
    w2q[(w2q & 0x7F) == 0x7F] = 0xB1
    w13s = torch.rand(E, 2 * I // 128, H // 128, generator=g) * 0.01 + 0.001
    w2s = torch.rand(E, H // 128, I // 128, generator=g) * 0.01 + 0.001
    ids = torch.stack([torch.randperm(E, generator=g)[:k] for _ in range(T)]).int()
    w = torch.rand(T, k, generator=g) + 0.1
    return x, w13q, w13s, w2q, w2s, ids, w


def deq(codes):
    return torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).double().numpy()


def test_fp8_layer_brute_force_with_library_dequant():
    # Independent evaluation: torch's e4m3 decode, numpy fp64 matmuls, torch's
    # e4m3 cast for the activation requantisation (s = amax/448 in fp32).
    T, H, I, E, k = 3, 256, 256, 3, 2
    x, w13q, w13s, w2q, w2s, ids, w = fp8_case(T, H, I, E, k, 8)
    xq, xs = oracle.quant_x(bits(x))
    got = oracle.moe_fp8(xq, xs, w13q.numpy(), w13s.numpy(), w2q.numpy(), w2s.numpy(),
                         ids.numpy(), w.numpy())
    X = deq(xq) * np.repeat(xs.astype(np.float64), 128, axis=1)
    for t in range(T):
        ref = np.zeros(H)
        for j in range(k):
            e = int(ids[t, j])
            S13 = np.kron(w13s[e].double().numpy(), np.ones((128, 128)))
            S2 = np.kron(w2s[e].double().numpy(), np.ones((128, 128)))
            W13 = deq(w13q[e].numpy()) * S13
            W2 = deq(w2q[e].numpy()) * S2
            G, U = W13[:I] @ X[t], W13[I:] @ X[t]
            a32 = (G / (1 + np.exp(-G)) * U).astype(np.float32)
            ad = np.zeros(I)
            for b in range(I // 128):
                blk = a32[b * 128:(b + 1) * 128]
                s = np.float32(np.abs(blk).max()) / np.float32(448.0)
                q = torch.from_numpy(blk / s).to(torch.float8_e4m3fn)
                ad[b * 128:(b + 1) * 128] = q.double().numpy() * float(s)
            ref += float(w[t, j]) * (W2 @ ad)
        np.testing.assert_allclose(got[t], ref, rtol=1e-9, atol=1e-12)


def test_fp8_layer_scale_linearity_and_zero_gate():
    # Scaling every Down block scale by 8 scales the output by exactly 8 (a
    # dropped or misplaced Down scale would not); a zero gate gives SiLU(0) = 0
    # activations and a zero output.
    T, H, I, E, k = 2, 128, 128, 2, 1
    x, w13q, w13s, w2q, w2s, ids, w = fp8_case(T, H, I, E, k, 9)
    xq, xs = oracle.quant_x(bits(x))
    args = (xq, xs, w13q.numpy(), w13s.numpy(), w2q.numpy(), w2s.numpy(), ids.numpy(), w.numpy())
    base = oracle.moe_fp8(*args)
    up = oracle.moe_fp8(xq, xs, w13q.numpy(), w13s.numpy(), w2q.numpy(), (w2s * 8).numpy(),
                        ids.numpy(), w.numpy())
    np.testing.assert_allclose(up, 8 * base, rtol=1e-14, atol=0)
    zg = w13q.clone()
    zg[:, :I] = 0
    z = oracle.moe_fp8(xq, xs, zg.numpy(), w13s.numpy(), w2q.numpy(), w2s.numpy(),
                       ids.numpy(), w.numpy())
    assert not z.any()
