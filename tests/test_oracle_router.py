"""Pins of the oracle's router ("a precision-aware BF16 formulation",
HPC-Ops × SGLang, section Router GEMM): the hi/lo split bound, fp64 scores
against numpy's matmul, top-k against numpy's stable argsort, and a negative
control showing that a bf16-only router misses the 2e-3 bound."""
import math

import numpy as np
import pytest
import torch

import oracle


def test_split_reconstruction_bound():
    rng = np.random.default_rng(1)
    W = (rng.standard_normal(200000) / math.sqrt(2048)).astype(np.float32)
    hi, lo = oracle.router_split(W)
    assert np.array_equal(hi, oracle.bf16_trunc(W))
    hv = oracle.bf16_value(hi)
    lv = oracle.bf16_value(lo)
    W64 = W.astype(np.float64)
    r = W64 - hv                           # exact in fp32 and fp64
    # lo is the bf16 RNE of r * 256 (torch's cast, a library routine)
    ref_lo = torch.from_numpy((r * 256).astype(np.float32)).to(torch.bfloat16)
    assert np.array_equal(lo, ref_lo.view(torch.int16).numpy().view(np.uint16))
    err = np.abs(W64 - hv - lv / 256.0)
    assert np.all(np.abs(r) < 2.0 ** -7 * np.abs(W64))
    # RNE to bf16's 8 significant bits errs by at most half a spacing: 2^-8 |r|
    assert np.all(err <= 2.0 ** -8 * np.abs(r))
    assert np.all(err < 2.0 ** -15 * np.abs(W64) + 1e-45)


def test_scores_match_numpy_fp64():
    g = torch.Generator().manual_seed(2)
    x = torch.randn(9, 256, generator=g).bfloat16()
    wr = torch.randn(16, 256, generator=g) / 16
    got = oracle.router_scores(x.view(torch.int16).numpy().view(np.uint16), wr.numpy())
    ref = x.double().numpy() @ wr.double().numpy().T
    np.testing.assert_allclose(got, ref, rtol=1e-13, atol=1e-14)


@pytest.mark.parametrize("fn,scale", [(0, 1.0), (1, 2.5)])
def test_topk_selection_and_weights(fn, scale):
    rng = np.random.default_rng(3)
    s = rng.standard_normal((50, 32))
    s[0, 5] = s[0, 9] = 10.0                          # tie: lower id first
    ids, w = oracle.router_topk(s, 4, fn, scale)
    ref_ids = np.argsort(-s, axis=1, kind="stable")[:, :4]
    assert np.array_equal(ids, ref_ids)
    assert ids[0, 0] == 5 and ids[0, 1] == 9
    p = np.exp(s - s.max(1, keepdims=True))
    p = p / p.sum(1, keepdims=True) if fn == 0 else 1 / (1 + np.exp(-s))
    sel = np.take_along_axis(p, ids, 1)
    np.testing.assert_allclose(w, scale * sel / sel.sum(1, keepdims=True), rtol=1e-13)
    np.testing.assert_allclose(w.sum(1), scale, rtol=1e-13)


def test_negative_control_bf16_only_router_misses_bound():
    # The two-bf16 scores stay within 2e-3 of the fp64 reference; dropping the
    # low part (a plain bf16 router) does not, for the same inputs.
    g = torch.Generator().manual_seed(4)
    x = torch.randn(64, 2048, generator=g).bfloat16()
    wr = (torch.randn(128, 2048, generator=g) / math.sqrt(2048)).float()
    xb = x.view(torch.int16).numpy().view(np.uint16)
    ref = oracle.router_scores(xb, wr.numpy())
    hi, lo = oracle.router_split(wr.numpy())
    X = x.double().numpy()
    two = X @ oracle.bf16_value(hi).T + (X @ oracle.bf16_value(lo).T) / 256
    one = X @ oracle.bf16_value(hi).T
    assert np.abs(two - ref).max() < 2e-3 * 0.01
    assert np.abs(one - ref).max() > 2e-3
