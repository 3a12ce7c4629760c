"""Pins for the oracle's combine + residual add + RMSNorm (CANN
aclnnMoeDistributeCombineAddRmsNorm; reading: x = combine + residual,
rstd = 1/sqrt(mean(x^2) + eps), y = x * rstd * gamma).  CPU only.

Pinned by a hand-worked row, closed forms (a constant row; scale invariance
with eps = 0), torch's own rms_norm in float64 (the library routine the
normalisation reduces to), and the derived tolerance accepting a float32
emulation of the same steps while rejecting a result off by a few bf16 steps.
"""
import numpy as np
import pytest
import torch

import oracle
from combine_ep_layout_03_gb300 import synth


def bits(v):
    a = np.asarray(v, np.float32)
    return oracle.bf16_from_f32(a).reshape(a.shape)


def test_hand_worked_row():
    # x = (1 + 2, 3 + 1) = (3, 4): mean of squares 12.5, rstd = 1/sqrt(12.5)
    c = np.array([[1.0, 3.0]])
    x, rstd, y = oracle.add_rms_norm_ref64(c, bits([2.0, 1.0]), bits([1.0, 2.0]), 0.0)
    assert np.array_equal(x, [[3.0, 4.0]])
    assert rstd[0] == pytest.approx(1.0 / np.sqrt(12.5), rel=1e-15)
    assert y[0] == pytest.approx([3.0 / np.sqrt(12.5), 8.0 / np.sqrt(12.5)], rel=1e-15)


@pytest.mark.parametrize("v,eps", [(0.75, 1e-6), (-3.0, 0.0), (1e-3, 1e-6)])
def test_constant_row(v, eps):
    H = 64
    g = np.linspace(0.5, 1.5, H).astype(np.float32)
    c = np.full((1, H), v - 0.5)
    x, rstd, y = oracle.add_rms_norm_ref64(c, bits(np.full(H, 0.5)), bits(g), eps)
    r = 1.0 / np.sqrt(v * v + eps)
    assert rstd[0] == pytest.approx(r, rel=1e-14)
    gb = oracle.bf16_bits_to_f64(bits(g))
    assert np.allclose(y[0], v * r * gb, rtol=1e-14, atol=0)


def test_scale_invariance_without_eps():
    rng = np.random.default_rng(5)
    H = 256
    c = rng.standard_normal((3, H))
    r0 = np.zeros(H, np.uint16)       # bf16 zero residual
    g = bits(rng.standard_normal(H))
    _, _, y1 = oracle.add_rms_norm_ref64(c, np.tile(r0, (3, 1)), g, 0.0)
    _, _, y2 = oracle.add_rms_norm_ref64(c * 1024.0, np.tile(r0, (3, 1)), g, 0.0)
    assert np.allclose(y1, y2, rtol=1e-13, atol=0)


@pytest.mark.parametrize("eps", [1e-6, 1e-2])
def test_matches_torch_rms_norm_float64(eps):
    rms_norm = getattr(torch.nn.functional, "rms_norm", None)
    if rms_norm is None:
        pytest.skip("torch without rms_norm")
    rng = np.random.default_rng(7)
    N, H = 9, 384
    c = rng.standard_normal((N, H)) * 3.0
    res = bits(rng.standard_normal((N, H)))
    g = bits(1.0 + 0.1 * rng.standard_normal(H))
    x, rstd, y = oracle.add_rms_norm_ref64(c, res, g, eps)
    xt = torch.from_numpy(c + oracle.bf16_bits_to_f64(res))
    yt = rms_norm(xt, (H,), torch.from_numpy(oracle.bf16_bits_to_f64(g)), eps).numpy()
    assert np.allclose(x, xt.numpy(), rtol=0, atol=0)
    assert np.allclose(y, yt, rtol=1e-12, atol=1e-14)
    assert np.allclose(rstd, 1.0 / np.sqrt((xt.numpy() ** 2).mean(axis=1) + eps), rtol=1e-14)


def f32_emulation(lay, y_bits, wts, res_bits, g_bits, eps):
    """float32 steps of an implementation: combine rounded to bf16, residual add,
    sum of squares, rstd, two products, bf16 outputs."""
    c_bits = oracle.combine(lay, y_bits, wts)
    c = oracle.bf16_bits_to_f64(c_bits).astype(np.float32)
    r = oracle.bf16_bits_to_f64(res_bits).astype(np.float32).reshape(c.shape)
    x = (c + r).astype(np.float32)
    ss = np.zeros(x.shape[0], np.float32)
    for h in range(x.shape[1]):
        ss = (ss + x[:, h] * x[:, h]).astype(np.float32)
    rstd = (np.float32(1.0) / np.sqrt((ss / np.float32(x.shape[1]) + np.float32(eps)).astype(np.float32))).astype(np.float32)
    g = oracle.bf16_bits_to_f64(g_bits).astype(np.float32)
    yv = ((x * rstd[:, None]).astype(np.float32) * g[None, :]).astype(np.float32)
    return oracle.bf16_from_f32(x).reshape(x.shape), rstd, oracle.bf16_from_f32(yv).reshape(yv.shape)


def test_tolerance_accepts_float32_steps_and_rejects_bf16_steps():
    w = synth.WORKLOADS[1].with_(T=16, H=256)
    topk = synth.gen_topk(w)
    wts = synth.gen_weights(w, topk)
    lay = oracle.layout(w.R, w.T, w.E, w.K, w.alpha, topk)
    x = synth.gen_x(w)
    y_bits, _ = oracle.dispatch(lay, x, 0)
    y_bits = y_bits.view(np.uint16).reshape(-1, w.H)
    res = synth.gen_residual(w)
    g = synth.gen_gamma(w)
    eps = synth.RMS_NORM_EPS
    ref = oracle.combine_add_rms_norm_ref64(lay, y_bits, wts, None, res, g, eps)
    xo, rs, yo = f32_emulation(lay, y_bits, wts, res, g, eps)
    ok, worst = oracle.add_rms_norm_within_tolerance(xo, rs, yo, ref, w.K, 0)
    assert ok, worst
    # the bound allows a few bf16 steps of y (the combine is rounded to bf16
    # before the residual add); one output moved by 2^-4 of its value (8 to 16
    # bf16 steps) is rejected
    bad = yo.copy().reshape(ref["y"].shape)
    bad[3, 17] = oracle.bf16_from_f32(np.float32(oracle.bf16_bits_to_f64(bad[3, 17]) * (1 + 2.0 ** -4)))[0]
    ok, _ = oracle.add_rms_norm_within_tolerance(xo, rs, bad, ref, w.K, 0)
    assert not ok
    # a residual left out is rejected
    ok, _ = oracle.add_rms_norm_within_tolerance(oracle.combine(lay, y_bits, wts), rs, yo, ref, w.K, 0)
    assert not ok


def f32_route_from_c(c_bits, res_bits, g_bits, eps):
    """numpy's binary32 operations, one step at a time (an independent route
    through the same IEEE operations), from the combine's bf16 output."""
    c = oracle.bf16_bits_to_f64(c_bits).astype(np.float32)
    r = oracle.bf16_bits_to_f64(res_bits).astype(np.float32).reshape(c.shape)
    x = (c + r).astype(np.float32)
    ss = np.zeros(x.shape[0], np.float32)
    for h in range(x.shape[1]):
        ss = (ss + (x[:, h] * x[:, h]).astype(np.float32)).astype(np.float32)
    mean = (ss / np.float32(x.shape[1])).astype(np.float32)
    rstd = (np.float32(1.0) / np.sqrt((mean + np.float32(eps)).astype(np.float32))).astype(np.float32)
    g = oracle.bf16_bits_to_f64(g_bits).astype(np.float32)
    yv = ((x * rstd[:, None]).astype(np.float32) * g[None, :]).astype(np.float32)
    xb = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    yb = torch.from_numpy(yv).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    return xb, rstd, yb


def test_f32_steps_hand_worked_exact():
    # c = 1, r = 1: x = 2 everywhere; sum of squares 16, mean 4, sqrt 2, rstd 0.5;
    # y = (2 * 0.5) * gamma = gamma; every step exact
    H = 4
    g = bits([1.0, -2.0, 0.75, 3.0])
    x, rstd, y = oracle.add_rms_norm_f32(bits(np.ones((1, H))), bits(np.ones((1, H))), g, 0.0)
    assert np.array_equal(x, bits(np.full((1, H), 2.0)))
    assert rstd[0] == np.float32(0.5)
    assert np.array_equal(y[0], g)
    # with eps = 12: mean 4 + 12 = 16, rstd 0.25, y = gamma / 2
    x, rstd, y = oracle.add_rms_norm_f32(bits(np.ones((1, H))), bits(np.ones((1, H))), g, 12.0)
    assert rstd[0] == np.float32(0.25)
    assert np.array_equal(y[0], bits(oracle.bf16_bits_to_f64(g) / 2))


@pytest.mark.parametrize("H,eps", [(256, 1e-6), (7168, 1e-6), (520, 0.5)])
def test_f32_steps_match_an_independent_float32_route(H, eps):
    rng = np.random.default_rng(H)
    N = 6
    c = bits(rng.standard_normal((N, H)) * 2.0)
    res = bits(rng.standard_normal((N, H)))
    g = bits(1.0 + 0.1 * rng.standard_normal(H))
    x, rstd, y = oracle.add_rms_norm_f32(c, res, g, eps)
    xe, re, ye = f32_route_from_c(c, res, g, eps)
    assert np.array_equal(x, xe)
    assert np.array_equal(rstd.view(np.uint32), re.view(np.uint32))
    assert np.array_equal(y, ye)


def test_f32_steps_within_the_derived_bound_of_the_exact_result():
    w = synth.WORKLOADS[1].with_(T=16, H=256)
    topk = synth.gen_topk(w)
    wts = synth.gen_weights(w, topk)
    lay = oracle.layout(w.R, w.T, w.E, w.K, w.alpha, topk)
    y_bits, _ = oracle.dispatch(lay, synth.gen_x(w), 0)
    y_bits = y_bits.view(np.uint16).reshape(-1, w.H)
    res = synth.gen_residual(w)
    g = synth.gen_gamma(w)
    eps = synth.RMS_NORM_EPS
    ref = oracle.combine_add_rms_norm_ref64(lay, y_bits, wts, None, res, g, eps)
    xo, rs, yo = oracle.add_rms_norm_f32(oracle.combine(lay, y_bits, wts), res.reshape(-1, w.H), g, eps)
    ok, worst = oracle.add_rms_norm_within_tolerance(xo, rs, yo, ref, w.K, 0)
    assert ok, worst
