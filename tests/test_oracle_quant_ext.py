"""Pins for the oracle's further quant modes (CPU only): per-token FP8
(quantMode 2 with an FP8 destination), per-group-128 FP8 (quantMode 3),
static int8 (quantMode 1) with scalar / per-channel / per-expert scales, and
smooth scales for the dynamic modes (CANN aclnnMoeDistributeDispatchV2,
Formula section, Cases 2-4); and the xActiveMask layout.

Independent routes: hand-worked rows (tests/golden/fp8_static_rows.txt), exact
rational arithmetic for the scale and the product with torch's float8 cast for
the element code, exact rationals for static int8, scale invariances, and the
brute-force layout for masks.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from combine_ep_layout_03_gb300 import synth
from test_oracle_layout import assert_layout_equal, brute_layout
from test_oracle_quant import _rne_f32, _rne_int, bf16_bits, read_cases

MODES = {"fp8t_e4m3": oracle.Q_FP8T_E4M3, "fp8t_e5m2": oracle.Q_FP8T_E5M2,
         "fp8g_e4m3": oracle.Q_FP8G_E4M3, "fp8g_e5m2": oracle.Q_FP8G_E5M2,
         "int8_static": oracle.Q_INT8_STATIC}
FP8 = {oracle.Q_FP8T_E4M3: (oracle.Q_E4M3, 448.0, torch.float8_e4m3fn),
       oracle.Q_FP8T_E5M2: (oracle.Q_E5M2, 57344.0, torch.float8_e5m2),
       oracle.Q_FP8G_E4M3: (oracle.Q_E4M3, 448.0, torch.float8_e4m3fn),
       oracle.Q_FP8G_E5M2: (oracle.Q_E5M2, 57344.0, torch.float8_e5m2)}


def f32_bits(v):
    return int(np.float32(v).view(np.uint32))


def row_from(case, H):
    x = np.zeros(H, np.float32)
    vals = [float(v) for v in case.get("x", [])]
    x[:len(vals)] = vals
    if "x128" in case:
        v2 = [float(v) for v in case["x128"]]
        x[128:128 + len(v2)] = v2
    return bf16_bits(x)


@pytest.mark.parametrize("case", read_cases("fp8_static_rows.txt"), ids=lambda c: c["name"])
def test_golden(case):
    q = MODES[case["mode"][0]]
    H = int(case["H"][0])
    x = row_from(case, H)
    if q == oracle.Q_INT8_STATIC:
        sc = [float(v) for v in case["scale"]]
        smooth = sc[0] if len(sc) == 1 else np.array(sc, np.float32)
        assert oracle.quant_int8_static_row(x, smooth).tolist() == [int(v) for v in case["q"]]
        return
    fp8 = FP8[q][0]
    if q in (oracle.Q_FP8T_E4M3, oracle.Q_FP8T_E5M2):
        codes, inv = oracle.quant_fp8_token_row(fp8, x)
        inv = [inv]
    else:
        codes, inv = oracle.quant_fp8_group_row(fp8, x)
    want = [int(v, 16) for v in case["codes"]]
    assert codes[:len(want)].tolist() == want
    if "codes128" in case:
        w2 = [int(v, 16) for v in case["codes128"]]
        assert codes[128:128 + len(w2)].tolist() == w2
    assert [f32_bits(v) for v in inv] == [int(v, 16) for v in case["inv"]]


def _exact_fp8_row(x_bits, fp8_mode, smooth=None):
    """Exact-rational scale and product, torch's float8 cast for the code."""
    fmt, dmax, tdt = FP8[fp8_mode]
    xf = (x_bits.astype(np.uint32) << 16).view(np.float32)
    if smooth is not None:
        xf = np.array([_rne_f32(Fraction(float(a)) * Fraction(float(b))) for a, b in zip(xf, smooth)],
                      dtype=object)
    xs = [Fraction(float(v)) for v in xf]
    amax = max(abs(v) for v in xs)
    if amax == 0:
        return np.zeros(len(xs), np.uint8), 0.0
    s = _rne_f32(Fraction(int(dmax)) / amax)
    prods = np.array([float(_rne_f32(v * s)) for v in xs], np.float32)
    codes = torch.from_numpy(prods).to(tdt).view(torch.uint8).numpy()
    return codes, float(_rne_f32(1 / s))


@pytest.mark.parametrize("mode", [oracle.Q_FP8T_E4M3, oracle.Q_FP8T_E5M2])
def test_fp8_token_exact_route(mode):
    rng = np.random.default_rng(31)
    for trial in range(25):
        x = bf16_bits((rng.standard_normal(96) * 10.0 ** rng.uniform(-6, 6)).astype(np.float32))
        codes, inv = oracle.quant_fp8_token_row(FP8[mode][0], x)
        wc, winv = _exact_fp8_row(x, mode)
        assert np.array_equal(codes, wc)
        assert float(inv) == winv
        # the largest element lands on the largest finite value
        assert np.max(np.abs(oracle.mini_decode(FP8[mode][0], codes))) == FP8[mode][1]


@pytest.mark.parametrize("mode", [oracle.Q_FP8G_E4M3, oracle.Q_FP8G_E5M2])
def test_fp8_group_exact_route(mode):
    rng = np.random.default_rng(32)
    for trial in range(8):
        H = 384
        x = bf16_bits((rng.standard_normal(H) * 10.0 ** rng.uniform(-3, 3, size=H)).astype(np.float32))
        x[128:256] = 0                                   # an all-zero group
        codes, inv = oracle.quant_fp8_group_row(FP8[mode][0], x)
        for g in range(3):
            wc, winv = _exact_fp8_row(x[g * 128:(g + 1) * 128], mode)
            assert np.array_equal(codes[g * 128:(g + 1) * 128], wc)
            assert float(inv[g]) == winv
        assert inv[1] == 0 and not codes[128:256].any()


def test_int8_static_exact_route():
    rng = np.random.default_rng(33)
    for trial in range(20):
        H = 64
        x = bf16_bits((rng.standard_normal(H) * 100).astype(np.float32))
        sc = (rng.standard_normal(H) * 2).astype(np.float32)
        q = oracle.quant_int8_static_row(x, sc)
        xf = (x.astype(np.uint32) << 16).view(np.float32)
        want = [max(-128, min(127, _rne_int(_rne_f32(Fraction(float(a)) * Fraction(float(b))))))
                for a, b in zip(xf, sc)]
        assert q.tolist() == want


@pytest.mark.parametrize("mode", [oracle.Q_INT8, oracle.Q_FP8T_E4M3, oracle.Q_FP8G_E5M2])
def test_smooth_scale_invariances(mode):
    # all-ones smooth scales change nothing; a uniform power of two leaves the codes and
    # multiplies the sent inverse scale by it (it dequantises the scaled row)
    rng = np.random.default_rng(34)
    x = bf16_bits((rng.standard_normal(256) * 3).astype(np.float32))
    d0, s0 = oracle.encode_row(mode, x)
    d1, s1 = oracle.encode_row(mode, x, np.ones(256, np.float32))
    assert np.array_equal(d0, d1) and np.array_equal(s0, s1)
    d2, s2 = oracle.encode_row(mode, x, np.full(256, 8.0, np.float32))
    assert np.array_equal(d0, d2)
    assert np.array_equal(s0.view(np.float32) * 8, s2.view(np.float32))


def test_smooth_scales_exact_route_fp8():
    rng = np.random.default_rng(35)
    x = bf16_bits((rng.standard_normal(128)).astype(np.float32))
    sm = (rng.random(128) * 4 + 0.1).astype(np.float32)
    codes, inv = oracle.quant_fp8_token_row(oracle.Q_E4M3, x, sm)
    wc, winv = _exact_fp8_row(x, oracle.Q_FP8T_E4M3, sm)
    assert np.array_equal(codes, wc) and float(inv) == winv


@pytest.mark.parametrize("mode", [oracle.Q_INT8_STATIC, oracle.Q_INT8, oracle.Q_FP8T_E4M3,
                                  oracle.Q_FP8G_E4M3])
def test_dispatch_per_expert_scales_pick_the_entrys_expert(mode):
    # scales[e] = 2^(e mod 3) uniformly: the row of entry (s,t,k) must be encoded with
    # the row of expert topk[s,t,k]
    w = synth.WORKLOADS[4].with_(T=6, H=256)
    topk = synth.gen_topk(w)
    x = synth.gen_x(w)
    lay = oracle.layout(w.R, w.T, w.E, w.K, w.alpha, topk)
    scales = np.repeat((2.0 ** (np.arange(w.E) % 3)).astype(np.float32)[:, None], w.H, axis=1)
    data, sc = oracle.dispatch_scaled(lay, x, mode, topk, scales, oracle.S_EXPERT)
    xs = x.reshape(w.N, w.H)
    tk = topk.reshape(w.N, w.K)
    for n in range(w.N):
        for k in range(w.K):
            e = int(tk[n, k])
            r = lay.dst_row.reshape(w.N, w.K)[n, k]
            d_ref, s_ref = oracle.encode_row(mode, xs[n], np.full(w.H, 2.0 ** (e % 3), np.float32))
            assert np.array_equal(data[r], d_ref)
            if sc.shape[1]:
                assert np.array_equal(sc[r], s_ref)
    # padding rows stay zero
    assert not data[lay.recv_src < 0].any()


@pytest.mark.parametrize("seed", range(12))
def test_masked_layout_matches_brute_force(seed):
    rng = np.random.default_rng(100 + seed)
    R, L = int(rng.integers(1, 4)), int(rng.integers(1, 4))
    E = R * L
    K = int(rng.integers(1, min(E, 3) + 1))
    T = int(rng.integers(1, 8))
    alpha = int(rng.integers(1, 4))
    topk = rng.integers(-1, E, size=(R, T, K))
    for dims in (1, 2):
        shape = (R, T) if dims == 1 else (R, T, K)
        mask = (rng.random(shape) < 0.6).astype(np.uint8)
        lay = oracle.layout(R, T, E, K, alpha, topk, mask=mask)
        sub = topk.copy()
        sub[(mask[..., None].repeat(K, -1) if dims == 1 else mask) == 0] = -1
        assert_layout_equal(lay, brute_layout(R, T, E, K, alpha, sub))
        if dims == 1:
            assert lay.is_token_in_rank[mask == 0].sum() == 0
