"""Pins for the oracle's dispatch and combine (CPU only).

Dispatch (CANN aclnnMoeDistributeDispatchV2, quantMode 0: the receive buffer is
the all-to-all of X): every valid entry's receive row equals its source token's
row, padding rows are zero.  Checked against numpy fancy indexing driven by the
brute-force layout, not by the oracle's own layout.

Combine (DeepEP "Normal Mode API" combine: multiply by weights and sum; MAX
EPBatchManager.ep_combine: weighted sum of routed expert outputs, plus the fused
shared-expert outputs) is checked against closed forms computed straight from
(topk_idx, weights, x) in float64 with numpy, with no layout in between:
  - identity experts: out = x * sum_k w_k (+ sum_q shared);
  - marked experts y = x * 2^-(e mod M): out = x * sum_k w_k 2^-(e_k mod M),
    which exposes a gather from the wrong slot of the same token.
"""
import numpy as np
import pytest

import oracle
from combine_ep_layout_03_gb300 import synth
from test_oracle_layout import brute_layout


def f64(bits):
    return oracle.bf16_bits_to_f64(bits)


def small(idx, T):
    return synth.WORKLOADS[idx].with_(T=T)


@pytest.mark.parametrize("idx,T", [(1, 64), (2, 16), (5, 8)])
def test_dispatch_bf16_rows_are_source_rows(idx, T):
    w = small(idx, T)
    topk = synth.gen_topk(w)
    x = synth.gen_x(w)
    ref = brute_layout(w.R, w.T, w.E, w.K, w.alpha, topk)
    lay = oracle.layout(w.R, w.T, w.E, w.K, w.alpha, topk)
    data, _ = oracle.dispatch(lay, x, oracle.Q_NONE)
    rows = data.view(np.uint16).reshape(-1, w.H)
    rows_total = int(ref["rank_base"][-1])
    expect = np.zeros((rows_total, w.H), np.uint16)
    d = ref["dst_row"].reshape(-1)
    src = np.repeat(np.arange(w.N), w.K)
    ok = d >= 0
    expect[d[ok]] = x.reshape(w.N, w.H)[src[ok]]
    assert np.array_equal(rows, expect)


def test_dispatch_rank_slices_and_rows_agree():
    w = small(3, 32)
    topk = synth.gen_topk(w)
    x = synth.gen_x(w)
    lay = oracle.layout(w.R, w.T, w.E, w.K, w.alpha, topk)
    q = oracle.Q_INT8
    full_d, full_s = oracle.dispatch(lay, x, q)
    # rank-by-rank slices concatenate to the whole buffer
    parts = [oracle.dispatch(lay, x, q, int(lay.rank_base[j]), int(lay.rank_base[j + 1]))
             for j in range(w.R)]
    assert np.array_equal(np.concatenate([p[0] for p in parts]), full_d)
    assert np.array_equal(np.concatenate([p[1] for p in parts]), full_s)
    # row-by-row through recv_src gives the same bytes, padding included
    rows = np.arange(lay.rows)
    d2, s2 = oracle.dispatch_rows(lay, x, q, rows)
    assert np.array_equal(d2, full_d) and np.array_equal(s2, full_s)
    # each non-padding row is the quantised source row
    for r in np.random.default_rng(0).choice(lay.rows, 50, replace=False):
        src = lay.recv_src[r]
        if src < 0:
            assert not full_d[r].any() and not full_s[r].any()
        else:
            qq, inv = oracle.quant_int8_row(x.reshape(w.N, w.H)[src])
            assert np.array_equal(full_d[r].view(np.int8), qq)
            assert full_s[r].view(np.float32)[0] == inv


@pytest.mark.parametrize("q", [oracle.Q_E4M3, oracle.Q_E5M2, oracle.Q_E2M1])
def test_dispatch_mx_rows(q):
    w = small(4, 16)
    topk = synth.gen_topk(w)
    x = synth.gen_x(w)
    lay = oracle.layout(w.R, w.T, w.E, w.K, w.alpha, topk)
    data, scales = oracle.dispatch(lay, x, q)
    for r in range(lay.rows):
        src = lay.recv_src[r]
        if src < 0:
            assert not data[r].any() and not scales[r].any()
        else:
            c, s = oracle.quant_mx_row(q, x.reshape(w.N, w.H)[src])
            assert np.array_equal(data[r], c) and np.array_equal(scales[r], s)


def closed_form(w, topk, wts, x, shared, mark_mod=0):
    xf = f64(x.reshape(w.N, w.H))
    tk = topk.reshape(w.N, w.K)
    ww = wts.reshape(w.N, w.K).astype(np.float64)
    valid = tk >= 0
    mark = np.where(valid, 2.0 ** -(np.where(valid, tk, 0) % mark_mod) if mark_mod else 1.0, 0.0)
    coef = (ww * mark * valid).sum(axis=1)
    ref = xf * coef[:, None]
    mag = np.abs(xf) * (np.abs(ww) * mark * valid).sum(axis=1)[:, None]
    if shared is not None:
        sh = f64(shared).transpose(0, 2, 1, 3).reshape(w.N, w.num_shared, w.H)
        ref = ref + sh.sum(axis=1)
        mag = mag + np.abs(sh).sum(axis=1)
    return ref, mag


@pytest.mark.parametrize("idx,T,mark_mod", [(1, 64, 0), (1, 64, 4), (2, 16, 8), (5, 8, 16), (5, 8, 0)])
def test_combine_identity_and_marked_experts(idx, T, mark_mod):
    w = small(idx, T)
    topk = synth.gen_topk(w)
    wts = synth.gen_weights(w, topk)
    x = synth.gen_x(w)
    shared = synth.gen_shared(w)
    lay = oracle.layout(w.R, w.T, w.E, w.K, w.alpha, topk)
    data, scales = oracle.dispatch(lay, x, oracle.Q_NONE)
    y = oracle.expert_rows(lay, np.arange(lay.rows), w.H, oracle.Q_NONE, data, scales, mark_mod)
    out = oracle.combine(lay, y, wts, shared)
    ref, mag = closed_form(w, topk, wts, x, shared, mark_mod)
    ok, excess, rel = oracle.combine_within_tolerance(out, ref, mag, w.K, w.num_shared)
    assert ok, (excess, rel)
    # the oracle's own float64 sum is the same closed form
    r64, m64 = oracle.combine_ref64(lay, y, wts, shared)
    assert np.all(np.abs(r64 - ref) <= 1e-12 * mag)
    assert np.allclose(m64, mag, rtol=1e-12, atol=0.0)


def test_combine_random_expert_outputs_against_numpy():
    # independent random y: the gather must pick dst_row[s,t,k] for every slot
    w = small(2, 32)
    topk = synth.gen_topk(w)
    wts = synth.gen_weights(w, topk)
    ref_lay = brute_layout(w.R, w.T, w.E, w.K, w.alpha, topk)
    lay = oracle.layout(w.R, w.T, w.E, w.K, w.alpha, topk)
    y = synth.gen_y(w, lay.rows)
    out = oracle.combine(lay, y, wts)
    d = ref_lay["dst_row"].reshape(w.N, w.K)
    yf = f64(y)
    ww = wts.reshape(w.N, w.K).astype(np.float64)
    terms = np.where((d >= 0)[:, :, None], ww[:, :, None] * yf[np.maximum(d, 0)], 0.0)
    ref, mag = terms.sum(axis=1), np.abs(terms).sum(axis=1)
    ok, excess, rel = oracle.combine_within_tolerance(out, ref, mag, w.K)
    assert ok, (excess, rel)


def test_combine_accumulates_in_float32_order():
    # three terms whose float32 sum in slot order differs from the exact sum:
    # 1 + 2^-24 + 2^-24 in float32 (left to right) stays 1, exact is 1 + 2^-23.
    R, T, E, K, H = 1, 1, 4, 3, 8
    topk = np.array([[[0, 1, 2]]], np.int64)
    lay = oracle.layout(R, T, E, K, 1, topk)
    y = np.zeros((lay.rows, H), np.uint16)
    y[:, 0] = np.array([1.0, 2.0 ** -24, 2.0 ** -24], np.float32).view(np.uint32) >> 16
    wts = np.ones((1, 1, 3), np.float32)
    out = oracle.combine(lay, y, wts)
    assert f64(out)[0, 0] == 1.0
    ref, _ = oracle.combine_ref64(lay, y, wts)
    assert ref[0, 0] == 1.0 + 2.0 ** -23


def test_combine_token_without_experts_gets_shared_only():
    w = synth.Workload(9, R=2, T=3, H=8, E=4, K=2, alpha=1, num_shared=2)
    topk = np.array([[[0, 1], [-1, -1], [3, 2]], [[-1, -1], [2, 0], [1, -1]]], np.int64)
    wts = synth.gen_weights(w, topk)
    x = synth.gen_x(w)
    shared = synth.gen_shared(w)
    lay = oracle.layout(2, 3, 4, 2, 1, topk)
    data, scales = oracle.dispatch(lay, x, oracle.Q_NONE)
    y = oracle.expert_rows(lay, np.arange(lay.rows), w.H, 0, data, scales)
    out = f64(oracle.combine(lay, y, wts, shared))
    shf = f64(shared)
    # token (0,1) and (1,0) have no expert: output = bf16 sum of their shared rows
    assert np.array_equal(out[1], f64(oracle.bf16_from_f32((shf[0, 0, 1] + shf[0, 1, 1]).astype(np.float32))))
    assert np.array_equal(out[3], f64(oracle.bf16_from_f32((shf[1, 0, 0] + shf[1, 1, 0]).astype(np.float32))))


@pytest.mark.parametrize("q", [oracle.Q_INT8, oracle.Q_E4M3, oracle.Q_E2M1])
def test_expert_dequant_rows(q):
    # the stand-in expert reproduces the dequantised row: int8 q*inv, MX code*2^se
    w = small(3 if q == oracle.Q_INT8 else 4, 8)
    topk = synth.gen_topk(w)
    x = synth.gen_x(w)
    lay = oracle.layout(w.R, w.T, w.E, w.K, w.alpha, topk)
    rows = np.flatnonzero(lay.recv_src >= 0)[:20]
    data, scales = oracle.dispatch_rows(lay, x, q, rows)
    y = f64(oracle.expert_rows(lay, rows, w.H, q, data, scales))
    for i, r in enumerate(rows):
        if q == oracle.Q_INT8:
            v = data[i].view(np.int8).astype(np.float64) * float(scales[i].view(np.float32)[0])
            want = f64(oracle.bf16_from_f32(v.astype(np.float32)))
        else:
            if q == oracle.Q_E2M1:
                c = [(data[i][h // 2] >> (4 * (h % 2))) & 0xF for h in range(w.H)]
            else:
                c = data[i]
            se = np.repeat(scales[i].astype(np.int64) - 127, 32)
            want = oracle.mini_decode(q, c) * 2.0 ** se
        assert np.array_equal(y[i], want)
        # and it is close to the source row
        src = f64(x.reshape(w.N, w.H)[lay.recv_src[r]])
        tol = {oracle.Q_INT8: 1 / 127, oracle.Q_E4M3: 2 ** -3, oracle.Q_E2M1: 0.5}[q]
        amax = np.max(np.abs(src))
        assert np.max(np.abs(y[i] - src)) <= tol * amax * 1.01


@pytest.mark.parametrize("idx,q", [(5, oracle.Q_NONE), (3, oracle.Q_INT8), (4, oracle.Q_E2M1)])
def test_sampled_combine_matches_full_oracle(idx, q):
    # the GPU tests' one-token-at-a-time oracle path equals the whole-buffer path
    from gpu_harness import oracle_combine_sampled
    w = small(idx, 12)
    topk = synth.gen_topk(w)
    wts = synth.gen_weights(w, topk)
    x = synth.gen_x(w)
    shared = synth.gen_shared(w)
    lay = oracle.layout(w.R, w.T, w.E, w.K, w.alpha, topk)
    data, scales = oracle.dispatch(lay, x, q)
    y = oracle.expert_rows(lay, np.arange(lay.rows), w.H, q, data, scales, 8)
    full = oracle.combine(lay, y, wts, shared)
    tokens = np.array([0, 3, w.N - 1, w.N // 2])
    sh_tok = None
    if shared is not None:
        sh_tok = shared.transpose(0, 2, 1, 3).reshape(w.N, w.num_shared, w.H)[tokens]
    o, ref, mag = oracle_combine_sampled(lay, x.reshape(w.N, w.H), wts, sh_tok, q, 8, tokens)
    assert np.array_equal(o, full[tokens])


@pytest.mark.parametrize("q", [oracle.Q_INT8_STATIC, oracle.Q_E5M2, oracle.Q_FP8T_E4M3, oracle.Q_FP8T_E5M2,
                               oracle.Q_FP8G_E4M3, oracle.Q_FP8G_E5M2])
def test_expert_dequant_rows_more_modes(q):
    # the stand-in expert's decode for the further modes, with torch's float8 decode as
    # the independent route: code value (x the row's or group's 1/s), then bf16
    import torch
    w = small(4, 8)
    topk = synth.gen_topk(w)
    x = synth.gen_x(w)
    lay = oracle.layout(w.R, w.T, w.E, w.K, w.alpha, topk)
    rows = np.flatnonzero(lay.recv_src >= 0)[:16]
    if q == oracle.Q_INT8_STATIC:
        sc = synth.gen_scales(w, 2)
        data, scales = oracle.dispatch_scaled(lay, x, q, topk, sc, 2)
        data, scales = data[rows], scales[rows]
    else:
        data, scales = oracle.dispatch_rows(lay, x, q, rows)
    y = f64(oracle.expert_rows(lay, rows, w.H, q, data, scales))
    e5 = q in (oracle.Q_E5M2, oracle.Q_FP8T_E5M2, oracle.Q_FP8G_E5M2)
    dt = torch.float8_e5m2 if e5 else torch.float8_e4m3fn
    for i in range(len(rows)):
        if q == oracle.Q_INT8_STATIC:
            v = data[i].view(np.int8).astype(np.float32)
        else:
            codes = torch.from_numpy(data[i].copy()).view(dt).to(torch.float32).numpy()
            if q == oracle.Q_E5M2:
                mul = np.repeat(np.ldexp(1.0, scales[i].astype(np.int64) - 127), 32).astype(np.float32)
            elif q in (oracle.Q_FP8T_E4M3, oracle.Q_FP8T_E5M2):
                mul = np.full(w.H, scales[i].view(np.float32)[0], np.float32)
            else:
                mul = np.repeat(scales[i].view(np.float32), 128)
            v = (codes * mul).astype(np.float32)
        want = f64(oracle.bf16_from_f32(v))
        assert np.array_equal(y[i], want)
