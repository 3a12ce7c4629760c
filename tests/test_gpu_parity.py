"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Bit-exact: every layout array, receive order, receive rows, int8/fp8/fp4 codes
and scales, the stand-in expert's bf16 rows.  Combine: within the tolerance
derived from the arithmetic (2 bf16 ulp + (2K+S+1) 2^-24 sum|terms| per
element; max relative error 1e-2 where |ref| >= 2^-10 sum|terms|).

Sizes: reduced-T copies of the five workloads (several layout tiles and a
ragged tail, all outputs compared), ragged hidden sizes, and the edge cases.
Full-size workloads are in test_gpu_fullsize.py.
"""
import numpy as np
import pytest
import torch

import oracle
from combine_ep_layout_03_gb300 import synth
from gpu_harness import (GpuPath, bf16_bits, compare_layout, oracle_combine_sampled, to_dev_bf16)

pytestmark = pytest.mark.gpu

QUANTS = {1: (0,), 2: (0,), 3: (2,), 4: (4, 5, 6), 5: (0,)}


def reduced(idx, T):
    return synth.WORKLOADS[idx].with_(T=T)


def inputs(w):
    topk = synth.gen_topk(w)
    wts = synth.gen_weights(w, topk)
    x = synth.gen_x(w)
    shared = synth.gen_shared(w)
    return topk, wts, x, shared


def check_dispatch(g, olay, x, q, data, scales):
    od, os_ = oracle.dispatch(olay, x, q)
    gd = data[: olay.rows].cpu().numpy()
    assert np.array_equal(gd, od), "receive rows differ"
    if os_.shape[1]:
        gs = scales[: olay.rows].cpu().numpy()
        assert np.array_equal(gs, os_), "receive scales differ"
    return od, os_


def check_combine(w, g, olay, x, wts, shared, q, y, out, mark_mod, tokens=None):
    if tokens is None:
        tokens = np.arange(w.N)
    sh_tok = None
    if shared is not None:
        sh = shared.transpose(0, 2, 1, 3).reshape(w.N, w.num_shared, w.H)
        sh_tok = sh[tokens]
    o, ref, mag = oracle_combine_sampled(olay, x.reshape(w.N, w.H), wts, sh_tok, q, mark_mod, tokens)
    got = bf16_bits(out)[tokens]
    ok, excess, rel = oracle.combine_within_tolerance(got, ref, mag, w.K, w.num_shared)
    assert ok, (excess, rel)
    # the oracle's own float32 result is within the same bound
    ok2, _, _ = oracle.combine_within_tolerance(o, ref, mag, w.K, w.num_shared)
    assert ok2
    return o, got


@pytest.mark.parametrize("idx,T", [(1, 64), (2, 333), (3, 150), (4, 201), (5, 97)])
def test_layout_dispatch_combine_reduced(idx, T):
    w = reduced(idx, T)
    topk, wts, x, shared = inputs(w)
    olay = oracle.layout(w.R, w.T, w.E, w.K, w.alpha, topk)
    g = GpuPath(w, topk)
    assert g.rows == olay.rows
    compare_layout(g.views_numpy(), olay)
    assert g.lay.status() == 0
    x_dev = to_dev_bf16(x)
    wts_dev = torch.from_numpy(wts).cuda()
    sh_dev = None if shared is None else to_dev_bf16(shared)
    for q in QUANTS[idx]:
        data, scales = g.dispatch(x_dev, q, fill=0xA5)
        od, os_ = check_dispatch(g, olay, x, q, data, scales)
        for mark in (0, 16):
            y = g.expert(q, data, scales, mark)
            oy = oracle.expert_rows(olay, np.arange(olay.rows), w.H, q, od, os_, mark)
            assert np.array_equal(bf16_bits(y[: olay.rows]), oy), "stand-in expert rows differ"
            out = g.combine(y, wts_dev, sh_dev)
            check_combine(w, g, olay, x, wts, shared, q, y, out, mark)
        assert g.lay.status() == 0


@pytest.mark.parametrize("H,q", [(1000, 0), (1000, 2), (1056, 4), (1056, 6), (8, 0), (8, 2),
                                 (32, 5), (8192, 0), (8192, 4)])
def test_ragged_and_extreme_hidden(H, q):
    w = synth.Workload(11, R=4, T=50, H=H, E=16, K=3, alpha=4)
    topk, wts, x, _ = inputs(w)
    olay = oracle.layout(w.R, w.T, w.E, w.K, w.alpha, topk)
    g = GpuPath(w, topk)
    compare_layout(g.views_numpy(), olay)
    data, scales = g.dispatch(to_dev_bf16(x), q, fill=0x5A)
    od, os_ = check_dispatch(g, olay, x, q, data, scales)
    y = g.expert(q, data, scales, 4)
    out = g.combine(y, torch.from_numpy(wts).cuda())
    check_combine(w, g, olay, x, wts, None, q, y, out, 4)


def test_random_expert_outputs_combine():
    # combine on an independent y (every slot distinct), not built by dispatch
    w = reduced(2, 128)
    topk, wts, _, _ = inputs(w)
    olay = oracle.layout(w.R, w.T, w.E, w.K, w.alpha, topk)
    g = GpuPath(w, topk)
    y_bits = synth.gen_y(w, olay.rows)
    out = g.combine(to_dev_bf16(y_bits), torch.from_numpy(wts).cuda())
    o = oracle.combine(olay, y_bits, wts)
    ref, mag = oracle.combine_ref64(olay, y_bits, wts)
    ok, excess, rel = oracle.combine_within_tolerance(bf16_bits(out), ref, mag, w.K)
    assert ok, (excess, rel)
    # most elements agree with the oracle's float32 result exactly
    assert np.mean(bf16_bits(out) == o) > 0.95


def test_edge_tokens_without_experts_and_shared_only():
    w = synth.Workload(12, R=2, T=40, H=256, E=8, K=4, alpha=8, num_shared=3, drop_p=0.5)
    topk, wts, x, shared = inputs(w)
    topk[0, :5] = -1          # tokens with no expert at all
    wts = synth.gen_weights(w, topk)
    olay = oracle.layout(w.R, w.T, w.E, w.K, w.alpha, topk)
    g = GpuPath(w, topk)
    compare_layout(g.views_numpy(), olay)
    assert g.views_numpy()["is_token_in_rank"][0, :5].sum() == 0
    data, scales = g.dispatch(to_dev_bf16(x), 0)
    check_dispatch(g, olay, x, 0, data, scales)
    y = g.expert(0, data, scales, 8)
    out = g.combine(y, torch.from_numpy(wts).cuda(), to_dev_bf16(shared))
    check_combine(w, g, olay, x, wts, shared, 0, y, out, 8)


def test_edge_T0_and_all_invalid():
    w = synth.Workload(13, R=3, T=0, H=64, E=6, K=2, alpha=4)
    topk = np.zeros((3, 0, 2), np.int64)
    g = GpuPath(w, topk)
    assert g.rows == 0 and g.lay.status() == 0
    v = g.views_numpy()
    assert np.all(v["expert_start"] == 0) and np.all(v["rank_base"] == 0)
    data, scales = g.dispatch(torch.empty((0, 64), dtype=torch.bfloat16, device="cuda"), 0, rows=1)
    out = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    g.lay.combine(data.view(torch.bfloat16).view(1, 64), torch.empty(0, device="cuda"), out)
    assert g.lay.status() == 0
    w = synth.Workload(14, R=2, T=7, H=64, E=4, K=2, alpha=3)
    topk = -np.ones((2, 7, 2), np.int64)
    olay = oracle.layout(2, 7, 4, 2, 3, topk)
    g = GpuPath(w, topk)
    compare_layout(g.views_numpy(), olay)
    assert g.rows == 0


def test_edge_alignment_larger_than_counts_L1_K1():
    for (R, E, K, alpha) in [(4, 4, 1, 64), (3, 3, 1, 1), (2, 8, 1, 7), (1, 5, 5, 2)]:
        w = synth.Workload(15, R=R, T=37, H=128, E=E, K=K, alpha=alpha)
        topk, wts, x, _ = inputs(w)
        olay = oracle.layout(R, w.T, E, K, alpha, topk)
        g = GpuPath(w, topk)
        compare_layout(g.views_numpy(), olay)
        data, scales = g.dispatch(to_dev_bf16(x), 2)
        check_dispatch(g, olay, x, 2, data, scales)


def test_edge_zipf_extreme_skew_all_to_expert0():
    w = synth.Workload(16, R=4, T=300, H=512, E=32, K=1, alpha=128)
    topk = np.zeros((4, 300, 1), np.int64)
    topk[1, 7, 0] = 31
    olay = oracle.layout(4, 300, 32, 1, 128, topk)
    g = GpuPath(w, topk)
    compare_layout(g.views_numpy(), olay)
    x = synth.gen_x(w)
    data, scales = g.dispatch(to_dev_bf16(x), 4)
    check_dispatch(g, olay, x, 4, data, scales)


def test_zero_rows_and_special_blocks_quant():
    # all-zero tokens, all-zero MX blocks, subnormal blocks, ties, saturation
    w = synth.Workload(17, R=2, T=6, H=64, E=4, K=2, alpha=1)
    topk = np.array([[[0, 1], [2, 3], [1, 2], [0, 3], [3, 1], [2, 0]]] * 2, np.int64)
    xf = np.zeros((12, 64), np.float32)
    xf[1, :4] = [1.0, 0.5, -0.25, -0.296875]
    xf[2, :32] = 2.0 ** -130                        # subnormal block
    xf[2, 32] = -2.0 ** -18
    xf[3, :] = np.linspace(-1.9375, 1.9375, 64)
    xf[4, :3] = [2.0, 1.0, 0.625]
    xf[5, 32:] = -0.0625                             # rounds to -0 in e2m1
    xf[6:] = np.random.default_rng(0).standard_normal((6, 64)) * 1e-3
    x = torch.from_numpy(xf).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).reshape(2, 6, 64)
    olay = oracle.layout(2, 6, 4, 2, 1, topk)
    g = GpuPath(w, topk)
    for q in (2, 4, 5, 6):
        data, scales = g.dispatch(to_dev_bf16(x), q)
        check_dispatch(g, olay, x, q, data, scales)


def test_bad_expert_id_sets_status_and_counts_as_invalid():
    w = synth.Workload(18, R=2, T=20, H=64, E=4, K=2, alpha=1)
    topk, wts, x, _ = inputs(w)
    topk[0, 3, 1] = 9
    topk[1, 5, 0] = -7
    olay = oracle.layout(2, 20, 4, 2, 1, topk)
    assert olay.status == 4
    g = GpuPath(w, topk)
    assert g.lay.status() == 4
    compare_layout(g.views_numpy(), olay)


def test_capacity_overflow_writes_nothing():
    w = synth.Workload(19, R=2, T=30, H=64, E=4, K=2, alpha=1)
    topk, wts, x, _ = inputs(w)
    olay = oracle.layout(2, 30, 4, 2, 1, topk)
    # layout capacity below the rows needed
    g = GpuPath(w, topk, recv_capacity_rows=olay.rows - 3)
    assert g.lay.status() == 3
    # dispatch / combine capacity below the rows needed: buffers untouched
    g = GpuPath(w, topk)
    data, scales = g.dispatch(to_dev_bf16(x), 2, rows=olay.rows - 1, fill=0x77)
    assert g.lay.status() == 3
    assert torch.all(data == 0x77) and torch.all(scales == 0x77)
    g = GpuPath(w, topk)
    y = torch.zeros((olay.rows - 1, 64), dtype=torch.bfloat16, device="cuda")
    out = torch.full((60, 64), 3.0, dtype=torch.bfloat16, device="cuda")
    g.lay.combine(y, torch.from_numpy(wts).cuda(), out)
    assert g.lay.status() == 3 and torch.all(out == 3.0)


def test_deterministic_across_runs():
    w = reduced(3, 200)
    topk, wts, x, _ = inputs(w)
    res = []
    for _ in range(2):
        g = GpuPath(w, topk)
        data, scales = g.dispatch(to_dev_bf16(x), 2)
        y = g.expert(2, data, scales, 0)
        out = g.combine(y, torch.from_numpy(wts).cuda())
        res.append((g.views_numpy()["dst_row"].copy(), data.cpu().numpy(), bf16_bits(out)))
    for a, b in zip(res[0], res[1]):
        assert np.array_equal(a, b)
