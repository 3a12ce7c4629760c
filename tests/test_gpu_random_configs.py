"""GPU parity on randomly drawn small problems: rank counts, experts per rank,
top-k, tokens (including none), hidden sizes, alignments, routing (uniform or
Zipf), dropped entries, shared-expert rows and every quant mode that needs no
input scales, each drawn from a seed.  Layout, receive rows and stand-in
expert rows bit for bit; combine within the derived tolerance; the per-rank
layout's rows bit for bit as well.
"""
import numpy as np
import pytest
import torch

import oracle
from combine_ep_layout_03_gb300 import ep, synth
from gpu_harness import GpuPath, bf16_bits, compare_layout, to_dev_bf16
from test_gpu_parity import check_combine, check_dispatch

pytestmark = pytest.mark.gpu

MODES = (0, 2, 4, 5, 6, 7, 8, 9, 10)


def draw(seed):
    rng = np.random.default_rng(5000 + seed)
    R = int(rng.integers(1, 9))
    L = int(rng.integers(1, 7))
    E = R * L
    K = int(rng.integers(1, min(E, 8) + 1))
    T = int(rng.choice([0, 1, 7, 33, 64, 129]))
    q = int(rng.choice(MODES))
    if q in (9, 10):
        H = 128 * int(rng.integers(1, 5))
    elif q in (4, 5, 6):
        H = 32 * int(rng.integers(1, 20))
    else:
        H = 8 * int(rng.integers(1, 80))
    alpha = int(rng.choice([1, 2, 3, 8, 64]))
    routing = "zipf" if (rng.random() < 0.3 and K < E) else "uniform"
    drop = float(rng.choice([0.0, 0.0, 0.2, 0.9]))
    S = int(rng.choice([0, 0, 1, 3]))
    w = synth.Workload(200 + seed, R=R, T=T, H=H, E=E, K=K, alpha=alpha, routing=routing, drop_p=drop,
                       num_shared=S)
    return w, q


@pytest.mark.parametrize("seed", range(24))
def test_random_config(seed):
    w, q = draw(seed)
    topk = synth.gen_topk(w)
    wts = synth.gen_weights(w, topk)
    x = synth.gen_x(w)
    shared = synth.gen_shared(w)
    olay = oracle.layout(w.R, w.T, w.E, w.K, w.alpha, topk)
    g = GpuPath(w, topk)
    assert g.rows == olay.rows
    compare_layout(g.views_numpy(), olay)
    x_dev = to_dev_bf16(x) if w.N else torch.empty((0, w.H), dtype=torch.bfloat16, device="cuda")
    data, scales = g.dispatch(x_dev, q, fill=0x77)
    od, os_ = check_dispatch(g, olay, x, q, data, scales)
    y = g.expert(q, data, scales, 8)
    oy = oracle.expert_rows(olay, np.arange(olay.rows), w.H, q, od, os_, 8)
    assert np.array_equal(bf16_bits(y[: olay.rows]), oy)
    if w.N:
        sh_dev = None if shared is None else to_dev_bf16(shared)
        out = g.combine(y, torch.from_numpy(wts).cuda(), sh_dev)
        check_combine(w, g, olay, x, wts, shared, q, y, out, 8)
    assert g.lay.status() == ep.EP_OK
    # the per-rank layout of the same routing
    tl = oracle.token_layout(w.R, w.T, w.E, w.K, topk, wts)
    ridx, rw = g.lay.token_layout(g.topk_dev, torch.from_numpy(wts).cuda())
    assert int(g.lay.token_rows()[-1]) == tl.rows
    td, ts = g.lay.alloc_recv(q, max(tl.rows, 1))
    g.lay.dispatch_tokens(x_dev, q, td, ts)
    otd, ots = oracle.token_dispatch(tl, x, q)
    assert np.array_equal(td[: tl.rows].cpu().numpy(), otd)
    if ots.shape[1]:
        assert np.array_equal(ts[: tl.rows].cpu().numpy(), ots)
    assert g.lay.status() == ep.EP_OK
