"""GPU parity at the edges of the parameter ranges: the most ranks (R = E =
512, one expert per rank, top-16), the most tokens per rank (T = 65536 on one
rank), the largest hidden size with MX, and the largest alignment.  Layout,
receive rows, per-rank layout and the two-phase form bit for bit; combine
within the derived tolerance."""
import numpy as np
import pytest
import torch

import oracle
from combine_ep_layout_03_gb300 import ep, synth
from gpu_harness import GpuPath, compare_layout, to_dev_bf16
from test_gpu_parity import check_combine, check_dispatch

pytestmark = pytest.mark.gpu

CASES = {
    "ranks512": (synth.Workload(400, R=512, T=4, H=64, E=512, K=16, alpha=1), 0),
    "tokens65536": (synth.Workload(401, R=1, T=65536, H=64, E=8, K=2, alpha=3), 0),
    "hidden8192_mx": (synth.Workload(402, R=2, T=40, H=8192, E=8, K=4, alpha=2), 4),
    "alpha4096": (synth.Workload(403, R=2, T=30, H=128, E=4, K=2, alpha=4096), 2),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_extreme_shapes(name):
    w, q = CASES[name]
    assert ep.ep_params_validate(ep.make_params(w.R, w.T, w.H, w.E, w.K, w.alpha, 0)) == ep.EP_OK
    topk = synth.gen_topk(w)
    wts = synth.gen_weights(w, topk)
    x = synth.gen_x(w)
    olay = oracle.layout(w.R, w.T, w.E, w.K, w.alpha, topk)
    g = GpuPath(w, topk)
    assert g.rows == olay.rows
    compare_layout(g.views_numpy(), olay)
    x_dev = to_dev_bf16(x)
    data, scales = g.dispatch(x_dev, q, fill=0x33)
    od, os_ = check_dispatch(g, olay, x, q, data, scales)
    y = g.expert(q, data, scales, 2)
    w_dev = torch.from_numpy(wts).cuda()
    out = g.combine(y, w_dev)
    tokens = np.unique(np.linspace(0, w.N - 1, min(w.N, 512)).astype(np.int64))
    check_combine(w, g, olay, x, wts, None, q, y, out, 2, tokens)
    # per-rank layout and the two-phase form on the same routing
    tl = oracle.token_layout(w.R, w.T, w.E, w.K, topk, wts)
    g.lay.token_layout(g.topk_dev, w_dev)
    assert int(g.lay.token_rows()[-1]) == tl.rows
    td, ts = g.lay.alloc_recv(q, max(tl.rows, 1))
    g.lay.dispatch_async(x_dev, q, td, ts)
    otd, _ = oracle.token_dispatch(tl, x, q)
    assert np.array_equal(td[: tl.rows].cpu().numpy(), otd)
    d2, s2 = g.lay.alloc_recv(q, max(olay.rows, 1))
    g.lay.dispatch_wait(q, td, ts, d2, s2)
    assert torch.equal(d2[: olay.rows], data[: olay.rows])
    ret = g.lay.alloc_return()
    g.lay.combine_async(y, ret)
    out2 = torch.empty_like(out)
    g.lay.combine_wait(ret, w_dev, out2)
    assert torch.equal(out2.view(torch.int16), out.view(torch.int16))
    assert g.lay.status() == ep.EP_OK
