"""The bounded mbarrier waits of the bulk-copy kernels end with a status code
instead of hanging (failure detection without a GPU fault).

The combine is run through its test hook with a producer warp that issues
nothing, so every consumer wait on a stage runs out after a small poll limit;
the status word must read EP_ERR_TIMEOUT, the output must be untouched, the
launch must end quickly, and the context must stay usable: the next layout
clears the status word and a normal combine gives the right result.
"""
import time

import numpy as np
import pytest
import torch

import oracle
from combine_ep_layout_03_gb300 import ep, synth
from gpu_harness import bf16_bits, to_dev_bf16

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("polls", [1, 64, 1024])
def test_stalled_producer_times_out_and_context_survives(polls):
    w = synth.WORKLOADS[1].with_(H=256)
    topk = synth.gen_topk(w)
    wts = synth.gen_weights(w, topk)
    x = synth.gen_x(w)
    lay = ep.EPLayout(w.R, w.T, w.H, w.E, w.K, w.alpha)
    topk_d = torch.from_numpy(topk).cuda()
    w_d = torch.from_numpy(wts).cuda()
    lay.layout(topk_d)
    rows = int(lay.recv_rows()[-1])
    data, _ = lay.alloc_recv(0, rows)
    lay.dispatch(to_dev_bf16(x), 0, data, None)
    y = data.view(torch.bfloat16).view(rows, w.H)
    out = torch.full((w.N, w.H), 7.0, dtype=torch.bfloat16, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    ep.ep_test_combine_stalled(lay.h, y, rows, w_d, out, polls)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert lay.status() == ep.EP_ERR_TIMEOUT
    assert torch.all(out == 7.0), "a timed-out combine wrote output"
    assert elapsed < 10.0, f"{polls} polls took {elapsed:.3f} s"
    print(f"stalled combine, {polls} polls per wait: {elapsed * 1e3:.3f} ms")
    # the context is usable and the next layout starts from a clean status word
    lay.layout(topk_d)
    assert lay.status() == ep.EP_OK
    lay.combine(y, w_d, out)
    assert lay.status() == ep.EP_OK
    olay = oracle.layout(w.R, w.T, w.E, w.K, w.alpha, topk)
    od, _ = oracle.dispatch(olay, x, 0)
    ref, mag = oracle.combine_ref64(olay, od.view(np.uint16).reshape(-1, w.H), wts)
    ok, excess, rel = oracle.combine_within_tolerance(bf16_bits(out), ref, mag, w.K, 0)
    assert ok, (excess, rel)
