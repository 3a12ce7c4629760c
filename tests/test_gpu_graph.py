"""The path's launches can be captured in a CUDA graph and replayed: layout,
dispatch, stand-in expert and combine of one step are captured once, then
replayed with new routing, weights and rows copied into the captured input
buffers; every replay must equal, bit for bit, the same calls made directly
(the path is deterministic), and the layout must match the oracle."""
import numpy as np
import pytest
import torch

import oracle
from combine_ep_layout_03_gb300 import ep, synth
from gpu_harness import to_dev_bf16

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("q", [0, 4])
def test_step_replays_in_a_cuda_graph(q):
    w = synth.WORKLOADS[1].with_(H=512)
    lay = ep.EPLayout(w.R, w.T, w.H, w.E, w.K, w.alpha)
    topk_in = torch.empty((w.R, w.T, w.K), dtype=torch.int64, device="cuda")
    w_in = torch.empty((w.R, w.T, w.K), dtype=torch.float32, device="cuda")
    x_in = torch.empty((w.N, w.H), dtype=torch.bfloat16, device="cuda")
    data, scales = lay.alloc_recv(q)
    y = torch.empty((data.shape[0], w.H), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((w.N, w.H), dtype=torch.bfloat16, device="cuda")

    def step(s=None):
        lay.layout(topk_in, s)
        lay.dispatch(x_in, q, data, scales, s)
        lay.expert_identity(q, data, scales, y, 4, stream=s)
        lay.combine(y, w_in, out, None, s)

    def load(seed):
        v = w.with_(index=300 + seed)
        topk = synth.gen_topk(v)
        topk_in.copy_(torch.from_numpy(topk))
        w_in.copy_(torch.from_numpy(synth.gen_weights(v, topk)))
        x_in.copy_(to_dev_bf16(synth.gen_x(v)).view(w.N, w.H))
        return topk

    load(0)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step(s)                       # warm-up outside capture (first-call setup)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for seed in (1, 2, 3):
        topk = load(seed)
        g.replay()
        torch.cuda.synchronize()
        assert lay.status() == ep.EP_OK
        got_out, got_data = out.clone(), data.clone()
        step()
        torch.cuda.synchronize()
        assert torch.equal(got_out.view(torch.int16), out.view(torch.int16))
        assert torch.equal(got_data, data)
        olay = oracle.layout(w.R, w.T, w.E, w.K, w.alpha, topk)
        assert np.array_equal(lay.views()["dst_row"].cpu().numpy().reshape(olay.dst_row.shape), olay.dst_row)
