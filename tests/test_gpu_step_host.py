"""One step from pinned host buffers through the C ABI (ep_step_host): the
host output equals, bit for bit, the device path's output for the same
inputs (layout, dispatch and combine called one by one), and is within the
derived tolerance of the oracle; two steps on two streams with two handles
give the same results as one after the other."""
import numpy as np
import pytest
import torch

import oracle
from combine_ep_layout_03_gb300 import ep, synth
from gpu_harness import to_dev_bf16
from test_gpu_parity import check_combine

pytestmark = pytest.mark.gpu


def pinned(a: np.ndarray, dtype=None) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.pin_memory()


def setup(w, q):
    lay = ep.EPLayout(w.R, w.T, w.H, w.E, w.K, w.alpha)
    data, scales = lay.alloc_recv(q)
    dev = dict(topk=torch.empty((w.R, w.T, w.K), dtype=torch.int64, device="cuda"),
               w=torch.empty((w.R, w.T, w.K), dtype=torch.float32, device="cuda"),
               x=torch.empty((w.N, w.H), dtype=torch.bfloat16, device="cuda"),
               sh=None if not w.num_shared else
               torch.empty((w.R, w.num_shared, w.T, w.H), dtype=torch.bfloat16, device="cuda"),
               out=torch.empty((w.N, w.H), dtype=torch.bfloat16, device="cuda"),
               data=data, scales=scales)
    return lay, dev


@pytest.mark.parametrize("idx,T,q", [(1, 64, 0), (5, 10, 0), (4, 40, 4)])
def test_step_from_host_buffers(idx, T, q):
    w = synth.WORKLOADS[idx].with_(T=T)
    topk = synth.gen_topk(w)
    wts = synth.gen_weights(w, topk)
    x = synth.gen_x(w)
    shared = synth.gen_shared(w)
    lay, dev = setup(w, q)
    y = None
    if q != 0:
        # stand-in expert outputs built once on the device path
        lay.layout(torch.from_numpy(topk).cuda())
        d0, s0 = lay.alloc_recv(q)
        lay.dispatch(to_dev_bf16(x).view(w.N, w.H), q, d0, s0)
        y = torch.empty((d0.shape[0], w.H), dtype=torch.bfloat16, device="cuda")
        lay.expert_identity(q, d0, s0, y, 4)
    bufs = ep.step_buffers(dev["topk"], dev["w"], dev["x"], dev["out"], dev["data"], dev["scales"],
                           dev["sh"], y, w.H)
    topk_h, w_h = pinned(topk), pinned(wts)
    x_h = pinned(x.view(np.int16), None).view(torch.bfloat16)
    sh_h = None if shared is None else pinned(shared.view(np.int16)).view(torch.bfloat16)
    out_h = torch.empty((w.N, w.H), dtype=torch.bfloat16).pin_memory()
    s = torch.cuda.Stream()
    ep.ep_step_host(lay.h, q, topk_h, w_h, x_h, sh_h, w.num_shared, out_h, bufs, s)
    s.synchronize()
    assert lay.status() == ep.EP_OK
    # the device path, call by call
    ref_out = torch.empty((w.N, w.H), dtype=torch.bfloat16, device="cuda")
    lay.layout(torch.from_numpy(topk).cuda())
    d1, s1 = lay.alloc_recv(q)
    lay.dispatch(to_dev_bf16(x).view(w.N, w.H), q, d1, s1)
    yy = y if y is not None else d1.view(torch.bfloat16).view(-1, w.H)
    lay.combine(yy, torch.from_numpy(wts).cuda(), ref_out, None if shared is None else to_dev_bf16(shared))
    assert torch.equal(out_h.cuda().view(torch.int16), ref_out.view(torch.int16))
    olay = oracle.layout(w.R, w.T, w.E, w.K, w.alpha, topk)
    check_combine(w, None, olay, x, wts, shared, q, yy, ref_out, 4 if q else 0,
                  np.unique(np.linspace(0, w.N - 1, min(w.N, 256)).astype(np.int64)))


def test_two_streams_two_handles():
    w = synth.WORKLOADS[1]
    steps = []
    for seed in range(4):
        v = w.with_(index=500 + seed)
        topk = synth.gen_topk(v)
        steps.append((pinned(topk), pinned(synth.gen_weights(v, topk)),
                      pinned(synth.gen_x(v).view(np.int16)).view(torch.bfloat16),
                      torch.empty((w.N, w.H), dtype=torch.bfloat16).pin_memory()))
    slots = [setup(w, 0) for _ in range(2)]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for i, (t, wt, x, o) in enumerate(steps):
        lay, dev = slots[i % 2]
        bufs = ep.step_buffers(dev["topk"], dev["w"], dev["x"], dev["out"], dev["data"], None)
        if i >= 2:
            streams[i % 2].synchronize()   # the slot's previous step is done before its buffers are reused
        ep.ep_step_host(lay.h, 0, t, wt, x, None, 0, o, bufs, streams[i % 2])
    torch.cuda.synchronize()
    lay, dev = setup(w, 0)
    for t, wt, x, o in steps:
        bufs = ep.step_buffers(dev["topk"], dev["w"], dev["x"], dev["out"], dev["data"], None)
        ref = torch.empty_like(o).pin_memory()
        ep.ep_step_host(lay.h, 0, t, wt, x, None, 0, ref, bufs, None)
        torch.cuda.synchronize()
        assert torch.equal(ref.view(torch.int16), o.view(torch.int16))
