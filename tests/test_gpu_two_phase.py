"""GPU parity for the two-phase dispatch and combine (Modular MAX
EPBatchManager ep_dispatch_async / ep_dispatch_wait, ep_combine_async /
ep_combine_wait) against the oracle.

Bit for bit: the arrival rows against the oracle's per-rank dispatch, the
expanded grouped rows against the oracle's dispatch (and the one-call GPU
dispatch), the return slots against the oracle's slots of its own expert
outputs, and the wait-phase combine against the one-call GPU combine (same
float32 order).  The combine is also within the derived tolerance of the
oracle's float64 sum.
"""
import numpy as np
import pytest
import torch

import oracle
from combine_ep_layout_03_gb300 import ep, synth
from gpu_harness import bf16_bits, for_row_chunks, to_dev_bf16

pytestmark = pytest.mark.gpu

MX = (ep.EP_QUANT_MXFP8_E4M3, ep.EP_QUANT_MXFP8_E5M2, ep.EP_QUANT_MXFP4_E2M1)


def run_two_phase(w, q, block_major=False, mark=4):
    topk = synth.gen_topk(w)
    wts = synth.gen_weights(w, topk)
    x = synth.gen_x(w)
    shared = synth.gen_shared(w)
    olay = oracle.layout(w.R, w.T, w.E, w.K, w.alpha, topk)
    tl = oracle.token_layout(w.R, w.T, w.E, w.K, topk, wts)
    lay = ep.EPLayout(w.R, w.T, w.H, w.E, w.K, w.alpha)
    topk_d = torch.from_numpy(topk).cuda()
    w_d = torch.from_numpy(wts).cuda()
    lay.layout(topk_d)
    lay.token_layout(topk_d, w_d)
    rows, trows = int(lay.recv_rows()[-1]), int(lay.token_rows()[-1])
    assert (rows, trows) == (olay.rows, tl.rows)
    x_d = to_dev_bf16(x)
    # send: arrival rows of the per-rank layout
    td, ts = lay.alloc_recv(q, max(trows, 1))
    lay.dispatch_async(x_d, q, td, ts)
    otd, ots = oracle.token_dispatch(tl, x, q)
    assert np.array_equal(td[:trows].cpu().numpy(), otd)
    if ots.shape[1]:
        assert np.array_equal(ts[:trows].cpu().numpy(), ots)
    # wait: grouped rows
    alloc = lay.alloc_recv_block_major if block_major else lay.alloc_recv
    data, scales = alloc(q, max(rows, 1))
    data.fill_(0x6B)
    if scales is not None:
        scales.fill_(0x6B)
    lay.dispatch_wait(q, td, ts, data, scales, block_major=block_major)
    assert lay.status() == ep.EP_OK
    od, os_ = oracle.dispatch(olay, x, q)
    os_rm = os_
    assert np.array_equal(data[:rows].cpu().numpy(), od)
    if os_.shape[1]:
        if block_major:
            es = 1 if q in MX else 4
            os_ = oracle.transpose_scales(os_, max(rows, 1), es)
            assert np.array_equal(scales.cpu().numpy()[:, : rows * es], os_[:, : rows * es])
        else:
            assert np.array_equal(scales[:rows].cpu().numpy(), os_)
    # the one-call dispatch writes the same bytes
    fd, fs = lay.alloc_recv_block_major(q, max(rows, 1)) if block_major else lay.alloc_recv(q, max(rows, 1))
    lay.dispatch_ex(x_d, q, fd, fs, block_major=block_major)
    assert torch.equal(fd[:rows], data[:rows])
    # stand-in expert, combine send and wait
    y = torch.empty((max(rows, 1), w.H), dtype=torch.bfloat16, device="cuda")
    if block_major and scales is not None:
        # the stand-in expert reads row-major scales
        rd, rs = lay.alloc_recv(q, max(rows, 1))
        lay.dispatch(x_d, q, rd, rs)
        lay.expert_identity(q, rd, rs, y, mark)
    else:
        lay.expert_identity(q, data, scales, y, mark)
    oy = oracle.expert_rows(olay, np.arange(rows, dtype=np.int64), w.H, q, od, os_rm, mark)
    assert np.array_equal(bf16_bits(y[:rows]), oy)
    ret = lay.alloc_return()
    lay.combine_async(y, ret)
    slots, valid = oracle.return_slots(olay, oy)
    got = bf16_bits(ret[: w.N * w.K])
    assert np.array_equal(got[valid], slots[valid])
    sh_d = None if shared is None else to_dev_bf16(shared)
    out = torch.empty((w.N, w.H), dtype=torch.bfloat16, device="cuda")
    lay.combine_wait(ret, w_d, out, sh_d)
    ref_out = torch.empty_like(out)
    lay.combine(y, w_d, ref_out, sh_d)
    assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
    ref, mag = oracle.combine_ref64(olay, oy, wts, shared)
    ok, excess, rel = oracle.combine_within_tolerance(bf16_bits(out), ref, mag, w.K, w.num_shared)
    assert ok, (excess, rel)
    assert lay.status() == ep.EP_OK


@pytest.mark.parametrize("idx,T,q,bm", [(1, 64, 0, False), (1, 64, 4, False), (1, 64, 6, True),
                                         (3, 24, 2, False), (4, 40, 4, True), (4, 40, 9, True),
                                         (5, 8, 0, False), (2, 16, 7, False)])
def test_two_phase_against_oracle(idx, T, q, bm):
    w = synth.WORKLOADS[idx].with_(T=T)
    if idx == 1:
        w = w.with_(H=1024, alpha=4)
    run_two_phase(w, q, bm)


def test_edges():
    # all entries -1: no arrival rows, no grouped rows, shared rows only
    run_two_phase(synth.WORKLOADS[5].with_(T=6, drop_p=1.0), 0)
    # grouped buffer too small: capacity error, nothing written
    w = synth.WORKLOADS[1].with_(H=256)
    topk = synth.gen_topk(w)
    lay = ep.EPLayout(w.R, w.T, w.H, w.E, w.K, w.alpha)
    topk_d = torch.from_numpy(topk).cuda()
    lay.layout(topk_d)
    lay.token_layout(topk_d, torch.from_numpy(synth.gen_weights(w, topk)).cuda())
    rows, trows = int(lay.recv_rows()[-1]), int(lay.token_rows()[-1])
    td, _ = lay.alloc_recv(0, trows)
    lay.dispatch_async(to_dev_bf16(synth.gen_x(w)), 0, td, None)
    data, _ = lay.alloc_recv(0, rows - 1)
    data.fill_(9)
    lay.dispatch_wait(0, td, None, data, None)
    assert lay.status() == ep.EP_ERR_CAPACITY
    assert torch.all(data == 9)


def _same(dev_rows, expected):
    assert np.array_equal(dev_rows.cpu().numpy(), expected)


def test_full_size_workload2_two_phase_equals_one_call():
    """Workload 2 at full size in the two-phase form (the bench's key 2a): every
    arrival row and grouped row against the oracle, and both phases' results
    equal to the one-call dispatch and combine bit for bit."""
    w = synth.WORKLOADS[2]
    topk = synth.gen_topk(w)
    wts = synth.gen_weights(w, topk)
    lay = ep.EPLayout(w.R, w.T, w.H, w.E, w.K, w.alpha)
    topk_d = torch.from_numpy(topk).cuda()
    w_d = torch.from_numpy(wts).cuda()
    lay.layout(topk_d)
    lay.token_layout(topk_d, w_d)
    rows, trows = int(lay.recv_rows()[-1]), int(lay.token_rows()[-1])
    x_d = synth.gen_x_device(w)
    td, _ = lay.alloc_recv(0, trows)
    lay.dispatch_async(x_d, 0, td, None)
    data, _ = lay.alloc_recv(0, rows)
    lay.dispatch_wait(0, td, None, data, None)
    torch.cuda.synchronize()
    # every arrival row (per-rank layout) and every grouped row against the oracle
    olay = oracle.layout(w.R, w.T, w.E, w.K, w.alpha, topk)
    tl = oracle.token_layout(w.R, w.T, w.E, w.K, topk, wts)
    assert olay.rows == rows and tl.rows == trows
    xb = np.ascontiguousarray(x_d.view(torch.int16).cpu().numpy()).view(np.uint8).reshape(w.N, -1)
    for_row_chunks(trows, lambda a, b: _same(td[a:b], oracle.dispatch_bytes(tl, xb, rows=b, row_begin=a)))
    for_row_chunks(rows, lambda a, b: _same(data[a:b], oracle.dispatch_bytes(olay, xb, rows=b, row_begin=a)))
    del td
    ref, _ = lay.alloc_recv(0, rows)
    lay.dispatch(x_d, 0, ref, None)
    assert torch.equal(data, ref)
    del ref
    y = data.view(torch.bfloat16).view(rows, w.H)
    ret = lay.alloc_return()
    lay.combine_async(y, ret)
    out = torch.empty((w.N, w.H), dtype=torch.bfloat16, device="cuda")
    lay.combine_wait(ret, w_d, out)
    one = torch.empty_like(out)
    lay.combine(y, w_d, one)
    assert torch.equal(out.view(torch.int16), one.view(torch.int16))
    assert lay.status() == ep.EP_OK
