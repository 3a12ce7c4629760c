"""GPU parity for the alternate formats of ep_dispatch_ex against the oracle.

- pre-encoded rows (DeepEP "Normal Mode API", Quantization: x as a (data,
  scale) tuple): random source bytes, moved unchanged -- receive data and
  scale rows bit for bit equal to the oracle's byte scatter, padding zero;
  per-expert and per-rank layouts;
- block-major scales (Modular MAX "EPBatchManager", ep_dispatch output_scales
  (hidden // block_size, max_recv_tokens)): the fused quantised dispatch and the
  pre-encoded move, bit for bit equal to the oracle's scales rearranged;
- full size (the 8 x 8192-token, H=4096, 128-expert MXFP8 workload): sampled
  rows and the block-major columns of the same rows.
"""
import numpy as np
import pytest
import torch

import oracle
from combine_ep_layout_03_gb300 import ep, synth
from gpu_harness import for_row_chunks, host_threads, to_dev_bf16

pytestmark = pytest.mark.gpu

MX = (ep.EP_QUANT_MXFP8_E4M3, ep.EP_QUANT_MXFP8_E5M2, ep.EP_QUANT_MXFP4_E2M1)


def elem_bytes(q):
    return 1 if q in MX else 4


def small(idx, **kw):
    w = synth.WORKLOADS[idx]
    return w.with_(**kw)


def expert_layout(w, topk):
    lay = ep.EPLayout(w.R, w.T, w.H, w.E, w.K, w.alpha)
    topk_d = torch.from_numpy(topk).cuda()
    lay.layout(topk_d)
    rows = int(lay.recv_rows()[-1])
    return lay, topk_d, rows


@pytest.mark.parametrize("q", [0, 2, 4, 5, 6, 7, 9])
@pytest.mark.parametrize("block_major", [False, True])
def test_pre_encoded_expert_layout(q, block_major):
    w = small(1, H=1024, alpha=4)
    topk = synth.gen_topk(w)
    olay = oracle.layout(w.R, w.T, w.E, w.K, w.alpha, topk)
    lay, _, rows = expert_layout(w, topk)
    assert rows == olay.rows
    db, sb = ep.ep_recv_row_bytes(w.H, q)
    src_d, src_s = synth.gen_encoded_rows(w, db, sb)
    cap = rows + 5
    if block_major:
        data, scales = lay.alloc_recv_block_major(q, cap)
    else:
        data, scales = lay.alloc_recv(q, cap)
    data.fill_(0x3C)
    if scales is not None:
        scales.fill_(0x3C)
    xs = torch.from_numpy(src_s).cuda() if sb else None
    lay.dispatch_ex(torch.from_numpy(src_d).cuda(), q, data, scales, x_scales=xs, pre_encoded=True,
                    block_major=block_major)
    assert lay.status() == ep.EP_OK
    od = oracle.dispatch_bytes(olay, src_d)
    assert np.array_equal(data[:rows].cpu().numpy(), od)
    # rows past the layout are not written
    assert torch.all(data[rows:] == 0x3C)
    if sb:
        os_ = oracle.dispatch_bytes(olay, src_s)
        if block_major:
            es = elem_bytes(q)
            ot = oracle.transpose_scales(os_, cap, es).reshape(sb // es, cap, es)
            got = scales.cpu().numpy().reshape(sb // es, cap, es)
            assert np.array_equal(got[:, :rows], ot[:, :rows])
            assert np.all(got[:, rows:] == 0x3C)
        else:
            assert np.array_equal(scales[:rows].cpu().numpy(), os_)


@pytest.mark.parametrize("q,H", [(4, 96), (5, 160), (9, 384)])
@pytest.mark.parametrize("block_major", [False, True])
def test_pre_encoded_scale_rows_not_16_byte_units(q, H, block_major):
    # 3, 5 and 12 scale bytes per row: the gather's byte / word paths without vector reads
    w = small(1, H=H, alpha=3, T=40)
    topk = synth.gen_topk(w)
    olay = oracle.layout(w.R, w.T, w.E, w.K, w.alpha, topk)
    lay, _, rows = expert_layout(w, topk)
    db, sb = ep.ep_recv_row_bytes(w.H, q)
    src_d, src_s = synth.gen_encoded_rows(w, db, sb)
    alloc = lay.alloc_recv_block_major if block_major else lay.alloc_recv
    data, scales = alloc(q, rows)
    scales.fill_(0x77)
    lay.dispatch_ex(torch.from_numpy(src_d).cuda(), q, data, scales, x_scales=torch.from_numpy(src_s).cuda(),
                    pre_encoded=True, block_major=block_major)
    assert lay.status() == ep.EP_OK
    assert np.array_equal(data.cpu().numpy(), oracle.dispatch_bytes(olay, src_d))
    os_ = oracle.dispatch_bytes(olay, src_s)
    if block_major:
        os_ = oracle.transpose_scales(os_, rows, elem_bytes(q))
    assert np.array_equal(scales.cpu().numpy(), os_)


def test_pre_encoded_scale_source_not_16_byte_aligned():
    # 16-byte scale rows whose source starts 4 bytes past a 16-byte boundary take
    # the gather instead of the bulk copies; the result is the same
    w = small(1, H=512, alpha=4, T=50)
    q = ep.EP_QUANT_MXFP8_E4M3
    topk = synth.gen_topk(w)
    olay = oracle.layout(w.R, w.T, w.E, w.K, w.alpha, topk)
    lay, _, rows = expert_layout(w, topk)
    db, sb = ep.ep_recv_row_bytes(w.H, q)
    src_d, src_s = synth.gen_encoded_rows(w, db, sb)
    buf = torch.zeros(src_s.size + 16, dtype=torch.uint8, device="cuda")
    xs = buf[4:4 + src_s.size]
    xs.copy_(torch.from_numpy(src_s.reshape(-1)))
    assert xs.data_ptr() % 16 == 4
    data, scales = lay.alloc_recv(q, rows)
    scales.fill_(0x21)
    lay.dispatch_ex(torch.from_numpy(src_d).cuda(), q, data, scales, x_scales=xs, pre_encoded=True)
    assert lay.status() == ep.EP_OK
    assert np.array_equal(data.cpu().numpy(), oracle.dispatch_bytes(olay, src_d))
    assert np.array_equal(scales.cpu().numpy(), oracle.dispatch_bytes(olay, src_s))


@pytest.mark.parametrize("q", [0, 4, 6, 9])
def test_pre_encoded_per_rank_layout(q):
    w = small(1, H=512, alpha=1, T=100)
    topk = synth.gen_topk(w)
    wts = synth.gen_weights(w, topk)
    tl = oracle.token_layout(w.R, w.T, w.E, w.K, topk, wts)
    lay, topk_d, _ = expert_layout(w, topk)
    lay.token_layout(topk_d, torch.from_numpy(wts).cuda())
    assert int(lay.token_rows()[-1]) == tl.rows
    db, sb = ep.ep_recv_row_bytes(w.H, q)
    src_d, src_s = synth.gen_encoded_rows(w, db, sb)
    data, scales = lay.alloc_recv(q, tl.rows)
    data.fill_(0x11)
    xs = torch.from_numpy(src_s).cuda() if sb else None
    lay.dispatch_ex(torch.from_numpy(src_d).cuda(), q, data, scales, x_scales=xs, pre_encoded=True,
                    per_rank=True)
    assert lay.status() == ep.EP_OK
    assert np.array_equal(data.cpu().numpy(), oracle.dispatch_bytes(tl, src_d))
    if sb:
        assert np.array_equal(scales.cpu().numpy(), oracle.dispatch_bytes(tl, src_s))


@pytest.mark.parametrize("q,kind", [(4, 0), (5, 0), (6, 0), (9, 0), (10, 2), (9, 3), (2, 0), (7, 1)])
def test_fused_dispatch_block_major_scales(q, kind):
    w = small(4, T=96, H=1024) if kind != 3 else small(1, H=1024, alpha=16)
    topk = synth.gen_topk(w)
    x = synth.gen_x(w)
    olay = oracle.layout(w.R, w.T, w.E, w.K, w.alpha, topk)
    lay, _, rows = expert_layout(w, topk)
    sc = synth.gen_scales(w, kind)
    if kind:
        od, os_ = oracle.dispatch_scaled(olay, x, q, topk, sc, kind)
    else:
        od, os_ = oracle.dispatch(olay, x, q)
    cap = rows + 3
    data, scales = lay.alloc_recv_block_major(q, cap)
    data.fill_(0x5A)
    scales.fill_(0x5A)
    lay.dispatch_ex(to_dev_bf16(x), q, data, scales, block_major=True,
                    scales=None if sc is None else torch.from_numpy(sc).cuda(), scale_kind=kind)
    assert lay.status() == ep.EP_OK
    assert np.array_equal(data[:rows].cpu().numpy(), od)
    es = elem_bytes(q)
    nb = os_.shape[1] // es
    got = scales.cpu().numpy().reshape(nb, cap, es)
    ot = oracle.transpose_scales(os_, cap, es).reshape(nb, cap, es)
    assert np.array_equal(got[:, :rows], ot[:, :rows])
    assert np.all(got[:, rows:] == 0x5A)


def test_per_rank_block_major_scales():
    w = small(1, H=1024, T=80)
    topk = synth.gen_topk(w)
    wts = synth.gen_weights(w, topk)
    x = synth.gen_x(w)
    tl = oracle.token_layout(w.R, w.T, w.E, w.K, topk, wts)
    lay, topk_d, _ = expert_layout(w, topk)
    lay.token_layout(topk_d, torch.from_numpy(wts).cuda())
    q = ep.EP_QUANT_MXFP8_E4M3
    data, scales = lay.alloc_recv_block_major(q, tl.rows)
    lay.dispatch_ex(to_dev_bf16(x), q, data, scales, per_rank=True, block_major=True)
    od, os_ = oracle.token_dispatch(tl, x, q)
    assert np.array_equal(data.cpu().numpy(), od)
    assert np.array_equal(scales.cpu().numpy(), oracle.transpose_scales(os_, tl.rows, 1))


def test_edge_cases():
    # no tokens: nothing to move, status stays OK
    w = small(1, T=0, H=256)
    topk = np.zeros((w.R, 0, w.K), np.int64)
    lay, _, rows = expert_layout(w, topk)
    assert rows == 0
    data, scales = lay.alloc_recv_block_major(4, 1)
    lay.dispatch_ex(torch.empty((0, 256), dtype=torch.uint8, device="cuda"), 4, data, scales,
                    x_scales=torch.empty((0, 8), dtype=torch.uint8, device="cuda"), pre_encoded=True,
                    block_major=True)
    assert lay.status() == ep.EP_OK
    # too small a receive buffer: nothing written, capacity error
    w = small(1, H=256)
    topk = synth.gen_topk(w)
    lay, _, rows = expert_layout(w, topk)
    db, sb = ep.ep_recv_row_bytes(w.H, 4)
    src_d, src_s = synth.gen_encoded_rows(w, db, sb)
    data, scales = lay.alloc_recv_block_major(4, rows - 1)
    data.fill_(7)
    lay.dispatch_ex(torch.from_numpy(src_d).cuda(), 4, data, scales,
                    x_scales=torch.from_numpy(src_s).cuda(), pre_encoded=True, block_major=True)
    assert lay.status() == ep.EP_ERR_CAPACITY
    assert torch.all(data == 7)


def test_full_size_mxfp8_pre_encoded_and_block_major():
    """Workload 4 at full size, the bench's keys 4p and 4x: every row."""
    w = synth.WORKLOADS[4]
    q = ep.EP_QUANT_MXFP8_E4M3
    topk = synth.gen_topk(w)
    olay = oracle.layout(w.R, w.T, w.E, w.K, w.alpha, topk)
    lay, _, rows = expert_layout(w, topk)
    assert rows == olay.rows
    db, sb = ep.ep_recv_row_bytes(w.H, q)
    src_d, src_s = synth.gen_encoded_rows_device(w, db, sb)
    data, scales = lay.alloc_recv_block_major(q, rows)
    data.fill_(0xA5)
    scales.fill_(0xA5)
    lay.dispatch_ex(src_d, q, data, scales, x_scales=src_s, pre_encoded=True, block_major=True)
    assert lay.status() == ep.EP_OK
    # every receive row and scale column against the oracle's byte scatter of
    # the pre-encoded source rows (padding rows zero), in chunks of rows
    sd, ss = src_d.cpu().numpy(), src_s.cpu().numpy()

    def check_pre(a, b):
        assert np.array_equal(data[a:b].cpu().numpy(), oracle.dispatch_bytes(olay, sd, rows=b, row_begin=a))
        assert np.array_equal(scales[:, a:b].cpu().numpy().T, oracle.dispatch_bytes(olay, ss, rows=b, row_begin=a))

    for_row_chunks(rows, check_pre)

    # the fused MXFP8 dispatch writing block-major scales: every row, and every
    # column against the oracle's row-major scales
    x_dev = synth.gen_x_device(w)
    x = x_dev.view(torch.int16).cpu().numpy().view(np.uint16).reshape(w.N, w.H)
    scales.fill_(0xA5)
    lay.dispatch_ex(x_dev, q, data, scales, block_major=True)
    assert lay.status() == ep.EP_OK
    enc_d, enc_s = oracle.encode_rows(q, x, host_threads())

    def check_fused(a, b):
        assert np.array_equal(data[a:b].cpu().numpy(), oracle.dispatch_bytes(olay, enc_d, rows=b, row_begin=a))
        assert np.array_equal(scales[:, a:b].cpu().numpy().T,
                              oracle.dispatch_bytes(olay, enc_s, rows=b, row_begin=a))

    for_row_chunks(rows, check_fused)
