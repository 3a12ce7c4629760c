"""GPU parity for the further quant modes and xActiveMask (CANN
aclnnMoeDistributeDispatchV2: quantMode 1 static int8 with scales of shape (1,),
(H,) or (E,H); quantMode 2 with FP8 destinations; quantMode 3 per-group FP8;
smooth scales for modes 1-3; xActiveMask 1-D / 2-D).

Receive rows, scales and the stand-in expert's rows are compared with the
oracle bit for bit; combine within the derived tolerance.  Hidden sizes cover
the bulk-store path (rows and group-scale rows multiples of 16 bytes), the
per-thread store path (H % 16 != 0) and the per-thread group-scale path
(H % 512 != 0).
"""
import os

import numpy as np
import pytest
import torch

import oracle
from combine_ep_layout_03_gb300 import ep, synth
from gpu_harness import GpuPath, bf16_bits, compare_layout, to_dev_bf16

pytestmark = pytest.mark.gpu

FP8T = (ep.EP_QUANT_FP8_E4M3_PER_TOKEN, ep.EP_QUANT_FP8_E5M2_PER_TOKEN)
FP8G = (ep.EP_QUANT_FP8_E4M3_PER_GROUP, ep.EP_QUANT_FP8_E5M2_PER_GROUP)


def run_case(w, q, kind, mark=16, check_combine=True):
    topk = synth.gen_topk(w)
    wts = synth.gen_weights(w, topk)
    x = synth.gen_x(w)
    scales = synth.gen_scales(w, kind)
    olay = oracle.layout(w.R, w.T, w.E, w.K, w.alpha, topk)
    g = GpuPath(w, topk)
    compare_layout(g.views_numpy(), olay)
    if kind == 0:
        od, os_ = oracle.dispatch(olay, x, q)
    else:
        od, os_ = oracle.dispatch_scaled(olay, x, q, topk, scales, kind)
    data, sc = g.lay.alloc_recv(q, max(olay.rows, 1))
    data.fill_(0xA5)
    if sc is not None:
        sc.fill_(0xA5)
    sdev = None if scales is None else torch.from_numpy(scales).cuda()
    g.lay.dispatch(to_dev_bf16(x), q, data, sc, scales=sdev, scale_kind=kind)
    assert g.lay.status() == 0
    assert np.array_equal(data[: olay.rows].cpu().numpy(), od), "receive rows differ"
    if os_.shape[1]:
        assert np.array_equal(sc[: olay.rows].cpu().numpy(), os_), "receive scales differ"
    if not check_combine:
        return
    y = g.expert(q, data, sc, mark)
    oy = oracle.expert_rows(olay, np.arange(olay.rows), w.H, q, od, os_, mark)
    assert np.array_equal(bf16_bits(y[: olay.rows]), oy), "stand-in expert rows differ"
    out = g.combine(y, torch.from_numpy(wts).cuda())
    ref, mag = oracle.combine_ref64(olay, oy, wts)
    ok, excess, rel = oracle.combine_within_tolerance(bf16_bits(out), ref, mag, w.K)
    assert ok, (excess, rel)


@pytest.mark.parametrize("q", FP8T + FP8G)
@pytest.mark.parametrize("kind", [0, 2, 3])
def test_fp8_token_and_group(q, kind):
    run_case(synth.WORKLOADS[4].with_(T=201), q, kind)


@pytest.mark.parametrize("q", FP8T + FP8G)
def test_fp8_group_scales_not_bulk_h1152(q):
    # H % 512 != 0: group-scale rows are not multiples of 16 bytes -> per-thread scale stores
    run_case(synth.Workload(21, R=4, T=60, H=1152, E=16, K=4, alpha=8), q, 2)


@pytest.mark.parametrize("kind", [1, 2, 3])
def test_int8_static(kind):
    run_case(synth.WORKLOADS[3].with_(T=150), ep.EP_QUANT_INT8_STATIC, kind)


@pytest.mark.parametrize("kind", [2, 3])
def test_int8_per_token_smooth(kind):
    run_case(synth.WORKLOADS[3].with_(T=150), ep.EP_QUANT_INT8_PER_TOKEN, kind)


@pytest.mark.parametrize("q", [ep.EP_QUANT_INT8_STATIC, ep.EP_QUANT_FP8_E4M3_PER_TOKEN,
                               ep.EP_QUANT_INT8_PER_TOKEN])
def test_rows_not_multiple_of_16_bytes(q):
    # H = 1000: 1000-byte rows take the per-thread store path
    kind = 1 if q == ep.EP_QUANT_INT8_STATIC else 0
    run_case(synth.Workload(22, R=4, T=50, H=1000, E=16, K=3, alpha=4), q, kind)


@pytest.mark.parametrize("q,H", [(ep.EP_QUANT_INT8_PER_TOKEN, 1000), (ep.EP_QUANT_FP8_E4M3_PER_TOKEN, 1000),
                                 (ep.EP_QUANT_INT8_STATIC, 1000), (ep.EP_QUANT_FP8_E4M3_PER_GROUP, 1152),
                                 (ep.EP_QUANT_INT8_PER_TOKEN, 8), (ep.EP_QUANT_FP8_E5M2_PER_TOKEN, 8184)])
def test_per_expert_scales_ragged_rows(q, H):
    # per-expert scales with rows that do not fill the last vectors of the CTA
    # (H = 1000: 125 vectors on 32 threads x 4; H = 1152: 144 on 64 x 4), a
    # single-warp CTA (H = 8) and the largest CTA with one vector short (H = 8184)
    run_case(synth.Workload(24, R=4, T=40, H=H, E=16, K=4, alpha=4), q, 3)


def test_zero_rows_and_groups():
    w = synth.Workload(23, R=2, T=6, H=256, E=4, K=2, alpha=1)
    topk = np.array([[[0, 1], [2, 3], [1, 2], [0, 3], [3, 1], [2, 0]]] * 2, np.int64)
    xf = np.zeros((12, 256), np.float32)
    xf[1, :128] = np.linspace(-3, 3, 128)       # group 1 of token 1 all zero
    xf[2, 128:] = 1e-30                         # tiny group
    xf[3] = np.random.default_rng(0).standard_normal(256) * 1e4
    x = torch.from_numpy(xf).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).reshape(2, 6, 256)
    olay = oracle.layout(2, 6, 4, 2, 1, topk)
    g = GpuPath(w, topk)
    for q in FP8T + FP8G:
        od, os_ = oracle.dispatch(olay, x, q)
        data, sc = g.lay.alloc_recv(q, olay.rows)
        g.lay.dispatch(to_dev_bf16(x), q, data, sc)
        assert np.array_equal(data.cpu().numpy(), od) and np.array_equal(sc.cpu().numpy(), os_)


@pytest.mark.parametrize("dims", [1, 2])
@pytest.mark.parametrize("idx,T", [(2, 300), (5, 90)])
def test_active_mask_layout_and_dispatch(dims, idx, T):
    w = synth.WORKLOADS[idx].with_(T=T)
    topk = synth.gen_topk(w)
    mask = synth.gen_mask(w, dims)
    olay = oracle.layout(w.R, w.T, w.E, w.K, w.alpha, topk, mask=mask)
    lay = ep.EPLayout(w.R, w.T, w.H, w.E, w.K, w.alpha)
    lay.layout(torch.from_numpy(topk).cuda(), active_mask=torch.from_numpy(mask).cuda())
    v = {k: t.cpu().numpy() for k, t in lay.views().items()}
    rows = int(lay.recv_rows()[-1])
    v["recv_src"] = v["recv_src"][:rows]
    compare_layout(v, olay)
    x = synth.gen_x(w)
    data, sc = lay.alloc_recv(0, max(rows, 1))
    lay.dispatch(to_dev_bf16(x), 0, data, sc)
    od, _ = oracle.dispatch(olay, x, 0)
    assert np.array_equal(data[:rows].cpu().numpy(), od)
    assert lay.status() == 0


@pytest.mark.parametrize("q,kind", [(ep.EP_QUANT_FP8_E4M3_PER_TOKEN, 0),
                                    (ep.EP_QUANT_FP8_E4M3_PER_GROUP, 0),
                                    (ep.EP_QUANT_INT8_STATIC, 2),
                                    (ep.EP_QUANT_INT8_PER_TOKEN, 3)])
def test_full_size_every_row(q, kind):
    """Workload 4 (or 3 for the int8 modes) at full size, the bench's keys 4t, 4g, 3s
    and 3e: every receive row and scale row against the oracle, streamed in
    chunks of receive rows (the oracle's dispatch of each chunk on a host
    thread; under the Zipf routing of workload 3 rank 0 alone receives most
    rows, so chunks rather than ranks keep the threads even)."""
    from concurrent.futures import ThreadPoolExecutor
    w = synth.WORKLOADS[4 if q in FP8T + FP8G else 3]
    topk = synth.gen_topk(w)
    olay = oracle.layout(w.R, w.T, w.E, w.K, w.alpha, topk)
    g = GpuPath(w, topk)
    x_dev = synth.gen_x_device(w)
    x = bf16_bits(x_dev).reshape(w.N, w.H)
    scales = synth.gen_scales(w, kind)
    data, sc = g.lay.alloc_recv(q, olay.rows)
    data.fill_(0xA5)
    if sc is not None:
        sc.fill_(0xA5)
    g.lay.dispatch(x_dev, q, data, sc, scales=None if scales is None else torch.from_numpy(scales).cuda(),
                   scale_kind=kind)
    torch.cuda.synchronize()
    assert g.lay.status() == 0
    threads = max(1, min(16, len(os.sched_getaffinity(0))))
    enc = oracle.encode_rows(q, x, threads) if kind == 0 else None

    step = 32768

    def chunk(a):
        b = min(olay.rows, a + step)
        if kind == 0:
            od = oracle.dispatch_bytes(olay, enc[0], rows=b, row_begin=a)
            os_ = oracle.dispatch_bytes(olay, enc[1], rows=b, row_begin=a)
        else:
            od, os_ = oracle.dispatch_scaled(olay, x, q, topk, scales, kind, a, b)
        assert np.array_equal(data[a:b].cpu().numpy(), od), f"receive rows {a}:{b} differ"
        if sc is not None:
            assert np.array_equal(sc[a:b].cpu().numpy(), os_), f"receive scales {a}:{b} differ"

    with ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(chunk, range(0, olay.rows, step)))
