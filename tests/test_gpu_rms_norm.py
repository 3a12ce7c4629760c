"""GPU parity for the combine fused with the residual add and RMSNorm (CANN
aclnnMoeDistributeCombineAddRmsNorm) against the oracle.

- x_out, rstd and y within the tolerance derived in the oracle (combine
  rounded to bf16, residual added and normalised in float32) of the float64
  reference built from the oracle's own layout, dispatch and stand-in expert;
- the oracle's float32 steps of the same reading (combine rounded to bf16,
  residual added in float32, a float32 sum of squares, rstd, two float32
  products): wherever the oracle's bf16 combine equals the GPU's plain
  combine (the combine's float32 summation order differs, so not quite
  everywhere), x_out equals the oracle's bit for bit and y is within one bf16
  step of it; rstd is within the float32 summation-order bound;
- the composition: x_out equals, bit for bit, bf16(float32(c) + residual) with
  c the plain combine's output of the same kernel arithmetic;
- edges: no tokens, tokens without experts, a receive buffer that is too small;
- full size (8 ranks x 4096 tokens, H = 7168, 256 experts, top-8): sampled
  tokens.
"""
import numpy as np
import pytest
import torch

import oracle
from combine_ep_layout_03_gb300 import ep, synth
from gpu_harness import GpuPath, bf16_bits, for_row_chunks, host_threads, to_dev_bf16

pytestmark = pytest.mark.gpu

EPS = synth.RMS_NORM_EPS


def run_norm(w, quant=0, mark=4, check_composition=True):
    topk = synth.gen_topk(w)
    wts = synth.gen_weights(w, topk)
    x = synth.gen_x(w)
    shared = synth.gen_shared(w)
    res = synth.gen_residual(w)
    gam = synth.gen_gamma(w)
    olay = oracle.layout(w.R, w.T, w.E, w.K, w.alpha, topk)
    g = GpuPath(w, topk)
    x_dev = to_dev_bf16(x)
    data, scales = g.dispatch(x_dev, quant)
    y = g.expert(quant, data, scales, mark)
    wts_dev = torch.from_numpy(wts).cuda()
    sh_dev = None if shared is None else to_dev_bf16(shared)
    res_dev = to_dev_bf16(res).view(w.N, w.H)
    gam_dev = to_dev_bf16(gam)
    out = torch.empty((w.N, w.H), dtype=torch.bfloat16, device="cuda")
    x_out = torch.empty_like(out)
    rstd = torch.empty(w.N, dtype=torch.float32, device="cuda")
    g.lay.combine_add_rms_norm(y, wts_dev, res_dev, gam_dev, out, x_out, rstd, sh_dev, EPS)
    assert g.lay.status() == ep.EP_OK
    # oracle: its own dispatch and stand-in expert, float64 combine and AddRmsNorm
    od, os_ = oracle.dispatch(olay, x, quant)
    rows = np.arange(olay.rows, dtype=np.int64)
    oy = oracle.expert_rows(olay, rows, w.H, quant, od, os_, mark)
    ref = oracle.combine_add_rms_norm_ref64(olay, oy, wts, shared, res, gam, EPS)
    ok, worst = oracle.add_rms_norm_within_tolerance(bf16_bits(x_out), rstd.cpu().numpy(), bf16_bits(out),
                                                     ref, w.K, w.num_shared)
    assert ok, worst
    c = g.combine(y, wts_dev, sh_dev)
    if check_composition:
        xf = (c.float() + res_dev.float()).to(torch.bfloat16)
        assert torch.equal(xf.view(torch.int16), x_out.view(torch.int16))
    # the oracle's float32 steps from its own bf16 combine
    c_or = oracle.combine(olay, oy, wts, shared)
    xo, ro, yo = oracle.add_rms_norm_f32(c_or, res.reshape(w.N, w.H), gam, EPS)
    check_against_f32_steps(bf16_bits(c), c_or, bf16_bits(x_out), xo, rstd.cpu().numpy(), ro,
                            bf16_bits(out), yo, w.H)
    return worst


def check_against_f32_steps(c_gpu, c_or, x_gpu, x_or, r_gpu, r_or, y_gpu, y_or, H, min_match=0.99):
    """Bit-exact x_out where the bf16 combines agree; rstd within the float32
    summation-order bound ((H + 8) 2^-24 relative: both sides add H positive
    squares, in different orders); y within one bf16 step where the combines
    agree (a relative rstd difference that small moves a product by less than
    one bf16 step, so at most one rounding flips)."""
    N = c_gpu.shape[0]
    c_gpu, c_or = c_gpu.reshape(N, H), c_or.reshape(N, H)
    match = c_gpu == c_or
    if match.size:
        assert match.mean() >= min_match, f"only {match.mean():.4f} of the combines agree"
    assert np.array_equal(x_gpu.reshape(N, H)[match], x_or[match]), "x_out differs where the combines agree"
    r_gpu = np.asarray(r_gpu, np.float64)
    r_or = np.asarray(r_or, np.float64)
    assert np.all(np.abs(r_gpu - r_or) <= (H + 8) * 2.0 ** -24 * r_or), "rstd outside the bound"
    yg = oracle.bf16_bits_to_f64(y_gpu.reshape(N, H))
    yr = oracle.bf16_bits_to_f64(y_or.reshape(N, H))
    step = oracle.ulp_bf16(np.maximum(np.abs(yg), np.abs(yr)))
    assert np.all(np.abs(yg - yr)[match] <= step[match]), "y more than one bf16 step from the oracle's"


@pytest.mark.parametrize("idx,T,quant", [(1, 64, 0), (1, 64, 4), (2, 48, 0), (3, 40, 2), (5, 12, 0)])
def test_combine_add_rms_norm_against_oracle(idx, T, quant):
    w = synth.WORKLOADS[idx].with_(T=T)
    if idx == 1:
        w = w.with_(H=1024)
    run_norm(w, quant)


def test_ragged_hidden_and_chunks():
    # H = 520: 65 vectors, a chunk size that does not divide the row
    w = synth.WORKLOADS[1].with_(T=33, H=520, K=2)
    run_norm(w)


def test_edges():
    # tokens without experts: x = shared sum + residual
    w = synth.WORKLOADS[5].with_(T=9, drop_p=1.0)
    run_norm(w)
    # no tokens at all: nothing to do
    w0 = synth.WORKLOADS[1].with_(T=0, H=256)
    g = GpuPath(w0, np.zeros((w0.R, 0, w0.K), np.int64))
    e = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    g.lay.combine_add_rms_norm(e, torch.empty((0, w0.K), device="cuda"), e, torch.ones(256, dtype=torch.bfloat16,
                               device="cuda"), e)
    assert g.lay.status() == ep.EP_OK
    # expert outputs shorter than the layout: capacity error, nothing written
    w = synth.WORKLOADS[1].with_(H=256)
    topk = synth.gen_topk(w)
    g = GpuPath(w, topk)
    y = torch.zeros((g.rows - 1, w.H), dtype=torch.bfloat16, device="cuda")
    out = torch.full((w.N, w.H), 3.0, dtype=torch.bfloat16, device="cuda")
    res = torch.zeros((w.N, w.H), dtype=torch.bfloat16, device="cuda")
    g.lay.combine_add_rms_norm(y, torch.ones((w.N, w.K), device="cuda"), res,
                               torch.ones(w.H, dtype=torch.bfloat16, device="cuda"), out)
    assert g.lay.status() == ep.EP_ERR_CAPACITY
    assert torch.all(out == 3.0)


def test_full_size_workload2_every_token():
    """Workload 2 at full size with the epilogue (the bench's key 2n): every
    token's x_out, rstd and y within the derived bound of the oracle's float64
    result, and against the oracle's float32 steps (bit-exact x_out where the
    combines agree), in chunks of tokens on host threads."""
    w = synth.WORKLOADS[2]
    topk = synth.gen_topk(w)
    wts = synth.gen_weights(w, topk)
    olay = oracle.layout(w.R, w.T, w.E, w.K, w.alpha, topk)
    g = GpuPath(w, topk)
    x_dev = synth.gen_x_device(w)
    x = bf16_bits(x_dev).reshape(w.N, w.H)
    data, _ = g.dispatch(x_dev, 0)
    y = data.view(torch.bfloat16).view(-1, w.H)
    res_dev = synth.gen_residual_device(w).view(w.N, w.H)
    gam = synth.gen_gamma(w)
    out = torch.empty((w.N, w.H), dtype=torch.bfloat16, device="cuda")
    x_out = torch.empty_like(out)
    rstd = torch.empty(w.N, dtype=torch.float32, device="cuda")
    wts_dev = torch.from_numpy(wts).cuda()
    g.lay.combine_add_rms_norm(y, wts_dev, res_dev, to_dev_bf16(gam), out, x_out, rstd, None, EPS)
    c_gpu = bf16_bits(g.combine(y, wts_dev)).reshape(w.N, w.H)
    torch.cuda.synchronize()
    assert g.lay.status() == ep.EP_OK
    res = bf16_bits(res_dev).reshape(w.N, w.H)
    xo_g, y_g, r_g = bf16_bits(x_out).reshape(w.N, w.H), bf16_bits(out).reshape(w.N, w.H), rstd.cpu().numpy()
    dr = olay.dst_row.reshape(w.N, w.K)
    wf = wts.reshape(w.N, w.K)

    def chunk(a, b):
        d = dr[a:b]
        rows = np.unique(d[d >= 0]).astype(np.int64)
        ymap = np.full(max(olay.rows, 1), -1, np.int64)
        ymap[rows] = np.arange(len(rows))
        od, _ = oracle.dispatch_rows(olay, x, 0, rows)   # identity experts: y = the receive rows
        yo = od.view(np.uint16).reshape(len(rows), w.H)
        mini = oracle.Layout(R=1, T=b - a, K=w.K, dst_row=np.ascontiguousarray(d.reshape(1, b - a, w.K)))
        c, mag = oracle.combine_ref64(mini, yo, wf[a:b], None, 0, b - a, ymap)
        xr, rs, yv = oracle.add_rms_norm_ref64(c, res[a:b], gam, EPS)
        ref = dict(c=c, mag=mag, x=xr, rstd=rs, y=yv, gamma=oracle.bf16_bits_to_f64(gam))
        ok, worst = oracle.add_rms_norm_within_tolerance(xo_g[a:b], r_g[a:b], y_g[a:b], ref, w.K, 0)
        assert ok, (a, worst)
        c_or = oracle.combine(mini, yo, wf[a:b], None, 0, b - a, ymap)
        xo, ro, yo32 = oracle.add_rms_norm_f32(c_or, res[a:b], gam, EPS)
        check_against_f32_steps(c_gpu[a:b], c_or, xo_g[a:b], xo, r_g[a:b], ro, y_g[a:b], yo32, w.H)

    for_row_chunks(w.N, chunk, step=1024, threads=host_threads(cap=12))
