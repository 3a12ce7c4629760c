"""GPU parity on rows holding non-finite and subnormal values.

Tokens cycle through row kinds: plain, with +-inf planted, with NaNs of
several payloads planted, all subnormal, all NaN, large values with -0, and
zeros with one subnormal.  bf16 dispatch (per-expert and per-rank receive
layouts) must move every bit pattern unchanged; per-token int8 (also with
per-channel and per-expert input scales), static int8 and the MX modes (no
NaN rows: the MX and FP8 casts of NaN are not defined by the formulas) must
match the oracle's codes and scales bit for bit; MX rows holding NaN
elements must match the oracle's scale bytes and the codes of every non-NaN
element (a NaN element's own code is left unspecified); combine
must give NaN exactly where the oracle's float32 combine does, the same
infinities, and finite values within the derived tolerance.
"""
import numpy as np
import pytest
import torch

import oracle
from combine_ep_layout_03_gb300 import ep, synth
from gpu_harness import GpuPath, bf16_bits, to_dev_bf16

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS[1].with_(T=48, H=256, K=2)
NAN_KINDS = (2, 4)


def special_rows(w, nan_rows=True):
    rng = np.random.default_rng(77)
    x = synth.gen_x(w).reshape(w.N, w.H).copy()
    H = w.H
    for n in range(w.N):
        kind = n % 7
        if kind in NAN_KINDS and not nan_rows:
            continue
        r = x[n]
        pos = rng.choice(H, 3, replace=False)
        if kind == 1:
            r[pos] = [0x7F80, 0xFF80, 0x7F80]
        elif kind == 2:
            r[pos] = [0x7FC0, 0x7F81, 0xFFC1]
        elif kind == 3:
            mant = rng.integers(1, 128, H).astype(np.uint16)
            r[:] = mant | (rng.integers(0, 2, H).astype(np.uint16) << 15)
            r[pos[:1]] = 0
        elif kind == 4:
            r[:] = 0x7FC0
        elif kind == 5:
            r[pos] = [0x7F00, 0xFF00, 0x8000]   # +-1.7e38 and -0
        elif kind == 6:
            r[:] = 0
            r[pos[0]] = 0x0005
    return x


def setup(nan_rows=True):
    w = W
    topk = synth.gen_topk(w)
    wts = synth.gen_weights(w, topk)
    x = special_rows(w, nan_rows)
    olay = oracle.layout(w.R, w.T, w.E, w.K, w.alpha, topk)
    g = GpuPath(w, topk)
    return w, topk, wts, x, olay, g


def test_bf16_rows_move_every_bit_pattern():
    w, topk, wts, x, olay, g = setup()
    xd = to_dev_bf16(x)
    data, _ = g.dispatch(xd, ep.EP_QUANT_NONE, fill=0x5A)
    od, _ = oracle.dispatch(olay, x, ep.EP_QUANT_NONE)
    assert np.array_equal(data[: olay.rows].cpu().numpy(), od)
    tl = oracle.token_layout(w.R, w.T, w.E, w.K, topk, wts)
    g.lay.token_layout(g.topk_dev, torch.from_numpy(wts).cuda())
    td, _ = g.lay.alloc_recv(ep.EP_QUANT_NONE, tl.rows)
    g.lay.dispatch_tokens(xd, ep.EP_QUANT_NONE, td, None)
    assert np.array_equal(td.cpu().numpy(), oracle.token_dispatch(tl, x, ep.EP_QUANT_NONE)[0])
    assert g.lay.status() == ep.EP_OK


@pytest.mark.parametrize("q", [ep.EP_QUANT_INT8_PER_TOKEN, ep.EP_QUANT_INT8_STATIC,
                               ep.EP_QUANT_MXFP8_E4M3, ep.EP_QUANT_MXFP8_E5M2, ep.EP_QUANT_MXFP4_E2M1])
def test_quantised_rows(q):
    mx = q in (ep.EP_QUANT_MXFP8_E4M3, ep.EP_QUANT_MXFP8_E5M2, ep.EP_QUANT_MXFP4_E2M1)
    w, topk, wts, x, olay, g = setup(nan_rows=not mx)
    data, sc = g.lay.alloc_recv(q, olay.rows)
    data.fill_(0xA5)
    if sc is not None:
        sc.fill_(0xA5)
    if q == ep.EP_QUANT_INT8_STATIC:
        one = np.ones(1, np.float32)
        g.lay.dispatch(to_dev_bf16(x), q, data, sc, scales=torch.from_numpy(one).cuda(),
                       scale_kind=ep.EP_SCALES_SCALAR)
        od, os_ = oracle.dispatch_scaled(olay, x, q, topk, one, ep.EP_SCALES_SCALAR)
    else:
        g.lay.dispatch(to_dev_bf16(x), q, data, sc)
        od, os_ = oracle.dispatch(olay, x, q)
    assert g.lay.status() == ep.EP_OK
    assert np.array_equal(data.cpu().numpy(), od), "receive rows differ"
    if os_.shape[1]:
        assert np.array_equal(sc.cpu().numpy(), os_), "receive scales differ"


@pytest.mark.parametrize("q", [ep.EP_QUANT_MXFP8_E4M3, ep.EP_QUANT_MXFP8_E5M2, ep.EP_QUANT_MXFP4_E2M1])
def test_mx_blocks_with_nan_elements(q):
    w, topk, wts, x, olay, g = setup(nan_rows=True)
    data, sc = g.lay.alloc_recv(q, olay.rows)
    data.fill_(0xA5)
    sc.fill_(0xA5)
    g.lay.dispatch(to_dev_bf16(x), q, data, sc)
    od, os_ = oracle.dispatch(olay, x, q)
    assert g.lay.status() == ep.EP_OK
    assert np.array_equal(sc.cpu().numpy(), os_), "scale bytes differ"
    src = olay.recv_src[: olay.rows]
    assert np.all(src >= 0)
    nan = is_nan(x)[src]                                # [rows, H] NaN source elements
    got = data.cpu().numpy()
    if q == ep.EP_QUANT_MXFP4_E2M1:
        # element 2i in the low nibble of byte i
        got = np.stack([got & 0xF, got >> 4], axis=-1).reshape(nan.shape)
        od = np.stack([od & 0xF, od >> 4], axis=-1).reshape(nan.shape)
    assert nan.any() and (~nan).any()
    assert np.array_equal(got[~nan], od[~nan]), "codes of non-NaN elements differ"


@pytest.mark.parametrize("kind", [ep.EP_SCALES_PER_CHANNEL, ep.EP_SCALES_PER_EXPERT])
def test_int8_with_input_scales(kind):
    # subnormal rows times scales in [0.5, 2) stay subnormal: the infinite-scale path
    w, topk, wts, x, olay, g = setup()
    q = ep.EP_QUANT_INT8_PER_TOKEN
    scales = synth.gen_scales(w, kind)
    data, sc = g.lay.alloc_recv(q, olay.rows)
    data.fill_(0xA5)
    sc.fill_(0xA5)
    g.lay.dispatch(to_dev_bf16(x), q, data, sc, scales=torch.from_numpy(scales).cuda(), scale_kind=kind)
    od, os_ = oracle.dispatch_scaled(olay, x, q, topk, scales, kind)
    assert g.lay.status() == ep.EP_OK
    assert np.array_equal(data.cpu().numpy(), od), "receive rows differ"
    assert np.array_equal(sc.cpu().numpy(), os_), "receive scales differ"


def is_nan(b):
    return ((b & 0x7F80) == 0x7F80) & ((b & 0x7F) != 0)


def test_combine_propagates_non_finite():
    w, topk, wts, x, olay, g = setup()
    data, _ = g.dispatch(to_dev_bf16(x), ep.EP_QUANT_NONE)
    y = data.view(torch.bfloat16).view(-1, w.H)
    out = g.combine(y, torch.from_numpy(wts).cuda())
    got = bf16_bits(out)
    oy = data[: olay.rows].cpu().numpy().view(np.uint16).reshape(olay.rows, w.H)
    o = oracle.combine(olay, oy, wts)
    nan_o = is_nan(o)
    assert np.array_equal(is_nan(got), nan_o), "NaN positions differ"
    inf_o = (o & 0x7FFF) == 0x7F80
    assert np.array_equal(got[inf_o], o[inf_o]), "infinities differ"
    assert not np.any(((got & 0x7FFF) == 0x7F80) & ~inf_o), "spurious infinities"
    ref, mag = oracle.combine_ref64(olay, oy, wts)
    fin = ~nan_o & ~inf_o
    assert np.all(np.isfinite(ref[fin]))
    ok, excess, rel = oracle.combine_within_tolerance(got[fin], ref[fin], mag[fin], w.K)
    assert ok, (excess, rel)
    assert g.lay.status() == ep.EP_OK
