"""GPU parity at the five workloads' full sizes, in the launch configuration the
benchmark times (the same library calls).

- layout: every array compared with the oracle, bit for bit;
- dispatch: sampled receive rows (random rows, both ends of every rank, every
  padding row of a few experts) compared bit for bit with rows the oracle
  computes one by one; every padding row checked zero on the device;
- combine: sampled source tokens against the oracle (its own dispatch and
  stand-in expert), plus, for every token, the closed form of dispatch ->
  identity expert -> combine: out = x * sum_k w_k (+ sum_q shared).
"""
import numpy as np
import pytest
import torch

import oracle
from combine_ep_layout_03_gb300 import synth
from gpu_harness import GpuPath, bf16_bits, compare_layout, oracle_combine_sampled

pytestmark = pytest.mark.gpu


def sample_rows(olay, rng, n=1500):
    rows = [rng.integers(0, olay.rows, n)]
    for j in range(olay.R):
        a, b = int(olay.rank_base[j]), int(olay.rank_base[j + 1])
        if b > a:
            rows.append(np.array([a, b - 1]))
    base = np.concatenate([[0], np.cumsum(olay.aligned)])
    for e in rng.choice(olay.E, min(olay.E, 6), replace=False):
        rows.append(np.arange(base[e] + olay.recv_cnt[e], base[e + 1]))
    return np.unique(np.concatenate(rows)).astype(np.int64)


def padding_rows_zero(olay, data, scales):
    base = np.concatenate([[0], np.cumsum(olay.aligned)])
    for e in range(olay.E):
        a, b = int(base[e] + olay.recv_cnt[e]), int(base[e + 1])
        if b > a:
            assert not torch.any(data[a:b]), f"padding rows of expert {e} not zero"
            if scales is not None:
                assert not torch.any(scales[a:b])


@pytest.mark.parametrize("idx", [1, 2, 3, 4, 5])
def test_full_size(idx):
    w = synth.WORKLOADS[idx]
    rng = np.random.default_rng(idx)
    topk = synth.gen_topk(w)
    wts = synth.gen_weights(w, topk)
    olay = oracle.layout(w.R, w.T, w.E, w.K, w.alpha, topk)
    g = GpuPath(w, topk)
    assert g.rows == olay.rows
    compare_layout(g.views_numpy(), olay)
    assert g.lay.status() == 0

    x_dev = synth.gen_x_device(w)
    x = bf16_bits(x_dev).reshape(w.N, w.H)
    sh_dev = synth.gen_shared_device(w)
    wts_dev = torch.from_numpy(wts).cuda()
    tokens = np.unique(np.concatenate([rng.integers(0, w.N, 200), [0, w.N - 1]]))
    sh_tok = None
    if sh_dev is not None:
        s_idx = torch.from_numpy(tokens // w.T).cuda()
        t_idx = torch.from_numpy(tokens % w.T).cuda()
        sh_tok = bf16_bits(sh_dev[s_idx, :, t_idx, :]).reshape(len(tokens), w.num_shared, w.H)

    for q in w.quants:
        data, scales = g.dispatch(x_dev, q, fill=0xA5)
        rows = sample_rows(olay, rng)
        od, os_ = oracle.dispatch_rows(olay, x, q, rows)
        ridx = torch.from_numpy(rows).cuda()
        assert np.array_equal(data[ridx].cpu().numpy(), od), "sampled receive rows differ"
        if scales is not None:
            assert np.array_equal(scales[ridx].cpu().numpy(), os_), "sampled scales differ"
        padding_rows_zero(olay, data, scales)

        # marked stand-in expert, combine, sampled tokens against the oracle
        mark = 16
        y = g.expert(q, data, scales, mark, inplace=(q == 0))
        out = g.combine(y, wts_dev, sh_dev)
        o, ref, mag = oracle_combine_sampled(olay, x, wts, sh_tok, q, mark, tokens)
        got = bf16_bits(out[torch.from_numpy(tokens).cuda()])
        ok, excess, rel = oracle.combine_within_tolerance(got, ref, mag, w.K, w.num_shared)
        assert ok, (q, excess, rel)
        assert g.lay.status() == 0
        del y, out, data, scales
        torch.cuda.empty_cache()

    if 0 in w.quants:
        # closed form at full size: identity experts
        data, _ = g.dispatch(x_dev, 0)
        y = data.view(torch.bfloat16).view(-1, w.H)
        out = g.combine(y, wts_dev, sh_dev)
        coef = wts_dev.view(w.N, w.K).masked_fill(torch.from_numpy(topk).cuda().view(w.N, w.K) < 0, 0)
        step = 8192
        for a in range(0, w.N, step):
            b = min(w.N, a + step)
            xf = x_dev.view(w.N, w.H)[a:b].double()
            ref = xf * coef[a:b].double().sum(1, keepdim=True)
            mag = xf.abs() * coef[a:b].double().abs().sum(1, keepdim=True)
            if sh_dev is not None:
                shf = sh_dev.view(w.R, w.num_shared, w.T, w.H).permute(0, 2, 1, 3).reshape(
                    w.N, w.num_shared, w.H)[a:b].double()
                ref = ref + shf.sum(1)
                mag = mag + shf.abs().sum(1)
            got = out[a:b].double()
            ulp = torch.ldexp(torch.ones_like(ref), torch.frexp(ref.abs())[1] - 8)
            ulp = torch.clamp(ulp, min=2.0 ** -133)
            bound = 2 * ulp + mag * (2 * w.K + w.num_shared + 1) * 2.0 ** -24
            assert torch.all((got - ref).abs() <= bound), f"closed form fails at tokens {a}:{b}"
