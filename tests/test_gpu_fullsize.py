"""GPU parity at the five workloads' full sizes, every output, in the launch
configuration the benchmark times (the same library calls):

- layout: every array compared with the oracle, bit for bit;
- dispatch: every receive row and scale row, streamed per destination rank:
  rank j's rows [rank_base[j], rank_base[j+1]) are copied back into host
  memory and compared bit for bit with the oracle's dispatch of the same rows
  (the oracle encodes each source token once and places the encoding by its
  own dst_row; padding rows are all zero);
- combine: every source token, in chunks of one source rank's tokens, against
  the oracle's own dispatch -> marked stand-in expert -> combine, within the
  derived tolerance (float64 reference);
- workloads without quantisation also get the closed form of dispatch ->
  identity expert -> combine for every token: out = x * sum_k w_k
  (+ sum_q shared).

The oracle's C calls run on the host cores in threads (they release the
interpreter lock and share no state); host memory stays bounded by a few
rank- or chunk-sized buffers at a time.
"""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle
from combine_ep_layout_03_gb300 import synth
from gpu_harness import GpuPath, bf16_bits, compare_layout

pytestmark = pytest.mark.gpu

MARK = 16      # stand-in expert e multiplies its rows by 2^-(e mod MARK)
CHUNK = 1024   # source tokens per combine check (divides every workload's T or equals it)


def host_threads(cap=12):
    try:
        n = len(os.sched_getaffinity(0))
    except Exception:
        n = os.cpu_count() or 1
    return max(1, min(cap, n))


def same_bytes(a: np.ndarray, b: np.ndarray) -> bool:
    a = np.ascontiguousarray(a).reshape(-1)
    b = np.ascontiguousarray(b).reshape(-1)
    if a.shape != b.shape:
        return False
    if a.nbytes % 8 == 0:   # eight bytes per comparison: a smaller temporary
        return bool(np.array_equal(a.view(np.uint64), b.view(np.uint64)))
    return bool(np.array_equal(a, b))


def check_dispatch(olay, q, H, data, scales, enc_d, enc_s):
    """Every receive row (and scale row) of every destination rank."""
    db, sb = oracle.row_bytes(q, H)

    def rank(j):
        a, b = int(olay.rank_base[j]), int(olay.rank_base[j + 1])
        if b == a:
            return
        exp = oracle.dispatch_bytes(olay, enc_d, rows=b, row_begin=a)
        assert same_bytes(data[a:b].cpu().numpy(), exp), f"receive rows of rank {j} differ"
        if sb:
            exp_s = oracle.dispatch_bytes(olay, enc_s, rows=b, row_begin=a)
            assert same_bytes(scales[a:b].cpu().numpy(), exp_s), f"receive scales of rank {j} differ"

    with ThreadPoolExecutor(max_workers=min(4, host_threads())) as ex:
        list(ex.map(rank, range(olay.R)))


def check_combine(w, olay, q, enc_d, enc_s, wts, sh_dev, out):
    """Every source token against the oracle's dispatch -> marked stand-in
    expert -> combine (float64 reference, derived tolerance)."""
    N, H, K, S, T = w.N, w.H, w.K, w.num_shared, w.T
    c = min(CHUNK, T)
    assert T % c == 0
    out_host = bf16_bits(out).reshape(N, H)
    dr = olay.dst_row.reshape(N, K)
    wf = np.ascontiguousarray(wts, np.float32).reshape(N, K)

    def chunk(a):
        b = a + c
        d = dr[a:b]
        rows = np.unique(d[d >= 0]).astype(np.int64)
        ymap = np.full(max(olay.rows, 1), -1, np.int64)
        ymap[rows] = np.arange(len(rows))
        src = olay.recv_src[rows]
        assert np.all(src >= 0)
        y = oracle.expert_rows(olay, rows, H, q, enc_d[src], enc_s[src], MARK)
        mini = oracle.Layout(R=1, T=c, K=K, dst_row=np.ascontiguousarray(d.reshape(1, c, K)))
        sh = None
        if sh_dev is not None:
            s, t0 = a // T, a % T
            sh = bf16_bits(sh_dev[s, :, t0:t0 + c, :]).reshape(1, S, c, H)
        ref, mag = oracle.combine_ref64(mini, y, wf[a:b], sh, 0, c, ymap)
        ok, excess, rel = oracle.combine_within_tolerance(out_host[a:b], ref, mag, K, S)
        assert ok, f"combine of tokens {a}:{b} outside the tolerance (excess {excess}, rel {rel})"

    with ThreadPoolExecutor(max_workers=host_threads()) as ex:
        list(ex.map(chunk, range(0, N, c)))


def check_closed_form(w, topk, x_dev, wts_dev, sh_dev, out):
    """Identity experts: out = x * sum_k w_k (+ sum_q shared) for every token."""
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


@pytest.mark.parametrize("idx", [1, 2, 3, 4, 5])
def test_full_size(idx):
    w = synth.WORKLOADS[idx]
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

    for q in w.quants:
        enc_d, enc_s = oracle.encode_rows(q, x, host_threads(cap=64))
        data, scales = g.dispatch(x_dev, q, fill=0xA5)
        torch.cuda.synchronize()
        assert g.lay.status() == 0
        check_dispatch(olay, q, w.H, data, scales, enc_d, enc_s)

        # marked stand-in expert (in place for bf16 rows), then combine
        y = g.expert(q, data, scales, MARK, inplace=(q == 0))
        out = g.combine(y, wts_dev, sh_dev)
        torch.cuda.synchronize()
        assert g.lay.status() == 0
        check_combine(w, olay, q, enc_d, enc_s, wts, sh_dev, out)
        del y, out, data, scales, enc_d, enc_s
        torch.cuda.empty_cache()

    if 0 in w.quants:
        data, _ = g.dispatch(x_dev, 0)
        y = data.view(torch.bfloat16).view(-1, w.H)
        out = g.combine(y, wts_dev, sh_dev)
        check_closed_form(w, topk, x_dev, wts_dev, sh_dev, out)
        assert g.lay.status() == 0


def test_full_size_active_mask():
    """Workload 5 at full size with a 2-D xActiveMask (the bench's key 5m): the
    masked layout, every receive row and every combine output against the
    oracle (masked entries take no part, like -1 ids)."""
    from combine_ep_layout_03_gb300 import ep
    w = synth.WORKLOADS[5]
    topk = synth.gen_topk(w)
    wts = synth.gen_weights(w, topk)
    mask = synth.gen_mask(w, 2)
    olay = oracle.layout(w.R, w.T, w.E, w.K, w.alpha, topk, mask=mask)
    lay = ep.EPLayout(w.R, w.T, w.H, w.E, w.K, w.alpha)
    lay.layout(torch.from_numpy(topk).cuda(), active_mask=torch.from_numpy(mask).cuda())
    v = {k: t.cpu().numpy() for k, t in lay.views().items()}
    v["recv_src"] = v["recv_src"][: olay.rows]
    compare_layout(v, olay)
    assert lay.status() == 0
    x_dev = synth.gen_x_device(w)
    x = bf16_bits(x_dev).reshape(w.N, w.H)
    sh_dev = synth.gen_shared_device(w)
    enc_d, enc_s = oracle.encode_rows(0, x, host_threads(cap=64))
    data, _ = lay.alloc_recv(0, max(olay.rows, 1))
    data.fill_(0xA5)
    lay.dispatch(x_dev, 0, data, None)
    torch.cuda.synchronize()
    assert lay.status() == 0
    check_dispatch(olay, 0, w.H, data, None, enc_d, enc_s)
    y = data.view(torch.bfloat16).view(-1, w.H)
    lay.expert_identity(0, data, None, y, MARK)
    # masked entries carry no weight, as in the benchmark
    wm = np.where(mask.reshape(wts.shape) != 0, wts, np.float32(0)).astype(np.float32)
    out = torch.empty((w.N, w.H), dtype=torch.bfloat16, device="cuda")
    lay.combine(y, torch.from_numpy(wm).cuda(), out, sh_dev)
    torch.cuda.synchronize()
    assert lay.status() == 0
    check_combine(w, olay, 0, enc_d, enc_s, wm, sh_dev, out)
